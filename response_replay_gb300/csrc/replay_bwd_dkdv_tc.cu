// replay_bwd_dkdv_tc.cu -- dK, dV of the response's own keys on the 5th-generation
// tensor cores.
//
// The captured prompt state is stopgrad (LongStraw paper digest, Method, last paragraph;
// explainer, Figure 2 caption), so K/V gradients exist only for the response's own keys
// (explainer, "Two incompatible architectures", Qwen bullet: K/V gradient pages only
// where a response backward touches them).  With P_{t,j} = exp(s_{t,j} - lse_t),
// D_t = <dO_t, O_t> and dS = P (<dO_t, v_j> - D_t), for response key j of KV head c:
//   dk_j = scale sum_{h in group(c)} sum_{t >= j} dS_{t,j} q_{t,h}
//   dv_j =       sum_{h in group(c)} sum_{t >= j} P_{t,j} dO_{t,h}
// Only the causal R x R triangle contributes; prompt keys never appear here.
//
// Key-stationary: an iteration pairs one 128-key tile of the response (K, V resident in
// shared memory for its segment) with one 128-token query tile of one query head, and
// computes the transposed tiles, keys on the tensor-memory lanes:
//   S^T  = K Q^T           (SS MMA, M = keys, N = queries, K = head dims)
//   dP^T = V dO^T          (SS)
//   P^T  = exp2(S^T scale log2e - lse2_t),   dS^T = P^T (dP^T - D_t)   (dS warps)
//   dV  += P^T dO          (TS: P^T from tensor memory, dO as an MN-major operand)
//   dK  += dS^T Q          (TS: dS^T from tensor memory, Q as an MN-major operand)
// lse2 = lse log2e and D arrive transposed ([head][token], padded to whole tiles with
// +inf / 0, so rows past R get P = 0 with no mask) from bwd_delta.  Iterations are
// spread over the grid by ls_dkdv.h (equal iteration counts per CTA; a key tile split
// between CTAs leaves partial sums that bwd_dkdv_tc_combine adds in CTA order).
//
// CTA (12 warps): warp 0 TMA producer (K/V per segment, then Q, dO and the 128 lse2 / D
// values of each iteration into a 2-stage ring); warp 1 MMA issuer (one thread); warps
// 4-7 and 8-11 the dS warpgroups, each owning 64 query columns of every key row.  Issue
// order per iteration i: dV(i) once P^T(i) is in tensor memory, then S^T(i+1) (it
// overwrites P^T(i), which dV(i) has read in issue order), dK(i) once dS^T(i) is in,
// then dP^T(i+1) (over dS^T(i)); the dS warps compute P^T(i+1) while dK(i) and dP^T(i+1)
// run.  Tensor memory: S^T [0,128) dP^T [128,256) dV [256,384) dK [384,512); P^T and
// dS^T overlay the first 32 columns of each warpgroup's half of S^T and dP^T.
#include <math.h>

#include "ls_device.cuh"
#include "ls_dkdv.h"
#include "ls_internal.h"
#include "ls_tmap.h"
#include "ls_umma.cuh"

namespace {

using namespace umma;

constexpr int kD = 128;
constexpr int kTile = 128;
constexpr int kThreads = 384;
constexpr int kStages = 2;
// Register split (setmaxnreg) as in the other tcgen05 kernels: control warpgroup 112,
// dS warpgroups 192 (64 P values kept while 64 dP values load): 128 x 112 + 256 x 192 =
// 63488 <= 384 x 168.
constexpr int kRegsLaunch = 168, kRegsControl = 112, kRegsDs = 192;
static_assert(128 * kRegsControl + 256 * kRegsDs <= kThreads * kRegsLaunch, "register split");
constexpr uint32_t kTileBytes = kTile * kD * 2;  // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // 128 rows x 64 dims
constexpr uint32_t kOffK = 0, kOffV = kTileBytes;
constexpr uint32_t kOffStage = 2 * kTileBytes;          // stage s: Q, then dO
constexpr uint32_t kStageBytes = 2 * kTileBytes;
constexpr uint32_t kOffStat = kOffStage + kStages * kStageBytes;  // stage s: lse2[128], D[128]
constexpr uint32_t kStatBytes = 2 * kTile * 4;
constexpr uint32_t kOffBar = kOffStat + kStages * kStatBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 384;

enum {
  B_KV_FULL = 0,
  B_KV_EMPTY,
  B_QD_FULL,                       // per stage
  B_QD_EMPTY = B_QD_FULL + kStages,
  B_S_FULL = B_QD_EMPTY + kStages,
  B_DP_FULL,
  B_P_FULL,
  B_DS_FULL,
  B_ACC_DONE,
  B_ACC_FREE,
  B_DONE,
  B_COUNT
};
static_assert(B_COUNT * 8 + 16 <= 256, "barrier area");

struct TmapSet {
  CUtensorMap q, d_o, kr, vr;
};

struct DkdvArgs {
  int32_t R, hkv, rp;       // rp: R rounded up to whole tiles (stride of lse2t / dt)
  float scale, scale_log2;
  const float* lse2t;       // [hq][rp]: lse log2(e), +inf past R
  const float* dt;          // [hq][rp]: D, 0 past R
  float* dk;                // [R][hkv][128]
  float* dv;
  float* part;              // [2 ctas][2][128][128]: dK, dV partial sums
  int32_t accumulate;
  uint32_t* err;
  LsSegs seg;               // segments of the response (one: a single response)
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + kOffBar + 8 * i; }

__global__ void __launch_bounds__(kThreads, 1)
bwd_dkdv_tc_kernel(const __grid_constant__ TmapSet tm, const __grid_constant__ DkdvArgs a,
                   const __grid_constant__ LsDkdvGeom gm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffBar + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + B_COUNT * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(bar_addr(sbase, B_KV_FULL), 1);
    mbar_init(bar_addr(sbase, B_KV_EMPTY), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_addr(sbase, B_QD_FULL + s), 1);
      mbar_init(bar_addr(sbase, B_QD_EMPTY + s), 1);
    }
    mbar_init(bar_addr(sbase, B_S_FULL), 1);
    mbar_init(bar_addr(sbase, B_DP_FULL), 1);
    mbar_init(bar_addr(sbase, B_P_FULL), 256);
    mbar_init(bar_addr(sbase, B_DS_FULL), 256);
    mbar_init(bar_addr(sbase, B_ACC_DONE), 1);
    mbar_init(bar_addr(sbase, B_ACC_FREE), 256);
    mbar_init(bar_addr(sbase, B_DONE), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&](void) {
    ls_report(a.err, LS_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm.q);
      tma_prefetch_desc(&tm.d_o);
      tma_prefetch_desc(&tm.kr);
      tma_prefetch_desc(&tm.vr);
      LsDkdvWalk w(gm, blockIdx.x);
      LsDkdvIter it;
      uint32_t n = 0, sg = 0;
      while (w.next(&it)) {
        if (it.first) {  // a new key tile: K and V once the last segment's MMAs are done
          if (sg > 0 && !mbar_wait(bar_addr(sbase, B_KV_EMPTY), (sg - 1) & 1)) { fail(); break; }
          if (*abort_flag) break;
          const uint32_t kb = bar_addr(sbase, B_KV_FULL);
          mbar_expect_tx(kb, 2 * kTileBytes);
          for (int hf = 0; hf < 2; ++hf) {
            tma_load_3d(sbase + kOffK + hf * kHalfBytes, &tm.kr, hf * 64, it.kvh, it.kt * kTile, kb);
            tma_load_3d(sbase + kOffV + hf * kHalfBytes, &tm.vr, hf * 64, it.kvh, it.kt * kTile, kb);
          }
          ++sg;
        }
        const uint32_t st = n & 1;
        if (!mbar_wait(bar_addr(sbase, B_QD_EMPTY + st), ((n >> 1) & 1) ^ 1)) { fail(); break; }
        if (*abort_flag) break;
        const uint32_t qb = bar_addr(sbase, B_QD_FULL + st);
        const uint32_t dst = sbase + kOffStage + st * kStageBytes;
        mbar_expect_tx(qb, kStageBytes + kStatBytes);
        for (int hf = 0; hf < 2; ++hf) {
          tma_load_3d(dst + hf * kHalfBytes, &tm.q, hf * 64, it.h, it.tt * kTile, qb);
          tma_load_3d(dst + kTileBytes + hf * kHalfBytes, &tm.d_o, hf * 64, it.h, it.tt * kTile, qb);
        }
        const int64_t so = (int64_t)it.h * a.rp + (int64_t)it.tt * kTile;
        const uint32_t sdst = sbase + kOffStat + st * kStatBytes;
        bulk_load(sdst, a.lse2t + so, kTile * 4, qb);
        bulk_load(sdst + kTile * 4, a.dt + so, kTile * 4, qb);
        ++n;
      }
      // do not leave while copies into this CTA's shared memory may be in flight
      for (uint32_t i = n > kStages ? n - kStages : 0; i < n; ++i)
        mbar_wait(bar_addr(sbase, B_QD_FULL + (i & 1)), (i >> 1) & 1);
      if (sg > 0) mbar_wait(bar_addr(sbase, B_KV_FULL), (sg - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(kTile, kTile, false);
      const uint32_t idG = idesc_bf16_f32(kTile, kD, true);
      const uint32_t k_lo = sdesc_lo(sbase + kOffK, 16), v_lo = sdesc_lo(sbase + kOffV, 16);
      auto q_k = [&](uint32_t st) { return sdesc_lo(sbase + kOffStage + st * kStageBytes, 16); };
      auto do_k = [&](uint32_t st) {
        return sdesc_lo(sbase + kOffStage + st * kStageBytes + kTileBytes, 16);
      };
      auto q_mn = [&](uint32_t st) {
        return sdesc_lo(sbase + kOffStage + st * kStageBytes, kHalfBytes);
      };
      auto do_mn = [&](uint32_t st) {
        return sdesc_lo(sbase + kOffStage + st * kStageBytes + kTileBytes, kHalfBytes);
      };
      // S^T = K Q^T (or dP^T = V dO^T) into tensor-memory columns col
      auto mma_kq = [&](uint32_t a_lo, uint32_t b_lo, uint32_t col, int bar) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_ss_lo(tmem + col, a_lo + off, b_lo + off, idS, kk > 0);
        }
        mma_commit(bar_addr(sbase, bar));
      };
      // acc += X^T B with X^T (P^T or dS^T) in tensor memory at column xcol, B MN-major
      auto mma_acc = [&](uint32_t acc_col, uint32_t xcol, uint32_t b_lo, bool accumulate) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t acol = kk < 4 ? kk * 8 : 64 + (kk - 4) * 8;
          mma_ts_lo(tmem + acc_col, tmem + xcol + acol, b_lo + ((kk * 2048) >> 4), idG,
                    (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      LsDkdvWalk w(gm, blockIdx.x);
      LsDkdvIter cur, nx;
      uint32_t n = 0, sg = 0;
      bool ok = w.next(&cur);
      if (ok) {
        ok = mbar_wait(bar_addr(sbase, B_KV_FULL), 0) && mbar_wait(bar_addr(sbase, B_QD_FULL), 0);
        if (ok) {
          tc_fence_after();
          mma_kq(k_lo, q_k(0), kColS, B_S_FULL);
          mma_kq(v_lo, do_k(0), kColDp, B_DP_FULL);
        } else {
          fail();
        }
      }
      while (ok) {
        const uint32_t st = n & 1, st1 = (n + 1) & 1;
        const bool has = w.next(&nx);
        const bool same = has && !nx.first;
        // a new segment's first dV overwrites the accumulators: the dS warps must have
        // read the last segment's
        if (cur.first && sg > 0 && !mbar_wait(bar_addr(sbase, B_ACC_FREE), (sg - 1) & 1)) { fail(); break; }
        if (!mbar_wait(bar_addr(sbase, B_P_FULL), n & 1)) { fail(); break; }
        tc_fence_after();
        mma_acc(kColDv, kColS, do_mn(st), !cur.first);
        if (same) {
          if (!mbar_wait(bar_addr(sbase, B_QD_FULL + st1), ((n + 1) >> 1) & 1)) { fail(); break; }
          tc_fence_after();
          mma_kq(k_lo, q_k(st1), kColS, B_S_FULL);
        }
        if (!mbar_wait(bar_addr(sbase, B_DS_FULL), n & 1)) { fail(); break; }
        tc_fence_after();
        mma_acc(kColDk, kColDp, q_mn(st), !cur.first);
        mma_commit(bar_addr(sbase, B_QD_EMPTY + st));
        if (cur.last) {
          mma_commit(bar_addr(sbase, B_ACC_DONE));
          mma_commit(bar_addr(sbase, B_KV_EMPTY));
        }
        if (!has) break;
        if (same) {
          mma_kq(v_lo, do_k(st1), kColDp, B_DP_FULL);
        } else {
          ++sg;
          if (!mbar_wait(bar_addr(sbase, B_KV_FULL), sg & 1)) { fail(); break; }
          if (!mbar_wait(bar_addr(sbase, B_QD_FULL + st1), ((n + 1) >> 1) & 1)) { fail(); break; }
          tc_fence_after();
          mma_kq(k_lo, q_k(st1), kColS, B_S_FULL);
          mma_kq(v_lo, do_k(st1), kColDp, B_DP_FULL);
        }
        ++n;
        cur = nx;
      }
      // every MMA this thread issued has finished before tensor memory is released
      mma_commit(bar_addr(sbase, B_DONE));
      mbar_wait(bar_addr(sbase, B_DONE), 0);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDs));
    // ------------------------------------------------------------ dS warpgroups
    const int cgrp = (warp - 4) >> 2;  // query columns [64 cgrp, 64 cgrp + 64)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // key within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c = a.scale_log2;
    const float2 c2 = make_float2(c, c);
    LsDkdvWalk w(gm, blockIdx.x);
    LsDkdvIter it;
    uint32_t n = 0, sg = 0;
    int32_t key_hi = a.R, key_kt = -1;  // end of this row's key's segment (its last query + 1)
    while (w.next(&it)) {
      const uint32_t st = n & 1;
      if (a.seg.n > 1 && it.kt != key_kt) {
        key_kt = it.kt;
        int32_t lo;
        ls_seg_bounds(a.seg, it.kt * kTile + row, &lo, &key_hi);
      }
      const float* lse2 = reinterpret_cast<const float*>(smem + kOffStat + st * kStatBytes) + 64 * cgrp;
      const float* dd = lse2 + kTile;
      if (!mbar_wait(bar_addr(sbase, B_S_FULL), n & 1)) { fail(); break; }
      tc_fence_after();
      const uint32_t s_col = tmem + lane_off + kColS + 64 * cgrp;
      const uint32_t dp_col = tmem + lane_off + kColDp + 64 * cgrp;
      float p[64];
      {
        uint32_t sv[64];
        tmem_ld32(s_col, sv);
        tmem_ld32(s_col + 32, sv + 32);
        tmem_wait_ld();
        reg_fence32(sv);
        reg_fence32(sv + 32);
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), c2,
                                make_float2(-lse2[k], -lse2[k + 1]));
          p[k] = fast_exp2(x.x);
          p[k + 1] = fast_exp2(x.y);
        }
      }
      if (it.tt == it.kt) {  // diagonal tile: query t sees key j only when j <= t
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (64 * cgrp + k < row) p[k] = 0.f;
      }
      if ((it.tt + 1) * kTile > key_hi) {  // queries of later segments do not see this key
        const int32_t q0 = it.tt * kTile + 64 * cgrp;
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (q0 + k >= key_hi) p[k] = 0.f;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = pack_bf16(p[2 * k], p[2 * k + 1]);
        tmem_st32(s_col, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, B_P_FULL));
      if (!mbar_wait(bar_addr(sbase, B_DP_FULL), n & 1)) { fail(); break; }
      tc_fence_after();
      {
        uint32_t dv[64];
        tmem_ld32(dp_col, dv);
        tmem_ld32(dp_col + 32, dv + 32);
        tmem_wait_ld();
        reg_fence32(dv);
        reg_fence32(dv + 32);
        uint32_t ds[32];
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float2 dpm = __fadd2_rn(make_float2(__uint_as_float(dv[k]), __uint_as_float(dv[k + 1])),
                                        make_float2(-dd[k], -dd[k + 1]));
          const float2 x = __fmul2_rn(make_float2(p[k], p[k + 1]), dpm);
          ds[k >> 1] = pack_bf16(x.x, x.y);
        }
        tmem_st32(dp_col, ds);
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, B_DS_FULL));
      ++n;
      if (it.last) {
        // the segment's dK / dV: key row `row`, head dims [64 cgrp, 64 cgrp + 64)
        if (!mbar_wait(bar_addr(sbase, B_ACC_DONE), sg & 1)) { fail(); break; }
        ++sg;
        tc_fence_after();
        const int key = it.kt * kTile + row;
        const bool valid = !it.complete || key < a.R;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {  // 0: dK, 1: dV
          const uint32_t col = tmem + lane_off + (which == 0 ? kColDk : kColDv) + 64 * cgrp;
          const float mul = which == 0 ? a.scale : 1.f;
          float* dst;
          bool acc = false;
          if (it.complete) {
            dst = (which == 0 ? a.dk : a.dv) + ((int64_t)(valid ? key : 0) * a.hkv + it.kvh) * kD + 64 * cgrp;
            acc = a.accumulate != 0;
          } else {
            dst = a.part + (((int64_t)it.slot * 2 + which) * kTile + row) * kD + 64 * cgrp;
          }
#pragma unroll 1
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(col + c0, v);
            tmem_wait_ld();
            reg_fence32(v);
            if (valid) {
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                float4 x = make_float4(__uint_as_float(v[i]) * mul, __uint_as_float(v[i + 1]) * mul,
                                       __uint_as_float(v[i + 2]) * mul, __uint_as_float(v[i + 3]) * mul);
                float4* p4 = reinterpret_cast<float4*>(dst + c0 + i);
                if (acc) {
                  const float4 o = *p4;
                  x.x += o.x; x.y += o.y; x.z += o.z; x.w += o.w;
                }
                *p4 = x;
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bar_addr(sbase, B_ACC_FREE));
      }
      if (*abort_flag) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Key tiles split between CTAs: add the partial sums of their segments in CTA order.
// Grid: (KV head x key tile, 16 groups of 8 keys); 128 threads, one float4 of dK or dV of
// one key each per step.  Blocks of key tiles that one CTA held whole exit at once.
constexpr int kCombineKeys = 8;
__global__ void __launch_bounds__(128) bwd_dkdv_tc_combine(const __grid_constant__ DkdvArgs a,
                                                           const __grid_constant__ LsDkdvGeom gm) {
  const int kvh = blockIdx.x / gm.nT, kt = blockIdx.x % gm.nT;
  const int64_t s = gm.tile_begin(kvh, kt), e = s + gm.tile_iters(kt);
  const int b0 = (int)(s / gm.per_cta), b1 = (int)((e - 1) / gm.per_cta);
  if (b0 == b1) return;
  constexpr int kVec = kD / 4;  // float4 per row
  for (int idx = threadIdx.x; idx < 2 * kCombineKeys * kVec; idx += blockDim.x) {
    const int which = idx / (kCombineKeys * kVec);
    const int r = blockIdx.y * kCombineKeys + (idx / kVec) % kCombineKeys, c4 = idx % kVec;
    const int key = kt * kTile + r;
    if (key >= a.R) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int b = b0; b <= b1; ++b) {
      const float4 x = *reinterpret_cast<const float4*>(
          a.part + (((int64_t)gm.slot(b, s) * 2 + which) * kTile + r) * kD + 4 * c4);
      acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
    }
    float4* dst = reinterpret_cast<float4*>((which == 0 ? a.dk : a.dv) +
                                            ((int64_t)key * a.hkv + kvh) * kD + 4 * c4);
    if (a.accumulate) {
      const float4 o = *dst;
      acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
    }
    *dst = acc;
  }
}

}  // namespace

size_t ls_dkdv_part_bytes(int R, int hq, int hkv, int num_sms, const LsSegs* segs) {
  const LsDkdvGeom gm = ls_make_dkdv_geom(R, hq / hkv, hkv, num_sms, segs);
  return (size_t)2 * gm.ctas * 2 * kTile * kD * sizeof(float);
}

cudaError_t ls_launch_bwd_dkdv(const LsAttnArgs& a, const LsSegs& seg, const LsBwdIn& b,
                               int num_sms, cudaStream_t st) {
  const LsDkdvGeom gm = ls_make_dkdv_geom(a.R, a.g, a.hkv, num_sms, &seg);
  if (gm.total == 0) return cudaSuccess;
  if (seg.n > 1 && !gm.ragged) return cudaErrorInvalidValue;  // checked by the entry point
  TmapSet tm;
  const uint32_t box[3] = {64, 1, kTile};
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)a.hq * kD * 2};
    if (!ls_make_tmap_bf16(&tm.q, a.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.d_o, b.d_o, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)a.hkv * kD * 2};
    if (!ls_make_tmap_bf16(&tm.kr, a.k_resp, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.vr, a.v_resp, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  DkdvArgs d;
  d.R = a.R;
  d.hkv = a.hkv;
  d.rp = gm.nT * kTile;
  d.scale = a.scale;
  d.scale_log2 = a.scale_log2;
  d.lse2t = b.lse2t;
  d.dt = b.dt;
  d.dk = b.dk;
  d.dv = b.dv;
  d.part = b.part_dkdv;
  d.accumulate = b.accumulate;
  d.err = a.err;
  d.seg = seg;
  cudaError_t e =
      cudaFuncSetAttribute(bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  bwd_dkdv_tc_kernel<<<gm.ctas, kThreads, kSmemBytes, st>>>(tm, d, gm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ls_note_launch();
  bool split = false;
  for (int c = 0; c < gm.hkv && !split; ++c)
    for (int kt = 0; kt < gm.nT && !split; ++kt) {
      const int64_t s = gm.tile_begin(c, kt), en = s + gm.tile_iters(kt);
      split = s / gm.per_cta != (en - 1) / gm.per_cta;
    }
  if (split) {
    bwd_dkdv_tc_combine<<<dim3(gm.hkv * gm.nT, kTile / kCombineKeys), 128, 0, st>>>(d, gm);
    e = cudaGetLastError();
    if (e == cudaSuccess) ls_note_launch();
  }
  return e;
}
