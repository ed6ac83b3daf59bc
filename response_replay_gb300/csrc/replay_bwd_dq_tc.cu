// replay_bwd_dq_tc.cu -- dQ of the replay backward on the 5th-generation tensor cores.
//
// With the prompt state stopgrad (LongStraw paper digest, Method, last paragraph),
// the prompt keys feed only dQ:
//   P_{t,j} = exp(s_{t,j} - lse_t),  dP_{t,j} = <dO_t, v_j>,  dS = P (dP - D_t),
//   dq_t = scale * sum_j dS_{t,j} k_j    over every prompt key and response keys j <= t.
// S and P are recomputed from the forward's LSE (storing P would need ~400 GB at
// 2M positions); D = <dO, O> comes from bwd_delta.
//
// CTA (one per SM, persistent, 12 warps) owns a unit = 128 consecutive response tokens
// of one query head; Q and dO stay in shared memory while K/V tiles stream past:
//   warp 0      TMA producer: Q and dO tiles, then K (4-stage ring) and V (one stage)
//               tiles of 128 keys, prompt tiles gathered page by page; rows of a ragged
//               last prompt K tile are zeroed before the tile is handed over.  V is read
//               only by dP, early in a tile, so one stage refills in time; K lives from
//               S(j) to dQ(j) and its load lead decides whether S waits (measured: 4 K /
//               1 V stages 1% faster than 3 / 2, 2 / 3 30% slower).
//   warp 1      MMA issuer (one thread; with warp 2 for token-block-major launches, see
//               issue_two): S = Q K^T (SS), dP = dO V^T (SS, into one of two
//               dP buffers), dQ += dS K (TS: dS from tensor memory, K as an MN-major
//               operand).  Per tile j: dP(j+1) once V(j+1) has landed; S(j+1) once the
//               dS warps hold S(j) and dP(j) in registers (both run while dS(j) is
//               computed); dQ(j) once dS(j) is in tensor memory.  Every wait sits behind
//               a group that is still running.  A K tile lives from S(j) to dQ(j), so the
//               4-stage ring gives each K load about three tiles of lead.
//   warps 2-3   idle (complete warpgroup 0; warp 2 issues S in token-block-major launches)
//   warps 4-7 / 8-11  two warpgroups split the 128 key columns of each query row (64
//               each): p = exp2(s scale log2e - lse log2e), ds = p (dp - D), packed as
//               bf16 pairs over their own dP columns; at the end of a unit they read dQ,
//               scale it and write dq (or a split partial).
// Tensor memory (512 columns): S [0,128), dP0 [128,256), dP1 [256,384), dQ [384,512).
// dS(j) of warpgroup c lives in columns [64c, 64c+32) of dP buffer j & 1.
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"
#include "ls_tiles.cuh"
#include "ls_tmap.h"
#include "ls_umma.cuh"

namespace {

using namespace umma;

constexpr int kD = 128;
constexpr int kTile = 128;
constexpr int kUnitRows = 128;
constexpr int kKStages = 4, kVStages = 1;
constexpr int kThreads = 384;
// Register split (setmaxnreg): the launch gives 168 per thread (384 x 168 = 64512);
// warpgroup 0 (TMA + MMA control) drops to 112 and the dS warpgroups (64 S and 64 dP
// values per thread held at once) rise to 192: 128 x 112 + 256 x 192 = 63488 <= 64512.
constexpr int kRegsLaunch = 168, kRegsControl = 112, kRegsDs = 192;
static_assert(128 * kRegsControl + 256 * kRegsDs <= kThreads * kRegsLaunch, "register split");
// Tensor memory columns: S, two dP buffers (dS(j) is written over dP(j)), dQ.
constexpr uint32_t kColS = 0, kColDp = 128, kColDq = 384;
constexpr uint32_t kTileBytes = kTile * kD * 2;
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr uint32_t kOffQ = 0, kOffDO = kTileBytes;
constexpr uint32_t kOffK = 2 * kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
constexpr float kLog2e = 1.4426950408889634f;

enum {
  B_K_FULL = 0,
  B_K_EMPTY = B_K_FULL + kKStages,
  B_V_FULL = B_K_EMPTY + kKStages,
  B_V_EMPTY = B_V_FULL + kVStages,
  B_Q_FULL = B_V_EMPTY + kVStages,
  B_Q_EMPTY,
  B_S_FULL,
  B_DP_FULL,   // 2: dP(j) in dP buffer j & 1
  B_SDP_FREE = B_DP_FULL + 2,  // the dS warps hold S(j) and dP(j) in registers
  B_DS_FULL,   // 2: dS(j) in dP buffer j & 1
  B_DQ_DONE = B_DS_FULL + 2,
  B_DONE,
  B_AUX,  // producer: ragged K tile landed
  B_COUNT
};
static_assert(B_COUNT * 8 + 16 <= 256, "barrier area");

struct TmapSet {
  CUtensorMap q, d_o, kp, vp, kr, vr;
};

// kSeg: one response cut into segments (ragged members back to back); kTb: units
// numbered token block major (short prompts)
template <bool kSeg, bool kTb, bool kPk>
using DqCursor = TileCursor<kUnitRows, kTile, kSeg ? 3 : 0, kTb, kPk>;

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + kOffBar + 8 * i; }

// The MMA issue of token-block-major launches on two threads (lane 0 of warps 1 and 2):
//   warp 2  S(j) = Q K^T, once the dS warps hold S(j-1) in registers;
//   warp 1  dP(j+1) = dO V^T, then dQ(j) += dS(j) K once dS(j) is in tensor memory.
// The threads' MMAs use disjoint tensor memory (S vs the dP buffers and dQ), so the only
// order between them is the one the dS warps' barriers give.  The unit's Q / dO are free
// once both its last S and its last dP are done (two arrivals), and both threads commit
// to B_DONE before tensor memory is released.
template <bool kSeg, bool kPk, typename Fail>
__device__ __forceinline__ void issue_two(int warp, uint32_t sbase, uint32_t tmem,
                                          const LsSched& sc, const LsAttnArgs& a, Fail fail) {
  const uint32_t idQK = idesc_bf16_f32(kTile, kTile, false);
  const uint32_t idDQ = idesc_bf16_f32(kTile, kD, true);
  DqCursor<kSeg, true, kPk> cursor(sc, blockIdx.x, a.R, a.g, a.pack);
  uint32_t qunits = 0;
  auto wait_q = [&]() -> bool {
    const bool w = mbar_wait(bar_addr(sbase, B_Q_FULL), qunits & 1);
    ++qunits;
    return w;
  };
  if (warp == 2) {
    const uint32_t dq_base = sdesc_lo(sbase + kOffQ, 16);
    const uint32_t dk_base = sdesc_lo(sbase + kOffK, 16);
    RingPos<kKStages> ks;
    bool f = false, l = false;
    uint32_t j = 0;
    while (cursor.next_flags(&f, &l)) {
      if (f && !wait_q()) { fail(); break; }
      if (!mbar_wait(bar_addr(sbase, B_K_FULL + ks.stage), ks.phase)) { fail(); break; }
      // S has one buffer: S(j) overwrites S(j-1) once the dS warps hold it
      if (j > 0 && !mbar_wait(bar_addr(sbase, B_SDP_FREE), (j - 1) & 1)) { fail(); break; }
      tc_fence_after();
      const uint32_t b0 = dk_base + ((ks.stage * kTileBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
        mma_ss_lo(tmem + kColS, dq_base + off, b0 + off, idQK, kk > 0);
      }
      mma_commit(bar_addr(sbase, B_S_FULL));
      if (l) mma_commit(bar_addr(sbase, B_Q_EMPTY));  // the unit's Q is free
      ks.advance();
      ++j;
    }
  } else {
    const uint32_t ddo_base = sdesc_lo(sbase + kOffDO, 16);
    const uint32_t dv_base = sdesc_lo(sbase + kOffV, 16);
    const uint32_t dkm_base = sdesc_lo(sbase + kOffK, kHalfBytes);
    bool f0 = false, l0 = false, f1 = false, l1 = false;
    bool have0 = cursor.next_flags(&f0, &l0);
    bool have1 = have0 && cursor.next_flags(&f1, &l1);
    RingPos<kKStages> kq;
    RingPos<kVStages> vs;
    uint32_t j = 0;
    bool ok = true;
    // dP into buffer db from V stage st; the unit's dO is free after its last dP
    auto mma_dp = [&](uint32_t st, uint32_t db, bool last_of_unit) {
      const uint32_t b0 = dv_base + ((st * kTileBytes) >> 4);
      const uint32_t d = tmem + kColDp + db * kTile;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
        mma_ss_lo(d, ddo_base + off, b0 + off, idQK, kk > 0);
      }
      mma_commit(bar_addr(sbase, B_DP_FULL + db));
      mma_commit(bar_addr(sbase, B_V_EMPTY + st));
      if (last_of_unit) mma_commit(bar_addr(sbase, B_Q_EMPTY));
    };
    if (have0) {
      ok = wait_q() && mbar_wait(bar_addr(sbase, B_V_FULL + vs.stage), vs.phase);
      if (ok) {
        tc_fence_after();
        mma_dp(vs.stage, 0, l0);
        vs.advance();
      } else {
        fail();
      }
    }
    while (ok && have0) {
      // dP(j+1) needs V(j+1) (its buffer's previous dS(j-1) went to dQ(j-1), issued before
      // it by this thread); dQ(j) needs dS(j) (K(j) landed before S(j) ran)
      if (have1) {
        if (f1 && !wait_q()) { fail(); break; }
        if (!mbar_wait(bar_addr(sbase, B_V_FULL + vs.stage), vs.phase)) { fail(); break; }
        tc_fence_after();
        mma_dp(vs.stage, (j + 1) & 1, l1);
        vs.advance();
      }
      if (!mbar_wait(bar_addr(sbase, B_DS_FULL + (j & 1)), (j >> 1) & 1)) { fail(); break; }
      if (!mbar_wait(bar_addr(sbase, B_K_FULL + kq.stage), kq.phase)) { fail(); break; }
      tc_fence_after();
      const uint32_t bq = dkm_base + ((kq.stage * kTileBytes) >> 4);
      const uint32_t aq = tmem + kColDp + (j & 1) * kTile;  // dS(j)
      mma_ts_lo(tmem + kColDq, aq, bq, idDQ, f0 ? 0u : 1u);
#pragma unroll
      for (int kk = 1; kk < 8; ++kk) {
        const uint32_t acol = kk < 4 ? kk * 8 : 64 + (kk - 4) * 8;
        mma_ts_lo(tmem + kColDq, aq + acol, bq + ((kk * 2048) >> 4), idDQ, 1u);
      }
      mma_commit(bar_addr(sbase, B_K_EMPTY + kq.stage));
      if (l0) mma_commit(bar_addr(sbase, B_DQ_DONE));
      kq.advance();
      f0 = f1;
      l0 = l1;
      have0 = have1;
      have1 = have1 && cursor.next_flags(&f1, &l1);
      ++j;
    }
  }
  // every MMA this thread issued has finished before tensor memory is released
  mma_commit(bar_addr(sbase, B_DONE));
  mbar_wait(bar_addr(sbase, B_DONE), 0);
}

template <bool kSeg, bool kTb, bool kPk>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_tc_kernel(const __grid_constant__ TmapSet tm, const LsAttnArgs a,
                 const __grid_constant__ LsSched sc, const LsBwdIn b) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffBar + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + B_COUNT * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(bar_addr(sbase, B_K_FULL + i), 1);
      mbar_init(bar_addr(sbase, B_K_EMPTY + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(bar_addr(sbase, B_V_FULL + i), 1);
      mbar_init(bar_addr(sbase, B_V_EMPTY + i), 1);
    }
    mbar_init(bar_addr(sbase, B_Q_FULL), 1);
    mbar_init(bar_addr(sbase, B_Q_EMPTY), kTb ? 2 : 1);  // the unit's last S (and last dP)
    mbar_init(bar_addr(sbase, B_S_FULL), 1);
    mbar_init(bar_addr(sbase, B_DP_FULL + 0), 1);
    mbar_init(bar_addr(sbase, B_DP_FULL + 1), 1);
    mbar_init(bar_addr(sbase, B_SDP_FREE), 256);
    mbar_init(bar_addr(sbase, B_DS_FULL + 0), 256);
    mbar_init(bar_addr(sbase, B_DS_FULL + 1), 256);
    mbar_init(bar_addr(sbase, B_DQ_DONE), 1);
    mbar_init(bar_addr(sbase, B_DONE), kTb ? 2 : 1);     // one commit per MMA issuer
    mbar_init(bar_addr(sbase, B_AUX), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  {
    // With grouped-query packing a tile holds pack * floor(128 / pack) rows; the rest of
    // the Q and dO tiles are never loaded and stay zero (their outputs are never written).
    const int used = a.pack * (kTile / a.pack);
    if (used < kTile) {
      const int per_half = (kTile - used) * 8;  // 16-byte chunks
      for (int i = tid; i < 4 * per_half; i += kThreads) {
        const int part = i / per_half, c = i % per_half;  // Q / dO x two halves
        *reinterpret_cast<uint4*>(smem + kOffQ + part * kHalfBytes + used * 128 + c * 16) =
            make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
    }
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
      tma_prefetch_desc(&tm.kp);
      tma_prefetch_desc(&tm.vp);
      tma_prefetch_desc(&tm.kr);
      tma_prefetch_desc(&tm.vr);
      DqCursor<kSeg, kTb, kPk> cur(sc, blockIdx.x, a.R, a.g, a.pack);
      TileRec r;
      uint32_t kc = 0, vc = 0, units = 0, aux = 0;
      const int32_t ps = 1 << a.ps_log2;
      const int32_t box_rows = ps < kTile ? ps : kTile;
      const int32_t pool_rows = a.num_pages * a.hkv * ps;
      bool ok = true;
      while (ok && cur.next(&r)) {
        if (r.first_of_unit) {
          if (units > 0 && !mbar_wait(bar_addr(sbase, B_Q_EMPTY), (units - 1) & 1)) { fail(); break; }
          // the tile holds floor(128 / pack) tokens x pack heads (pack = 1: 128 tokens)
          const uint32_t qb = bar_addr(sbase, B_Q_FULL);
          mbar_expect_tx(qb, 2u * 2u * 128u * (uint32_t)(a.pack * (kTile / a.pack)));
          for (int hf = 0; hf < 2; ++hf) {
            tma_load_3d(sbase + kOffQ + hf * kHalfBytes, &tm.q, hf * 64, r.h, r.t0, qb);
            tma_load_3d(sbase + kOffDO + hf * kHalfBytes, &tm.d_o, hf * 64, r.h, r.t0, qb);
          }
          ++units;
        }
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t cnt = kv == 0 ? kc : vc;
          const int nst = kv == 0 ? kKStages : kVStages;
          const uint32_t st = cnt % nst;
          const int be = (kv == 0 ? B_K_EMPTY : B_V_EMPTY) + st;
          const int bf = (kv == 0 ? B_K_FULL : B_V_FULL) + st;
          if (!mbar_wait(bar_addr(sbase, be), ((cnt / nst) & 1) ^ 1)) { fail(); ok = false; break; }
          if (*abort_flag) { ok = false; break; }
          // K rows past the end of a ragged last prompt tile may hold stale page data
          // (even NaN); their dS is 0 but 0 x NaN is not, so they are zeroed before
          // the tile is handed to the MMA issuer.
          const bool ragged_k = kv == 0 && !r.resp && r.key0 + kTile > a.P;
          const uint32_t fb = bar_addr(sbase, ragged_k ? (int)B_AUX : bf);
          const uint32_t dst = sbase + (kv == 0 ? kOffK : kOffV) + st * kTileBytes;
          mbar_expect_tx(fb, kTileBytes);
          if (r.resp) {
            const void* map = kv == 0 ? (const void*)&tm.kr : (const void*)&tm.vr;
            for (int hf = 0; hf < 2; ++hf) tma_load_3d(dst + hf * kHalfBytes, map, hf * 64, r.kvh, r.key0, fb);
          } else {
            const void* map = kv == 0 ? (const void*)&tm.kp : (const void*)&tm.vp;
            for (int bb = 0; bb < kTile / box_rows; ++bb) {
              const int32_t pos = r.key0 + bb * box_rows;
              int32_t y = pool_rows;
              if (pos < a.P) {
                const int32_t phys = __ldg(a.page_table + (pos >> a.ps_log2));
                if ((uint32_t)phys < (uint32_t)a.num_pages)
                  y = (phys * a.hkv + r.kvh) * ps + (pos & (ps - 1));
                else
                  ls_report(a.err, LS_DEVERR_CHECK);
              }
              for (int hf = 0; hf < 2; ++hf)
                tma_load_2d(dst + hf * kHalfBytes + bb * box_rows * 128, map, hf * 64, y, fb);
            }
          }
          if (ragged_k) {
            if (!mbar_wait(fb, aux & 1)) { fail(); ok = false; break; }
            ++aux;
            uint8_t* kb = smem + kOffK + st * kTileBytes;
            for (int i = (int)(a.P - r.key0) * 8; i < kTile * 8; ++i) {
              const int row = i >> 3, c = i & 7;
              *reinterpret_cast<uint4*>(kb + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(kb + kHalfBytes + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar_addr(sbase, bf));
          }
          if (kv == 0) ++kc; else ++vc;
        }
      }
      for (uint32_t i = kc > kKStages ? kc - kKStages : 0; i < kc; ++i)
        mbar_wait(bar_addr(sbase, B_K_FULL + i % kKStages), (i / kKStages) & 1);
      for (uint32_t i = vc > kVStages ? vc - kVStages : 0; i < vc; ++i)
        mbar_wait(bar_addr(sbase, B_V_FULL + i % kVStages), (i / kVStages) & 1);
      if (units > 0) mbar_wait(bar_addr(sbase, B_Q_FULL), (units - 1) & 1);
    }
  } else if (warp == 1 || (kTb && warp == 2)) {
    // ------------------------------------------------------------ MMA issuers
    // Issuing a tcgen05.mma holds the thread until the tensor core has nearly taken the
    // instruction (it runs about one MMA ahead of its issuer), so nothing but MMAs may sit
    // between groups of one issuing thread.
    //  * Token-block-major launches (short prompts, long causal items): two threads issue,
    //    warp 2 the S groups and warp 1 dP and dQ, so each one's waits and commits are
    //    covered by the other's MMAs (P = 0, R = 8,192: 1.27 -> 1.17 ms).
    //  * Otherwise one thread, per tile j: settle the loads of tile j+1, then as soon as
    //    the dS warps hold S(j) and dP(j) in registers issue S(j+1) and dP(j+1) (they run
    //    while dS(j) is computed), then once dS(j) is in tensor memory issue dQ(j).  Two
    //    threads measured 8% slower here: S then interleaves with dQ and delays the
    //    chain S -> dS -> dQ.
    if constexpr (kTb) {
      if (lane == 0) issue_two<kSeg, kPk>(warp, sbase, tmem, sc, a, [&]() { fail(); });
    } else {
      if (lane == 0) {
        const uint32_t idQK = idesc_bf16_f32(kTile, kTile, false);
        const uint32_t idDQ = idesc_bf16_f32(kTile, kD, true);
        const uint32_t dq_base = sdesc_lo(sbase + kOffQ, 16);
        const uint32_t ddo_base = sdesc_lo(sbase + kOffDO, 16);
        const uint32_t dk_base = sdesc_lo(sbase + kOffK, 16);
        const uint32_t dv_base = sdesc_lo(sbase + kOffV, 16);
        const uint32_t dkm_base = sdesc_lo(sbase + kOffK, kHalfBytes);
        DqCursor<kSeg, kTb, kPk> cursor(sc, blockIdx.x, a.R, a.g, a.pack);
        // first / last of unit of tiles j (f0, l0) and j+1 (f1, l1)
        bool f0 = false, l0 = false, f1 = false, l1 = false;
        bool have0 = cursor.next_flags(&f0, &l0);
        bool have1 = have0 && cursor.next_flags(&f1, &l1);
        RingPos<kKStages> ks, kq;  // K ring: next S, next dQ
        RingPos<kVStages> vs;      // V ring: next dP
        uint32_t qunits = 0, j = 0;
        bool ok = true;
        auto wait_q = [&]() -> bool {
          const bool w = mbar_wait(bar_addr(sbase, B_Q_FULL), qunits & 1);
          ++qunits;
          return w;
        };
        // S = Q K^T from K stage st
        auto mma_s = [&](uint32_t st, bool last_of_unit) {
          const uint32_t b0 = dk_base + ((st * kTileBytes) >> 4);
  #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
            mma_ss_lo(tmem + kColS, dq_base + off, b0 + off, idQK, kk > 0);
          }
          mma_commit(bar_addr(sbase, B_S_FULL));
          // the unit's Q and dO are free once its last S (issued after its last dP) is done
          if (last_of_unit) mma_commit(bar_addr(sbase, B_Q_EMPTY));
        };
        // dP = dO V^T into dP buffer db from V stage st
        auto mma_dp = [&](uint32_t st, uint32_t db) {
          const uint32_t b0 = dv_base + ((st * kTileBytes) >> 4);
          const uint32_t d = tmem + kColDp + db * kTile;
  #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
            mma_ss_lo(d, ddo_base + off, b0 + off, idQK, kk > 0);
          }
          mma_commit(bar_addr(sbase, B_DP_FULL + db));
          mma_commit(bar_addr(sbase, B_V_EMPTY + st));
        };
        // prologue: S(0), dP(0)
        if (have0) {
          ok = wait_q() && mbar_wait(bar_addr(sbase, B_K_FULL + ks.stage), ks.phase) &&
               mbar_wait(bar_addr(sbase, B_V_FULL + vs.stage), vs.phase);
          if (ok) {
            tc_fence_after();
            mma_dp(vs.stage, 0);
            mma_s(ks.stage, l0);
            ks.advance();
            vs.advance();
          } else {
            fail();
          }
        }
        while (ok && have0) {
          // Groups of tile j+1 and j, each wait placed so that the group before it is
          // still running on the tensor core:
          //   dP(j+1) needs V(j+1) (its buffer's previous dS(j-1) went to dQ(j-1), issued
          //     earlier by this thread); a new unit's dO also needs that unit's Q/dO load,
          //     which follows the old unit's last S;
          //   S(j+1) needs K(j+1) and the dS warps to hold S(j) in registers;
          //   dQ(j) needs dS(j).
          const uint32_t bq = dkm_base + ((kq.stage * kTileBytes) >> 4);
          const uint32_t aq = tmem + kColDp + (j & 1) * kTile;  // dS(j)
          if (have1) {
            if (f1 && !wait_q()) { fail(); break; }
            if (!mbar_wait(bar_addr(sbase, B_V_FULL + vs.stage), vs.phase)) { fail(); break; }
            tc_fence_after();
            mma_dp(vs.stage, (j + 1) & 1);
            vs.advance();
            if (!mbar_wait(bar_addr(sbase, B_K_FULL + ks.stage), ks.phase)) { fail(); break; }
          }
          if (!mbar_wait(bar_addr(sbase, B_SDP_FREE), j & 1)) { fail(); break; }
          tc_fence_after();
          if (have1) {
            mma_s(ks.stage, l1);
            ks.advance();
          }
          if (!mbar_wait(bar_addr(sbase, B_DS_FULL + (j & 1)), (j >> 1) & 1)) { fail(); break; }
          tc_fence_after();
          mma_ts_lo(tmem + kColDq, aq, bq, idDQ, f0 ? 0u : 1u);
  #pragma unroll
          for (int kk = 1; kk < 8; ++kk) {
            const uint32_t acol = kk < 4 ? kk * 8 : 64 + (kk - 4) * 8;
            mma_ts_lo(tmem + kColDq, aq + acol, bq + ((kk * 2048) >> 4), idDQ, 1u);
          }
          mma_commit(bar_addr(sbase, B_K_EMPTY + kq.stage));
          if (l0) mma_commit(bar_addr(sbase, B_DQ_DONE));
          kq.advance();
          f0 = f1;
          l0 = l1;
          have0 = have1;
          have1 = have1 && cursor.next_flags(&f1, &l1);
          ++j;
        }
        mma_commit(bar_addr(sbase, B_DONE));
        mbar_wait(bar_addr(sbase, B_DONE), 0);
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDs));
    // ------------------------------------------------------------ dS warpgroups
    const int cgrp = (warp - 4) >> 2;       // key columns [64 cgrp, 64 cgrp + 64)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c = a.scale_log2;
    // this thread's row: token row / pack of the unit, head row % pack
    const int32_t tok_off = row / a.pack, head_off = row % a.pack;
    const bool row_used = row < a.pack * (kTile / a.pack);
    DqCursor<kSeg, kTb, kPk> cursor(sc, blockIdx.x, a.R, a.g, a.pack);
    TileRec r;
    uint32_t j = 0, uc = 0;
    float lse2 = 0.f, dd = 0.f;
    int32_t row_lo = 0;  // first response key this row's token may see (segments)
    while (cursor.next(&r)) {
      const int32_t tq = r.t0 + tok_off;
      const int32_t hrow = row_used ? r.h + head_off : r.h;
      if (r.first_of_unit) {
        const int64_t idx = (int64_t)(tq < a.R ? tq : a.R - 1) * a.hq + hrow;
        lse2 = b.lse[idx] * kLog2e;
        dd = b.delta[idx];
        if constexpr (kSeg) {
          int32_t hi;
          ls_seg_bounds(sc.seg, tq, &row_lo, &hi);
        }
      }
      const uint32_t db = j & 1;  // dP buffer of tile j; dS(j) is written over it
      if (!mbar_wait(bar_addr(sbase, B_S_FULL), j & 1)) { fail(); break; }
      if (!mbar_wait(bar_addr(sbase, B_DP_FULL + db), (j >> 1) & 1)) { fail(); break; }
      tc_fence_after();
      int32_t lim = kTile, lo = 0;  // keys [key0 + lo, key0 + lim) visible
      if (r.resp) {
        const int32_t lr = (tq + 1 < a.R ? tq + 1 : a.R) - r.key0;
        lim = lr < kTile ? lr : kTile;
        if constexpr (kSeg) lo = row_lo - r.key0;
      } else if (r.key0 + kTile > a.P) {
        lim = (int32_t)(a.P - r.key0);
      }
      // take S(j) and this warpgroup's dP(j) columns into registers, then let the MMA
      // issuer start S(j+1) and dP(j+1) while dS(j) is computed
      const uint32_t dp_col = tmem + lane_off + kColDp + db * kTile + 64 * cgrp;
      uint32_t sv[64], pv[64];
      tmem_ld32(tmem + lane_off + kColS + 64 * cgrp, sv);
      tmem_ld32(tmem + lane_off + kColS + 64 * cgrp + 32, sv + 32);
      tmem_ld32(dp_col, pv);
      tmem_ld32(dp_col + 32, pv + 32);
      tmem_wait_ld();
      reg_fence32(sv);
      reg_fence32(sv + 32);
      reg_fence32(pv);
      reg_fence32(pv + 32);
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, B_SDP_FREE));
      const float2 c2 = make_float2(c, c), nl2 = make_float2(-lse2, -lse2);
      const float2 nd2 = make_float2(-dd, -dd);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int col0 = 64 * cgrp + 32 * q;
        float d2[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {  // packed fp32x2 arithmetic
          const int e = 32 * q + i;
          float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nl2);
          x.x = fast_exp2(x.x);
          x.y = fast_exp2(x.y);
          const float2 dpm = __fadd2_rn(make_float2(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), nd2);
          const float2 ds2 = __fmul2_rn(x, dpm);
          d2[i] = ds2.x;
          d2[i + 1] = ds2.y;
        }
        if (col0 + 32 > lim || col0 < lo) {  // ragged prompt tail, diagonal, segment start
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col0 + i >= lim || col0 + i < lo) d2[i] = 0.f;
        }
        uint32_t ds[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) ds[i >> 1] = pack_bf16(d2[i], d2[i + 1]);
        // dS of keys [64 cgrp, 64 cgrp + 64) as bf16 pairs in this warpgroup's own
        // (already read) dP columns [64 cgrp, 64 cgrp + 32)
        tmem_st16(dp_col + 16 * q, ds);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, B_DS_FULL + db));
      ++j;
      if (r.last_of_unit) {
        if (!mbar_wait(bar_addr(sbase, B_DQ_DONE), uc & 1)) { fail(); break; }
        ++uc;
        tc_fence_after();
        const bool valid = row_used && tq < a.R;
        float* dst;
        bool acc = false;
        if (r.complete) {
          dst = b.dq + ((int64_t)(valid ? tq : 0) * a.hq + hrow) * kD;
          acc = b.accumulate != 0;
        } else {
          dst = b.part_dq + ((int64_t)r.slot * kUnitRows + row) * kD;
        }
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
          const int col0 = 64 * cgrp + 32 * q;
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + kColDq + col0, v);
          tmem_wait_ld();
          reg_fence32(v);
          if (valid || !r.complete) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              float4 x = make_float4(__uint_as_float(v[i]) * a.scale, __uint_as_float(v[i + 1]) * a.scale,
                                     __uint_as_float(v[i + 2]) * a.scale, __uint_as_float(v[i + 3]) * a.scale);
              float4* p4 = reinterpret_cast<float4*>(dst + col0 + i);
              if (acc) {
                const float4 o = *p4;
                x.x += o.x; x.y += o.y; x.z += o.z; x.w += o.w;
              }
              *p4 = x;
            }
          }
        }
        tc_fence_before();
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

// Sum the partial dQ of the pieces of each tail unit in piece order.
// Grid: (tail units, row groups of kCombineRows); one thread per head_dim column.
constexpr int kCombineRows = 8;
__global__ void __launch_bounds__(kD) bwd_dq_tc_combine(const LsAttnArgs a, const LsSched sc,
                                                        const LsBwdIn b) {
  const int tu = blockIdx.x, T = sc.tail_units, Q = sc.pieces;
  const int u = sc.tail_unit0() + tu;
  const int tok_per_unit = kTile / a.pack;
  const int nTB = (a.R + tok_per_unit - 1) / tok_per_unit;
  int grp, tb;
  unit_coords(u, a.hq / a.pack, nTB, sc.tb_major != 0, &grp, &tb);
  const int t0 = tb * tok_per_unit;
  const int h0 = grp * a.pack;
  const int col = threadIdx.x;
  for (int r = blockIdx.y * kCombineRows; r < (blockIdx.y + 1) * kCombineRows; ++r) {
    if (r >= a.pack * tok_per_unit) continue;
    const int t = t0 + r / a.pack, h = h0 + r % a.pack;
    if (t >= a.R) continue;
    float acc = 0.f;
    for (int k = 0; k < Q; ++k) acc += b.part_dq[((int64_t)(k * T + tu) * kUnitRows + r) * kD + col];
    float* dst = b.dq + ((int64_t)t * a.hq + h) * kD + col;
    *dst = b.accumulate ? *dst + acc : acc;
  }
}
}  // namespace

int ls_bwd_unit_rows() { return kUnitRows; }
// Responses shorter than a unit: a tile holds `pack` query heads of one KV head (pack
// dividing g) for floor(128 / pack) tokens; the pack with the fewest tiles, ties to the
// larger pack except that one head per tile wins any tie.
namespace {
int64_t bwd_tiles_for(int R, int hq, int pack) {
  const int tpt = kTile / pack;
  return (int64_t)(hq / pack) * ((R + tpt - 1) / tpt);
}
}  // namespace
int ls_bwd_pack(int R, int hq, int hkv) {
  const int g = hq / hkv;
  int best = 1;
  int64_t bt = INT64_MAX;
  for (int p = g < 64 ? g : 64; p >= 2; --p) {
    if (g % p) continue;
    const int64_t t = bwd_tiles_for(R, hq, p);
    if (t < bt) {
      best = p;
      bt = t;
    }
  }
  return bwd_tiles_for(R, hq, 1) <= bt ? 1 : best;
}
int ls_bwd_units(int R, int hq, int hkv) {
  const int pack = ls_bwd_pack(R, hq, hkv);
  const int tok_per_unit = kTile / pack;
  return (hq / pack) * ((R + tok_per_unit - 1) / tok_per_unit);
}
int ls_bwd_tile() { return kTile; }
int ls_bwd_ctas_per_sm() { return 1; }

cudaError_t ls_launch_bwd_dq(const LsAttnArgs& a, const LsSched& sc, const LsBwdIn& b,
                             cudaStream_t st) {
  TmapSet tm;
  const uint32_t box_q[3] = {64, 1, kTile};
  // Q and dO boxes: 128 tokens of one head, or floor(128 / pack) tokens x pack heads
  const uint32_t box_qp[3] = {64, (uint32_t)a.pack, (uint32_t)(kTile / a.pack)};
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)a.hq * kD * 2};
    if (!ls_make_tmap_bf16(&tm.q, a.q, 3, dims, strides, box_qp)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.d_o, b.d_o, 3, dims, strides, box_qp)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)a.hkv * kD * 2};
    if (!ls_make_tmap_bf16(&tm.kr, a.k_resp, 3, dims, strides, box_q)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.vr, a.v_resp, 3, dims, strides, box_q)) return cudaErrorInvalidValue;
  }
  {
    const int ps = 1 << a.ps_log2;
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.num_pages * a.hkv * ps};
    const uint64_t strides[1] = {(uint64_t)kD * 2};
    const uint32_t box[2] = {64, (uint32_t)(ps < kTile ? ps : kTile)};
    if (!ls_make_tmap_bf16(&tm.kp, a.k_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.vp, a.v_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const bool seg = sc.seg.n > 1, tb = sc.tb_major != 0, pk = a.pack > 1;
  const void* const fns[8] = {
      (const void*)bwd_dq_tc_kernel<false, false, false>,
      (const void*)bwd_dq_tc_kernel<false, false, true>,
      (const void*)bwd_dq_tc_kernel<false, true, false>,
      (const void*)bwd_dq_tc_kernel<false, true, true>,
      (const void*)bwd_dq_tc_kernel<true, false, false>,
      (const void*)bwd_dq_tc_kernel<true, false, true>,
      (const void*)bwd_dq_tc_kernel<true, true, false>,
      (const void*)bwd_dq_tc_kernel<true, true, true>};
  const void* fn = fns[(seg ? 4 : 0) + (tb ? 2 : 0) + (pk ? 1 : 0)];
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&tm, (void*)&a, (void*)&sc, (void*)&b};
  e = cudaLaunchKernel(fn, dim3(sc.ctas), dim3(kThreads), args, kSmemBytes, st);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ls_note_launch();
  if (sc.has_partials()) {
    bwd_dq_tc_combine<<<dim3((unsigned)sc.tail_units, kUnitRows / kCombineRows), kD, 0, st>>>(a, sc, b);
    e = cudaGetLastError();
    if (e == cudaSuccess) ls_note_launch();
  }
  return e;
}
