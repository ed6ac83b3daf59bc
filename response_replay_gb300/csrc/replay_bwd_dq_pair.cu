// replay_bwd_dq_pair.cu -- dQ of the replay backward on CTA pairs (tcgen05 cta_group::2).
//
// The computation of replay_bwd_dq_tc.cu (LongStraw paper digest, Method, last
// paragraph: the prompt state is stopgrad, so prompt keys feed only dQ):
//   P_{t,j} = exp(s_{t,j} - lse_t),  dS = P (dO v_j - D_t),  dq_t = scale sum_j dS_{t,j} k_j
// over every prompt key and the response keys j <= t, S and P recomputed from the LSE.
//
// Here the two CTAs of a cluster pair share each K/V tile: a unit is 256 rows, 128 per
// CTA, and rank 0 issues every MMA of the pair at M = 256 (each CTA's 128 rows of A and
// of the accumulators in its own shared and tensor memory).  The B operand of an MMA is
// split by its N columns between the two CTAs, so each CTA loads and reads half of each
// K/V tile:
//   S  = Q K^T   B = K, N = keys: CTA c holds keys [64c, 64c + 64) of the tile
//   dP = dO V^T  B = V, N = keys: CTA c holds keys [64c, 64c + 64)
//   dQ += dS K   B = K, N = dims: CTA c holds dims [64c, 64c + 64) of all 128 keys
// Per CTA and 128-key step that is 160 KB of shared-memory traffic (operand reads plus
// TMA fills) instead of 224 KB on one SM, against the SM's 128 bytes per clock.
//
// Roles per CTA (12 warps, as in the one-CTA kernel):
//   warp 0      TMA producer of this CTA's halves (both CTAs); loads complete on rank 0's
//               barriers (.cta_group::2 loads), each producer arriving there once per
//               stage with its own byte count.
//   warp 1      rank 0: the MMA issuer of the pair; commits arrive on both CTAs' barriers.
//               Rank 1: allocates / frees its tensor memory with rank 0.
//   warps 4-11  dS of this CTA's 128 rows (two warpgroups of 64 key columns); each warp
//               reports "S / dP taken" and "dS written" on rank 0's barriers.
// Tensor memory (each CTA, 512 columns): S [0,128), dP0 [128,256), dP1 [256,384),
// dQ [384,512); dS(j) of warpgroup c in columns [64c, 64c+32) of dP buffer j & 1.
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
constexpr int kUnitRows = 2 * kTile;  // one 128-row tile per CTA of the pair
constexpr int kKStages = 3, kVStages = 3;
constexpr int kThreads = 384;
constexpr int kDsWarps = 8;
// Register split as in the one-CTA kernel: 128 x 112 + 256 x 192 = 63488 <= 384 x 168.
constexpr int kRegsLaunch = 168, kRegsControl = 112, kRegsDs = 192;
static_assert(128 * kRegsControl + 256 * kRegsDs <= kThreads * kRegsLaunch, "register split");
constexpr uint32_t kColS = 0, kColDp = 128, kColDq = 384;
constexpr uint32_t kTileBytes = kTile * kD * 2;      // 32 KB: a Q or dO tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;      // 16 KB: 128 rows x 64 dims
constexpr uint32_t kKsBytes = 64 * kD * 2;           // 16 KB: 64 keys x 128 dims (S, dP operand)
constexpr uint32_t kKsHalf = kKsBytes / 2;           // 8 KB: 64 keys x 64 dims
constexpr uint32_t kKdBytes = kTile * 64 * 2;        // 16 KB: 128 keys x 64 dims (dQ operand)
constexpr uint32_t kKStageBytes = kKsBytes + kKdBytes;
constexpr uint32_t kVStageBytes = kKsBytes;
constexpr uint32_t kOffQ = 0, kOffDO = kTileBytes;
constexpr uint32_t kOffK = 2 * kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kKStageBytes;
constexpr uint32_t kOffBar = kOffV + kVStages * kVStageBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr float kLog2e = 1.4426950408889634f;

// Barriers: the *_FULL ones of the loads and the dS warps' reports live in rank 0 (the
// issuer's); the MMA completions arrive in both CTAs at the same offset.
enum {
  B_K_FULL = 0,                     // rank 0: one arrival per CTA + both CTAs' bytes
  B_K_EMPTY = B_K_FULL + kKStages,  // each CTA: the issuer's commit
  B_V_FULL = B_K_EMPTY + kKStages,
  B_V_EMPTY = B_V_FULL + kVStages,
  B_Q_FULL = B_V_EMPTY + kVStages,  // rank 0: one arrival per CTA
  B_Q_EMPTY,
  B_S_FULL,
  B_DP_FULL,                   // 2
  B_SDP_FREE = B_DP_FULL + 2,  // rank 0: one arrival per dS warp of both CTAs
  B_DS_FULL,                   // 2, rank 0: the same
  B_DQ_DONE = B_DS_FULL + 2,
  B_DONE,
  B_AUX,  // each CTA: its own ragged K tile landed
  B_COUNT
};
static_assert(B_COUNT * 8 + 16 <= 256, "barrier area");

struct TmapSet {
  CUtensorMap q, d_o;      // boxes {64, pack, 128 / pack}
  CUtensorMap kp64, vp64;  // prompt pool, boxes {64, min(page, 64)} (S / dP operand halves)
  CUtensorMap kp128;       // prompt pool, box {64, min(page, 128)} (dQ operand)
  CUtensorMap kr64, vr64;  // response K / V, boxes {64, 1, 64}
  CUtensorMap kr128;       // response K, box {64, 1, 128}
};

template <bool kSeg, bool kTb, bool kPk>
using PairCursor = TileCursor<kUnitRows, kTile, kSeg ? 3 : 0, kTb, kPk>;

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + kOffBar + 8 * i; }

template <bool kSeg, bool kTb, bool kPk>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_pair_kernel(const __grid_constant__ TmapSet tm, const LsAttnArgs a,
                   const __grid_constant__ LsSched sc, const LsBwdIn b) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffBar + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + B_COUNT * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0 issues the pair's MMAs
  const int pair = blockIdx.x >> 1;
  // rank 0's barrier i in the cluster window
  auto lead = [&](int i) -> uint32_t { return mapa_shared(bar_addr(sbase, i), 0); };

  if (tid == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(bar_addr(sbase, B_K_FULL + i), 2);
      mbar_init(bar_addr(sbase, B_K_EMPTY + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(bar_addr(sbase, B_V_FULL + i), 2);
      mbar_init(bar_addr(sbase, B_V_EMPTY + i), 1);
    }
    mbar_init(bar_addr(sbase, B_Q_FULL), 2);
    mbar_init(bar_addr(sbase, B_Q_EMPTY), 1);
    mbar_init(bar_addr(sbase, B_S_FULL), 1);
    mbar_init(bar_addr(sbase, B_DP_FULL + 0), 1);
    mbar_init(bar_addr(sbase, B_DP_FULL + 1), 1);
    mbar_init(bar_addr(sbase, B_SDP_FREE), 2 * kDsWarps);
    mbar_init(bar_addr(sbase, B_DS_FULL + 0), 2 * kDsWarps);
    mbar_init(bar_addr(sbase, B_DS_FULL + 1), 2 * kDsWarps);
    mbar_init(bar_addr(sbase, B_DQ_DONE), 1);
    mbar_init(bar_addr(sbase, B_DONE), 1);
    mbar_init(bar_addr(sbase, B_AUX), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish_pair();
  }
  {
    // grouped-query packing: rows of the Q / dO tiles past pack * floor(128 / pack) are
    // never loaded and stay zero
    const int used = a.pack * (kTile / a.pack);
    if (used < kTile) {
      const int per_half = (kTile - used) * 8;
      for (int i = tid; i < 4 * per_half; i += kThreads) {
        const int part = i / per_half, c = i % per_half;
        *reinterpret_cast<uint4*>(smem + kOffQ + part * kHalfBytes + used * 128 + c * 16) =
            make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
    }
  }
  // both CTAs' barriers initialised and tensor memory allocated before either touches
  // the other's
  tc_fence_before();
  cluster_sync();
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
      tma_prefetch_desc(&tm.kp64);
      tma_prefetch_desc(&tm.vp64);
      tma_prefetch_desc(&tm.kp128);
      tma_prefetch_desc(&tm.kr64);
      tma_prefetch_desc(&tm.vr64);
      tma_prefetch_desc(&tm.kr128);
      PairCursor<kSeg, kTb, kPk> cur(sc, pair, a.R, a.g, a.pack);
      TileRec r;
      uint32_t kc = 0, vc = 0, units = 0, aux = 0;
      const int32_t ps = 1 << a.ps_log2;
      const int32_t rows64 = ps < 64 ? ps : 64, rows128 = ps < kTile ? ps : kTile;
      const int32_t pool_rows = a.num_pages * a.hkv * ps;
      const int32_t tpt = kTile / a.pack;
      const int32_t koff = 64 * (int32_t)rank;  // this CTA's keys of a tile (S / dP halves)
      // pool row of prompt position pos of KV head kvh (out of range: zero fill)
      auto pool_row = [&](int32_t pos, int32_t kvh) -> int32_t {
        int32_t y = pool_rows;
        if (pos < a.P) {
          const int32_t phys = __ldg(a.page_table + (pos >> a.ps_log2));
          if ((uint32_t)phys < (uint32_t)a.num_pages)
            y = (phys * a.hkv + kvh) * ps + (pos & (ps - 1));
          else
            ls_report(a.err, LS_DEVERR_CHECK);
        }
        return y;
      };
      bool ok = true;
      while (ok && cur.next(&r)) {
        if (r.first_of_unit) {
          if (units > 0 && !mbar_wait(bar_addr(sbase, B_Q_EMPTY), (units - 1) & 1)) { fail(); break; }
          const uint32_t qb = lead(B_Q_FULL);
          mbar_expect_tx_cluster(qb, 2u * 2u * 128u * (uint32_t)(a.pack * tpt));
          const int32_t t0 = r.t0 + (int32_t)rank * tpt;  // this CTA's tile of the unit
          for (int hf = 0; hf < 2; ++hf) {
            tma_load_3d_pair(sbase + kOffQ + hf * kHalfBytes, &tm.q, hf * 64, r.h, t0, qb);
            tma_load_3d_pair(sbase + kOffDO + hf * kHalfBytes, &tm.d_o, hf * 64, r.h, t0, qb);
          }
          ++units;
        }
        // K: the S operand (this CTA's 64 keys, all dims) and the dQ operand (all 128
        // keys, this CTA's 64 dims).  Rows past a ragged last prompt tile may hold stale
        // page data (even NaN): dS is 0 there but 0 x NaN is not, so such a tile lands on
        // this CTA's own barrier, is cleaned, and is then reported to rank 0.
        {
          const uint32_t st = kc % kKStages;
          if (!mbar_wait(bar_addr(sbase, B_K_EMPTY + st), ((kc / kKStages) & 1) ^ 1)) { fail(); break; }
          if (*abort_flag) break;
          const bool ragged = !r.resp && r.key0 + kTile > a.P;
          const uint32_t fb = ragged ? bar_addr(sbase, B_AUX) : lead(B_K_FULL + st);
          if (ragged)
            mbar_expect_tx(fb, kKStageBytes);
          else
            mbar_expect_tx_cluster(fb, kKStageBytes);
          const uint32_t ks = sbase + kOffK + st * kKStageBytes, kd = ks + kKsBytes;
          if (r.resp) {
            for (int hf = 0; hf < 2; ++hf)
              tma_load_3d_pair(ks + hf * kKsHalf, &tm.kr64, hf * 64, r.kvh, r.key0 + koff, fb);
            tma_load_3d_pair(kd, &tm.kr128, koff, r.kvh, r.key0, fb);
          } else {
            for (int bb = 0; bb < 64 / rows64; ++bb) {
              const int32_t y = pool_row(r.key0 + koff + bb * rows64, r.kvh);
              for (int hf = 0; hf < 2; ++hf)
                tma_load_2d_pair(ks + hf * kKsHalf + bb * rows64 * 128, &tm.kp64, hf * 64, y, fb);
            }
            for (int bb = 0; bb < kTile / rows128; ++bb)
              tma_load_2d_pair(kd + bb * rows128 * 128, &tm.kp128, koff,
                               pool_row(r.key0 + bb * rows128, r.kvh), fb);
          }
          if (ragged) {
            if (!mbar_wait(fb, aux & 1)) { fail(); break; }
            ++aux;
            uint8_t* kb = smem + kOffK + st * kKStageBytes;
            // S operand rows: key key0 + koff + row, row < 64
            for (int row = a.P - r.key0 - koff > 0 ? a.P - r.key0 - koff : 0; row < 64; ++row)
              for (int c = 0; c < 8; ++c) {
                *reinterpret_cast<uint4*>(kb + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(kb + kKsHalf + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
              }
            // dQ operand rows: key key0 + row, row < 128
            for (int row = a.P - r.key0; row < kTile; ++row)
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(kb + kKsBytes + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            mbar_arrive_cluster_release(lead(B_K_FULL + st));
          }
          ++kc;
        }
        // V: this CTA's 64 keys, all dims
        {
          const uint32_t st = vc % kVStages;
          if (!mbar_wait(bar_addr(sbase, B_V_EMPTY + st), ((vc / kVStages) & 1) ^ 1)) { fail(); break; }
          if (*abort_flag) break;
          const uint32_t fb = lead(B_V_FULL + st);
          mbar_expect_tx_cluster(fb, kVStageBytes);
          const uint32_t vs = sbase + kOffV + st * kVStageBytes;
          if (r.resp) {
            for (int hf = 0; hf < 2; ++hf)
              tma_load_3d_pair(vs + hf * kKsHalf, &tm.vr64, hf * 64, r.kvh, r.key0 + koff, fb);
          } else {
            for (int bb = 0; bb < 64 / rows64; ++bb) {
              const int32_t y = pool_row(r.key0 + koff + bb * rows64, r.kvh);
              for (int hf = 0; hf < 2; ++hf)
                tma_load_2d_pair(vs + hf * kKsHalf + bb * rows64 * 128, &tm.vp64, hf * 64, y, fb);
            }
          }
          ++vc;
        }
      }
      // Loads into either CTA complete on rank 0's barriers: rank 0 waits for the last
      // fills of its rings (both CTAs' bytes), and neither CTA leaves before the
      // closing cluster barrier.
      if (rank == 0) {
        for (uint32_t i = kc > kKStages ? kc - kKStages : 0; i < kc; ++i)
          mbar_wait(bar_addr(sbase, B_K_FULL + i % kKStages), (i / kKStages) & 1);
        for (uint32_t i = vc > kVStages ? vc - kVStages : 0; i < vc; ++i)
          mbar_wait(bar_addr(sbase, B_V_FULL + i % kVStages), (i / kVStages) & 1);
        if (units > 0) mbar_wait(bar_addr(sbase, B_Q_FULL), (units - 1) & 1);
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    // The schedule of the one-CTA kernel: per tile j, settle the loads of tile j+1, then
    // once both CTAs' dS warps hold S(j) and dP(j) in registers issue S(j+1) and dP(j+1),
    // then once dS(j) is in both CTAs' tensor memory issue dQ(j).
    if (lane == 0) {
      const uint32_t idQK = idesc_bf16_f32(kUnitRows, kTile, false);
      const uint32_t idDQ = idesc_bf16_f32(kUnitRows, kD, true);
      const uint32_t dq_base = sdesc_lo(sbase + kOffQ, 16);
      const uint32_t ddo_base = sdesc_lo(sbase + kOffDO, 16);
      const uint32_t dks_base = sdesc_lo(sbase + kOffK, 16);
      const uint32_t dvs_base = sdesc_lo(sbase + kOffV, 16);
      // dQ operand: MN-major, one 64-dim block per CTA (LBO unused)
      const uint32_t dkd_base = sdesc_lo(sbase + kOffK + kKsBytes, kKdBytes);
      PairCursor<kSeg, kTb, kPk> cursor(sc, pair, a.R, a.g, a.pack);
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
      auto mma_s = [&](uint32_t st, bool last_of_unit) {
        const uint32_t b0 = dks_base + ((st * kKStageBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          const uint32_t boff = ((kk >> 2) * kKsHalf + (kk & 3) * 32) >> 4;
          mma_ss_pair(tmem + kColS, dq_base + aoff, b0 + boff, idQK, kk > 0);
        }
        mma_commit_pair(bar_addr(sbase, B_S_FULL));
        if (last_of_unit) mma_commit_pair(bar_addr(sbase, B_Q_EMPTY));
      };
      auto mma_dp = [&](uint32_t st, uint32_t db) {
        const uint32_t b0 = dvs_base + ((st * kVStageBytes) >> 4);
        const uint32_t d = tmem + kColDp + db * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          const uint32_t boff = ((kk >> 2) * kKsHalf + (kk & 3) * 32) >> 4;
          mma_ss_pair(d, ddo_base + aoff, b0 + boff, idQK, kk > 0);
        }
        mma_commit_pair(bar_addr(sbase, B_DP_FULL + db));
        mma_commit_pair(bar_addr(sbase, B_V_EMPTY + st));
      };
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
        const uint32_t bq = dkd_base + ((kq.stage * kKStageBytes) >> 4);
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
        mma_ts_pair(tmem + kColDq, aq, bq, idDQ, f0 ? 0u : 1u);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk) {
          const uint32_t acol = kk < 4 ? kk * 8 : 64 + (kk - 4) * 8;
          mma_ts_pair(tmem + kColDq, aq + acol, bq + ((kk * 2048) >> 4), idDQ, 1u);
        }
        mma_commit_pair(bar_addr(sbase, B_K_EMPTY + kq.stage));
        if (l0) mma_commit_pair(bar_addr(sbase, B_DQ_DONE));
        kq.advance();
        f0 = f1;
        l0 = l1;
        have0 = have1;
        have1 = have1 && cursor.next_flags(&f1, &l1);
        ++j;
      }
      mma_commit_pair(bar_addr(sbase, B_DONE));
      mbar_wait(bar_addr(sbase, B_DONE), 0);
    }
  } else if (warp == 1) {
    // rank 1: every MMA that wrote this CTA's tensor memory has finished
    if (lane == 0) mbar_wait(bar_addr(sbase, B_DONE), 0);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDs));
    // ------------------------------------------------------------ dS warpgroups
    const int cgrp = (warp - 4) >> 2;  // key columns [64 cgrp, 64 cgrp + 64)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c = a.scale_log2;
    const int32_t tpt = kTile / a.pack;
    // this thread's row: token (rank * tpt + row / pack) of the unit, head row % pack
    const int32_t tok_off = (int32_t)rank * tpt + row / a.pack, head_off = row % a.pack;
    const bool row_used = row < a.pack * tpt;
    const uint32_t sdp_free = lead(B_SDP_FREE);
    const uint32_t ds_full[2] = {lead(B_DS_FULL), lead(B_DS_FULL + 1)};
    PairCursor<kSeg, kTb, kPk> cursor(sc, pair, a.R, a.g, a.pack);
    TileRec r;
    uint32_t j = 0, uc = 0;
    float lse2 = 0.f, dd = 0.f;
    int32_t row_lo = 0;
    while (cursor.next(&r)) {
      const int32_t tq = r.t0 + tok_off;
      const int32_t hrow = row_used ? r.h + head_off : r.h;
      if (r.first_of_unit) {
        const int64_t idx = (int64_t)(tq < a.R ? tq : a.R - 1) * a.hq + hrow;
        lse2 = b.lse[idx] * kLog2e;
        dd = b.delta[idx];
        if constexpr (kSeg) {
          int32_t hi;
          ls_seg_bounds(sc.seg, tq < a.R ? tq : a.R - 1, &row_lo, &hi);
        }
      }
      const uint32_t db = j & 1;
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
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(sdp_free);
      const float2 c2 = make_float2(c, c), nl2 = make_float2(-lse2, -lse2);
      const float2 nd2 = make_float2(-dd, -dd);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int col0 = 64 * cgrp + 32 * q;
        float d2[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int e = 32 * q + i;
          float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nl2);
          x.x = fast_exp2(x.x);
          x.y = fast_exp2(x.y);
          const float2 dpm = __fadd2_rn(make_float2(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), nd2);
          const float2 ds2 = __fmul2_rn(x, dpm);
          d2[i] = ds2.x;
          d2[i + 1] = ds2.y;
        }
        if (col0 + 32 > lim || col0 < lo) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col0 + i >= lim || col0 + i < lo) d2[i] = 0.f;
        }
        uint32_t ds[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) ds[i >> 1] = pack_bf16(d2[i], d2[i + 1]);
        tmem_st16(dp_col + 16 * q, ds);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(db ? ds_full[1] : ds_full[0]);
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
          dst = b.part_dq + ((int64_t)r.slot * kUnitRows + rank * kTile + row) * kD;
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
  __syncwarp();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Sum the partial dQ of the pieces of each tail unit in piece order.
// Grid: (tail units, row groups of kCombineRows); one thread per head_dim column.
constexpr int kCombineRows = 8;
__global__ void __launch_bounds__(kD) bwd_dq_pair_combine(const LsAttnArgs a, const LsSched sc,
                                                          const LsBwdIn b) {
  const int tu = blockIdx.x, T = sc.tail_units, Q = sc.pieces;
  const int u = sc.tail_unit0() + tu;
  const int tpt = kTile / a.pack, tok_per_unit = 2 * tpt;
  const int nTB = (a.R + tok_per_unit - 1) / tok_per_unit;
  int grp, tb;
  unit_coords(u, a.hq / a.pack, nTB, sc.tb_major != 0, &grp, &tb);
  const int t0 = tb * tok_per_unit;
  const int h0 = grp * a.pack;
  const int col = threadIdx.x;
  for (int r = blockIdx.y * kCombineRows; r < (blockIdx.y + 1) * kCombineRows; ++r) {
    const int l = r % kTile;  // row within its CTA's tile
    if (l >= a.pack * tpt) continue;
    const int t = t0 + (r / kTile) * tpt + l / a.pack, h = h0 + l % a.pack;
    if (t >= a.R) continue;
    float acc = 0.f;
    for (int k = 0; k < Q; ++k) acc += b.part_dq[((int64_t)(k * T + tu) * kUnitRows + r) * kD + col];
    float* dst = b.dq + ((int64_t)t * a.hq + h) * kD + col;
    *dst = b.accumulate ? *dst + acc : acc;
  }
}

const void* pair_kernel(bool seg, bool tb, bool pk) {
  const void* const fns[8] = {
      (const void*)bwd_dq_pair_kernel<false, false, false>,
      (const void*)bwd_dq_pair_kernel<false, false, true>,
      (const void*)bwd_dq_pair_kernel<false, true, false>,
      (const void*)bwd_dq_pair_kernel<false, true, true>,
      (const void*)bwd_dq_pair_kernel<true, false, false>,
      (const void*)bwd_dq_pair_kernel<true, false, true>,
      (const void*)bwd_dq_pair_kernel<true, true, false>,
      (const void*)bwd_dq_pair_kernel<true, true, true>};
  return fns[(seg ? 4 : 0) + (tb ? 2 : 0) + (pk ? 1 : 0)];
}

// Tiles of a unit of two 128-row tiles for a pack (pack heads x floor(128 / pack) tokens
// per tile): the pack with the fewest units, ties to the larger pack except that one
// head per tile wins any tie.
int64_t pair_units_for(int R, int hq, int pack) {
  const int tpu = 2 * (kTile / pack);
  return (int64_t)(hq / pack) * ((R + tpu - 1) / tpu);
}
}  // namespace

int ls_bwd_pair_unit_rows() { return kUnitRows; }
int ls_bwd_pair_pack(int R, int hq, int hkv) {
  const int g = hq / hkv;
  int best = 1;
  int64_t bu = INT64_MAX;
  for (int p = g < 64 ? g : 64; p >= 2; --p) {
    if (g % p) continue;
    const int64_t u = pair_units_for(R, hq, p);
    if (u < bu) {
      best = p;
      bu = u;
    }
  }
  return pair_units_for(R, hq, 1) <= bu ? 1 : best;
}
int ls_bwd_pair_units(int R, int hq, int hkv) {
  return (int)pair_units_for(R, hq, ls_bwd_pair_pack(R, hq, hkv));
}

// Pairs that fit on the device at once (one CTA per SM, both SMs of a pair in one
// cluster): the persistent grid's size.
cudaError_t ls_bwd_pair_workers(int* pairs) {
  const void* fn = pair_kernel(false, false, false);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  int sms = 0, dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms & ~1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
  if (e != cudaSuccess) return e;
  *pairs = n;
  return n > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t ls_launch_bwd_dq_pair(const LsAttnArgs& a, const LsSched& sc, const LsBwdIn& b,
                                  cudaStream_t st) {
  TmapSet tm;
  const int ps = 1 << a.ps_log2;
  {
    const uint32_t box[3] = {64, (uint32_t)a.pack, (uint32_t)(kTile / a.pack)};
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)a.hq * kD * 2};
    if (!ls_make_tmap_bf16(&tm.q, a.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.d_o, b.d_o, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint32_t box64[3] = {64, 1, 64}, box128[3] = {64, 1, kTile};
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)a.R};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)a.hkv * kD * 2};
    if (!ls_make_tmap_bf16(&tm.kr64, a.k_resp, 3, dims, strides, box64)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.vr64, a.v_resp, 3, dims, strides, box64)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.kr128, a.k_resp, 3, dims, strides, box128)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.num_pages * a.hkv * ps};
    const uint64_t strides[1] = {(uint64_t)kD * 2};
    const uint32_t box64[2] = {64, (uint32_t)(ps < 64 ? ps : 64)};
    const uint32_t box128[2] = {64, (uint32_t)(ps < kTile ? ps : kTile)};
    if (!ls_make_tmap_bf16(&tm.kp64, a.k_pool, 2, dims, strides, box64)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.vp64, a.v_pool, 2, dims, strides, box64)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.kp128, a.k_pool, 2, dims, strides, box128)) return cudaErrorInvalidValue;
  }
  const void* fn = pair_kernel(sc.seg.n > 1, sc.tb_major != 0, a.pack > 1);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * sc.ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {(void*)&tm, (void*)&a, (void*)&sc, (void*)&b};
  e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ls_note_launch();
  if (sc.has_partials()) {
    bwd_dq_pair_combine<<<dim3((unsigned)sc.tail_units, kUnitRows / kCombineRows), kD, 0, st>>>(a, sc, b);
    e = cudaGetLastError();
    if (e == cudaSuccess) ls_note_launch();
  }
  return e;
}
