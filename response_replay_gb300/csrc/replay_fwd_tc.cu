// replay_fwd_tc.cu -- replay attention forward on the 5th-generation tensor cores.
//
// Definition (LongStraw explainer, "Serial replay makes G a schedule" and "Two
// incompatible architectures", Qwen bullet; paper digest, Method step 3):
//   s_{t,j} = scale <q_{t,h}, k_{j,h/g}>,  j over every prompt position and response j <= t
//   lse_t = log sum_j exp(s_{t,j}),  o_t = sum_j exp(s_{t,j} - lse_t) v_j
// Prompt splits are merged on chip by the online-softmax rescaling when one CTA runs
// them back to back, and by log-sum-exp in replay_fwd_tc_combine otherwise.
//
// CTA (one per SM, persistent, 12 warps) owns a unit = 256 consecutive response tokens
// of one query head, as two 128-row tiles A and B that share every K/V tile:
//   warp 0      TMA producer: Q tiles, then K and V tiles (128 keys x 128 dims, two
//               128-byte-swizzled halves each) into a 5-stage ring; prompt tiles are
//               gathered page by page through the page table.
//   warps 1, 2  MMA issuers, one thread each, for tile A and tile B: S_t = Q_t K^T into
//               tensor memory (SS MMA, M=128 N=128 K=128), O_t += P_t V with P_t read
//               from tensor memory (TS MMA); the two tiles' MMAs interleave on the tensor
//               core, so it has one tile's work while the other tile's softmax runs.
//   warp 3      idle (it completes warpgroup 0, whose registers go to the softmax)
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: each thread owns one
//               query row; reads its S row from tensor memory, masks, updates the
//               running max (log2 domain; O is rescaled only when the max grows by more
//               than 2^8) and the compensated row sum, writes P as bf16 pairs back over
//               its S columns, and at the end of a unit normalises O and writes O / LSE.
// Tensor memory (512 columns): S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512);
// P_t overlays the first 64 columns of S_t.
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"
#include "ls_tiles.cuh"
#include "ls_tmap.h"
#include "ls_umma.cuh"

namespace {

using namespace umma;

constexpr int kD = 128;
constexpr int kTile = 128;                 // query rows per tile, keys per KV tile
constexpr int kUnitRows = 2 * kTile;       // tokens per unit
constexpr int kStages = 5;
constexpr int kThreads = 384;
// Register split (setmaxnreg): the launch gives 168 per thread (384 x 168 = 64512);
// warpgroup 0 (TMA + MMA control) drops to 112 and the two softmax warpgroups (a full
// 128-column S row per thread) rise to 192: 128 x 112 + 256 x 192 = 63488 <= 64512.
constexpr int kRegsLaunch = 168, kRegsControl = 112, kRegsSoftmax = 192;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
// The packed-members layout (member masks in the softmax) spills at 192; it takes 200 and
// leaves 96 to the control warps: 128 x 96 + 256 x 200 = 63488.
template <int kMode> constexpr int regs_control() { return kMode == 2 ? 96 : kRegsControl; }
template <int kMode> constexpr int regs_softmax() { return kMode == 2 ? 200 : kRegsSoftmax; }
static_assert(128 * 96 + 256 * 200 <= kThreads * kRegsLaunch, "register split (members)");
constexpr uint32_t kTileBytes = kTile * kD * 2;  // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // 16 KB: 128 rows x 64 dims
constexpr uint32_t kOffQ = 0;                    // Q_A, Q_B
constexpr uint32_t kOffRing = 2 * kTileBytes;
constexpr uint32_t kOffBar = kOffRing + kStages * kTileBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

// barrier indices (8 bytes each from kOffBar)
enum {
  B_KV_FULL = 0,
  B_KV_EMPTY = B_KV_FULL + kStages,
  B_Q_FULL = B_KV_EMPTY + kStages,
  B_Q_EMPTY,
  B_S_FULL,          // 2
  B_P_FULL = B_S_FULL + 2,   // 4: tile t, key half hf at 2 t + hf
  B_O_DONE = B_P_FULL + 4,
  B_DONE = B_O_DONE + 2,   // 2
  B_AUX = B_DONE + 2,      // producer: ragged V tile landed
  B_PV_DONE,               // 2: P_t V of a tile finished (orders the issuers)
  B_COUNT = B_PV_DONE + 2
};
static_assert(B_COUNT * 8 + 16 <= 256, "barrier area");

struct TmapSet {
  CUtensorMap q, kp, vp, kr, vr;
};

template <int kMode, bool kTb, bool kPk>
using FwdCursor = TileCursor<kUnitRows, kTile, kMode, kTb, kPk>;

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + kOffBar + 8 * i; }

// kMode (the unit layouts of ls_tiles.cuh): 0 one response; 1 several responses of
// equal length, units per member (4-D Q and response maps); 2 several responses packed
// into shared tiles (Q as one token sequence, 4-D response maps, rows masked by member);
// 3 one response cut into segments (ragged members back to back, rows masked by segment).
// kTb: units numbered token block major (short prompts; ls_tiles.cuh unit_coords);
// kPk: tiles hold a.pack > 1 heads (grouped-query packing).
template <int kMode, bool kTb, bool kPk>
__global__ void __launch_bounds__(kThreads, 1)
replay_fwd_tc_kernel(const __grid_constant__ TmapSet tm, const LsAttnArgs a,
                     const __grid_constant__ LsSched sc, const LsFwdOut out) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffBar + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + B_COUNT * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_addr(sbase, B_KV_FULL + i), 1);
      mbar_init(bar_addr(sbase, B_KV_EMPTY + i), a.tiles);  // one commit per issuer
    }
    mbar_init(bar_addr(sbase, B_Q_FULL), 1);
    mbar_init(bar_addr(sbase, B_Q_EMPTY), a.tiles);
    mbar_init(bar_addr(sbase, B_AUX), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_addr(sbase, B_S_FULL + t), 1);
      mbar_init(bar_addr(sbase, B_P_FULL + 2 * t), kTile);
      mbar_init(bar_addr(sbase, B_P_FULL + 2 * t + 1), kTile);
      mbar_init(bar_addr(sbase, B_O_DONE + t), 1);
      mbar_init(bar_addr(sbase, B_DONE + t), 1);
      mbar_init(bar_addr(sbase, B_PV_DONE + t), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  {
    // With grouped-query packing a Q tile holds pack * floor(128 / pack) rows; the rest
    // are never loaded and stay zero (their outputs are never written).
    const int used = a.pack * (kTile / a.pack);
    if (used < kTile) {
      const int per_half = (kTile - used) * 8;  // 16-byte chunks
      for (int i = tid; i < 4 * per_half; i += kThreads) {
        const int part = i / per_half, c = i % per_half;  // part = tile * 2 + half
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
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(regs_control<kMode>()));
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm.q);
      tma_prefetch_desc(&tm.kp);
      tma_prefetch_desc(&tm.vp);
      tma_prefetch_desc(&tm.kr);
      tma_prefetch_desc(&tm.vr);
      FwdCursor<kMode, kTb, kPk> cur(sc, blockIdx.x, a.R, a.g, a.pack, a.tiles, a.upm, a.rt);
      TileRec r;
      uint32_t ring = 0, units = 0, aux = 0;
      const int32_t ps = 1 << a.ps_log2;
      const int32_t box_rows = ps < kTile ? ps : kTile;
      const int32_t pool_rows = a.num_pages * a.hkv * ps;
      bool ok = true;
      while (ok && cur.next(&r)) {
        if (r.first_of_unit) {
          if (units > 0 && !mbar_wait(bar_addr(sbase, B_Q_EMPTY), (units - 1) & 1)) { fail(); break; }
          // a tile holds tpt tokens x pack heads (pack = 1: 128 tokens of one head)
          const uint32_t qb = bar_addr(sbase, B_Q_FULL);
          const int32_t tpt = kTile / a.pack;
          mbar_expect_tx(qb, (uint32_t)a.tiles * 2u * 128u * (uint32_t)(a.pack * tpt));
          for (int tt = 0; tt < a.tiles; ++tt)
            for (int hf = 0; hf < 2; ++hf)
              if constexpr (kMode == 1)
                tma_load_4d(sbase + kOffQ + tt * kTileBytes + hf * kHalfBytes, &tm.q, hf * 64,
                            r.h, r.t0 + tt * tpt, r.m, qb);
              else
                tma_load_3d(sbase + kOffQ + tt * kTileBytes + hf * kHalfBytes, &tm.q, hf * 64,
                            r.h, r.t0 + tt * tpt, qb);
          ++units;
        }
        for (int kv = 0; kv < 2 && ok; ++kv) {
          const uint32_t st = ring % kStages;
          if (!mbar_wait(bar_addr(sbase, B_KV_EMPTY + st), ((ring / kStages) & 1) ^ 1)) {
            fail();
            ok = false;
            break;
          }
          if (*abort_flag) { ok = false; break; }
          // The last prompt tile may end inside a page whose later slots hold stale data
          // (even NaN); P is 0 there but 0 x NaN is not, so those V rows are zeroed
          // before the tile is handed to the MMA issuers.
          const bool ragged_v = kv == 1 && !r.resp && r.key0 + kTile > a.P;
          const uint32_t fb = bar_addr(sbase, ragged_v ? B_AUX : B_KV_FULL + st);
          const uint32_t dst = sbase + kOffRing + st * kTileBytes;
          mbar_expect_tx(fb, kTileBytes);
          if (r.resp) {
            const void* map = kv == 0 ? (const void*)&tm.kr : (const void*)&tm.vr;
            int32_t rmem = r.m, key = r.key0;
            if constexpr (kMode == 2)
              packed_resp_tile<kTile>(r.key0, r.t0 / a.R, a.R, &rmem, &key);
            for (int hf = 0; hf < 2; ++hf)
              if constexpr (kMode == 1 || kMode == 2)
                tma_load_4d(dst + hf * kHalfBytes, map, hf * 64, r.kvh, key, rmem, fb);
              else
                tma_load_3d(dst + hf * kHalfBytes, map, hf * 64, r.kvh, key, fb);
          } else {
            const void* map = kv == 0 ? (const void*)&tm.kp : (const void*)&tm.vp;
            for (int b = 0; b < kTile / box_rows; ++b) {
              const int32_t pos = r.key0 + b * box_rows;
              int32_t y = pool_rows;  // out of bounds: zero fill
              if (pos < a.P) {
                const int32_t phys = __ldg(a.page_table + (pos >> a.ps_log2));
                if ((uint32_t)phys < (uint32_t)a.num_pages)
                  y = (phys * a.hkv + r.kvh) * ps + (pos & (ps - 1));
                else
                  ls_report(a.err, LS_DEVERR_CHECK);
              }
              for (int hf = 0; hf < 2; ++hf)
                tma_load_2d(dst + hf * kHalfBytes + b * box_rows * 128, map, hf * 64, y, fb);
            }
          }
          if (ragged_v) {
            if (!mbar_wait(fb, aux & 1)) { fail(); ok = false; break; }
            ++aux;
            uint8_t* vb = smem + kOffRing + st * kTileBytes;
            for (int i = (int)(a.P - r.key0) * 8; i < kTile * 8; ++i) {
              const int row = i >> 3, c = i & 7;
              *reinterpret_cast<uint4*>(vb + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(vb + kHalfBytes + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar_addr(sbase, B_KV_FULL + st));
          }
          ++ring;
        }
      }
      // Do not leave while loads into this CTA's shared memory may still be in flight.
      for (uint32_t i = ring > kStages ? ring - kStages : 0; i < ring; ++i)
        mbar_wait(bar_addr(sbase, B_KV_FULL + i % kStages), (i / kStages) & 1);
      if (units > 0) mbar_wait(bar_addr(sbase, B_Q_FULL), (units - 1) & 1);
    }
  } else if (warp == 1 || (warp == 2 && a.tiles == 2)) {
    // ------------------------------------------------------------ MMA issuers
    // One thread per tile: warp 1 drives tile A, warp 2 tile B.  A tcgen05.mma issue
    // stalls the issuing thread while the tensor core's queue is full, so a single
    // thread driving both tiles could not take up one tile's finished P while it sat in
    // the other tile's issue; with one thread per tile each tile's S -> softmax -> P V
    // loop runs on its own and the two interleave on the tensor core.
    if (lane == 0) {
      const int t = warp - 1;
      const uint32_t idS = idesc_bf16_f32(kTile, kTile, false);
      const uint32_t idPV = idesc_bf16_f32(kTile, kD, true);
      // Descriptor bases built once; every MMA below only adds a compile-time offset
      // (descriptor start addresses are in 16-byte units in the low bits).
      const uint32_t dq = sdesc_lo(sbase + kOffQ + t * kTileBytes, 16);
      const uint32_t dk_base = sdesc_lo(sbase + kOffRing, 16);
      const uint32_t dv_base = sdesc_lo(sbase + kOffRing, kHalfBytes);
      const uint32_t d_s = tmem + t * kTile, d_o = tmem + 256 + t * kTile;
      auto issue_s = [&](uint32_t kstage) {
        const uint32_t b0 = dk_base + ((kstage * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_ss_lo(d_s, dq + off, b0 + off, idS, kk > 0);
        }
      };
      // P_t V over keys [64 hf, 64 hf + 64): K steps 4 hf .. 4 hf + 3
      auto issue_pv_half = [&](uint32_t vstage, int hf, bool accumulate) {
        const uint32_t b0 = dv_base + ((vstage * kTileBytes) >> 4);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * hf + k4;
          mma_ts_lo(d_o, d_s + kk * 8, b0 + ((kk * 2048) >> 4), idPV,
                    (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      FwdCursor<kMode, kTb, kPk> cursor(sc, blockIdx.x, a.R, a.g, a.pack, a.tiles, a.upm, a.rt);
      TileRec cur, nxt;
      uint32_t ring = 0, units = 0, kc = 0;
      bool ok = cursor.next(&cur);
      // S_t of the first tile
      if (ok) {
        if (!mbar_wait(bar_addr(sbase, B_Q_FULL), units & 1)) { fail(); ok = false; }
        ++units;
        const uint32_t kstage = ring % kStages;
        if (ok && !mbar_wait(bar_addr(sbase, B_KV_FULL + kstage), (ring / kStages) & 1)) { fail(); ok = false; }
        ++ring;
        if (ok) {
          tc_fence_after();
          issue_s(kstage);
          mma_commit(bar_addr(sbase, B_S_FULL + t));
          mma_commit(bar_addr(sbase, B_KV_EMPTY + kstage));
          if (cur.last_of_unit) mma_commit(bar_addr(sbase, B_Q_EMPTY));
        }
      }
      while (ok) {
        const bool has_nxt = cursor.next(&nxt);
        // Loads first, then the one real dependency (P_t), then the MMAs back to back:
        // V of this tile, and K of the next one unless that tile opens a new unit (its
        // K is loaded only after the new unit's Q, which waits for this unit's last S).
        const uint32_t vstage = ring % kStages, vpar = (ring / kStages) & 1;
        const uint32_t kstage = (ring + 1) % kStages, kpar = ((ring + 1) / kStages) & 1;
        ring += has_nxt ? 2 : 1;
        const bool early_k = has_nxt && !nxt.first_of_unit;
        if (!mbar_wait(bar_addr(sbase, B_KV_FULL + vstage), vpar)) { fail(); break; }
        if (early_k && !mbar_wait(bar_addr(sbase, B_KV_FULL + kstage), kpar)) { fail(); break; }
        // first half of P_t (keys [0,64)); the softmax still works on the second
        if (!mbar_wait(bar_addr(sbase, B_P_FULL + 2 * t), kc & 1)) { fail(); break; }
        // Keep the tiles half a period apart: tile B's group for tile k follows tile A's
        // P V of tile k, tile A's group for tile k follows tile B's P V of tile k - 1.
        // Each group then lands in the tensor core's queue while the other tile's S is
        // still running, and each tile's softmax overlaps the other tile's MMAs instead
        // of both softmax warpgroups contending for the exp2 units at the same time.
        if (t == 1 && !mbar_wait(bar_addr(sbase, B_PV_DONE + 0), kc & 1)) { fail(); break; }
        if (t == 0 && kc > 0 && a.tiles == 2 &&
            !mbar_wait(bar_addr(sbase, B_PV_DONE + 1), (kc - 1) & 1)) { fail(); break; }
        tc_fence_after();
        issue_pv_half(vstage, 0, !cur.first_of_unit);
        if (!mbar_wait(bar_addr(sbase, B_P_FULL + 2 * t + 1), kc & 1)) { fail(); break; }
        ++kc;
        tc_fence_after();
        issue_pv_half(vstage, 1, true);
        mma_commit(bar_addr(sbase, B_PV_DONE + t));
        if (cur.last_of_unit) mma_commit(bar_addr(sbase, B_O_DONE + t));
        mma_commit(bar_addr(sbase, B_KV_EMPTY + vstage));
        if (!has_nxt) break;
        // S_t of the next tile (after P_t V in issue order: it overwrites P_t)
        if (!early_k) {
          if (!mbar_wait(bar_addr(sbase, B_Q_FULL), units & 1)) { fail(); break; }
          ++units;
          if (!mbar_wait(bar_addr(sbase, B_KV_FULL + kstage), kpar)) { fail(); break; }
          tc_fence_after();
        }
        issue_s(kstage);
        mma_commit(bar_addr(sbase, B_S_FULL + t));
        mma_commit(bar_addr(sbase, B_KV_EMPTY + kstage));
        if (nxt.last_of_unit) mma_commit(bar_addr(sbase, B_Q_EMPTY));
        cur = nxt;
      }
      // every MMA this thread issued has finished before tensor memory is released
      mma_commit(bar_addr(sbase, B_DONE + t));
      mbar_wait(bar_addr(sbase, B_DONE + t), 0);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(regs_softmax<kMode>()));
    // ------------------------------------------------------------ softmax warpgroups
    const int t = (warp - 4) >> 2;         // tile A (0) or B (1)
    const bool tile_used = t < a.tiles;    // one-tile units leave tile B's warps idle
    const int quad = warp & 3;             // tensor-memory lane quadrant of this warp
    const int row = quad * 32 + lane;      // query row within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_col = tmem + lane_off + t * kTile;
    const uint32_t o_col = tmem + lane_off + 256 + t * kTile;
    const float c = a.scale_log2;
    // this thread's row within a tile: token row / pack of the tile, head row % pack
    const int32_t tpt = kTile / a.pack;
    const int32_t tok_off = t * tpt + row / a.pack, head_off = row % a.pack;
    const bool row_used = row < a.pack * tpt;
    FwdCursor<kMode, kTb, kPk> cursor(sc, blockIdx.x, a.R, a.g, a.pack, a.tiles, a.upm, a.rt);
    TileRec r;
    uint32_t kc = 0, oc = 0;
    float m = -INFINITY, l = 0.f, lcomp = 0.f;
    // kMode 2: this row's member and the unit's first member, for the unit at row_t0
    int32_t row_t0 = -1, row_m = 0, row_um = 0;
    while (tile_used && cursor.next(&r)) {
      if (!mbar_wait(bar_addr(sbase, B_S_FULL + t), kc & 1)) { fail(); break; }
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld32(s_col + 0, sr);
      tmem_ld32(s_col + 32, sr + 32);
      tmem_ld32(s_col + 64, sr + 64);
      tmem_ld32(s_col + 96, sr + 96);
      tmem_wait_ld();
      reg_fence32(sr);
      reg_fence32(sr + 32);
      reg_fence32(sr + 64);
      reg_fence32(sr + 96);
      // this row's token: in kMode 2 a number in the members' joint sequence, split
      // into its member and the token within that member's response
      const int32_t vt = r.t0 + tok_off;
      int32_t tq = vt, rmem = 0, unit_m = 0;
      if constexpr (kMode == 2) {
        if (r.t0 != row_t0) {  // once per unit, not per tile
          row_t0 = r.t0;
          row_m = vt / a.R;
          row_um = r.t0 / a.R;
        }
        rmem = row_m;
        unit_m = row_um;
        tq = vt - rmem * a.R;
      }
      int32_t lim = kTile, lo = 0;                  // keys [key0 + lo, key0 + lim) visible
      if (r.resp) {
        int32_t km = 0, key0 = r.key0;              // member and first key of the tile
        if constexpr (kMode == 2) packed_resp_tile<kTile>(r.key0, unit_m, a.R, &km, &key0);
        const int32_t lr = (tq + 1 < a.R ? tq + 1 : a.R) - key0;
        lim = lr < kTile ? lr : kTile;
        if (kMode == 2 && rmem != km) lim = 0;      // another member's keys
        if constexpr (kMode == 3) {                 // keys of earlier segments (ragged
          int32_t s0, s1;                           // members: response tiles only)
          ls_seg_bounds(sc.seg, vt, &s0, &s1);
          lo = s0 - key0;
        }
      } else if (r.key0 + kTile > a.P) {
        lim = (int32_t)(a.P - r.key0);
      }
      if (lim < kTile || lo > 0) {  // the ragged prompt tail, the diagonal, segment starts
        const int32_t l0 = lo > 0 ? lo : 0, l1 = lim > l0 ? lim : l0;  // visible [l0, l1)
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if ((uint32_t)(j - l0) >= (uint32_t)(l1 - l0)) sr[j] = __float_as_uint(-INFINITY);
      }
      // row max: 8 independent chains of three-operand max
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[k + 8]));
#pragma unroll
      for (int j = 16; j < 128; j += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mx8[k] = fmax3(mx8[k], __uint_as_float(sr[j + k]), __uint_as_float(sr[j + 8 + k]));
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      const float mt = mx * c;
      bool rescale = false;
      float alpha = 1.f;
      if (r.first_of_unit) {
        m = mt;
        l = lcomp = 0.f;
      } else if (mt > m + kRescaleLog2) {
        alpha = fast_exp2(m - mt);
        m = mt;
        l *= alpha;
        lcomp *= alpha;
        rescale = true;
      }
      const float msub = (m == -INFINITY) ? 0.f : m;
      // rescale O first (rare): P_t V of this tile adds to it as soon as the first half
      // of P is in tensor memory
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(o_col + c0, ov);
          tmem_wait_ld();
          reg_fence32(ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st32(o_col + c0, ov);
        }
      }
      // packed fp32x2 arithmetic: one instruction per pair of columns
      const float2 c2 = make_float2(c, c), nm2 = make_float2(-msub, -msub);
      float2 ls4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // P in two 64-key halves, released one by one
        uint32_t pk[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = half * 32 + jj;
          float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1])),
                                c2, nm2);
          x.x = fast_exp2(x.x);
          x.y = fast_exp2(x.y);
          ls4[jj & 3] = __fadd2_rn(ls4[jj & 3], x);
          pk[jj] = pack_bf16(x.x, x.y);
        }
        tmem_st32(s_col + half * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_addr(sbase, B_P_FULL + 2 * t + half));
      }
      const float2 lsa = __fadd2_rn(__fadd2_rn(ls4[0], ls4[1]), __fadd2_rn(ls4[2], ls4[3]));
      const float ls = lsa.x + lsa.y;
      {
        const float tsum = l + ls;
        lcomp += (l - tsum) + ls;
        l = tsum;
      }
      ++kc;
      if (r.last_of_unit) {
        if (!mbar_wait(bar_addr(sbase, B_O_DONE + t), oc & 1)) { fail(); break; }
        ++oc;
        tc_fence_after();
        const float lt = l + lcomp;
        const float inv = 1.f / lt;
        const float lse = (m + log2f(lt)) * kLn2;
        if (r.complete) {
          const bool valid = row_used && vt < a.rt;
          const int32_t hrow = r.h + head_off;
          // output row of token vt (of member r.m when units are per member)
          const int64_t mrow = kMode == 1 ? (int64_t)r.m * a.R : 0;
          const int64_t orow_idx = valid ? (mrow + vt) * a.hq + hrow : 0;
          __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(out.o) + orow_idx * kD;
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t ov[32];
            tmem_ld32(o_col + c0, ov);
            tmem_wait_ld();
            reg_fence32(ov);
            if (valid) {
#pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint4 w;
                w.x = pack_bf16(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv);
                w.y = pack_bf16(__uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
                w.z = pack_bf16(__uint_as_float(ov[i + 4]) * inv, __uint_as_float(ov[i + 5]) * inv);
                w.w = pack_bf16(__uint_as_float(ov[i + 6]) * inv, __uint_as_float(ov[i + 7]) * inv);
                *reinterpret_cast<uint4*>(orow + c0 + i) = w;
              }
            }
          }
          if (valid) out.lse[orow_idx] = lse;
        } else {
          const int slot = r.slot;
          float* prow = out.part_o + ((int64_t)slot * kUnitRows + t * kTile + row) * kD;
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t ov[32];
            tmem_ld32(o_col + c0, ov);
            tmem_wait_ld();
            reg_fence32(ov);
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(prow + c0 + i) =
                  make_float4(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv,
                              __uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
          }
          out.part_lse[(int64_t)slot * kUnitRows + t * kTile + row] = lse;
        }
        tc_fence_before();
        m = -INFINITY;
        l = lcomp = 0.f;
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

// Merge the partial (o, lse) of the pieces of every tail unit (fixed piece order):
//   lse = log sum_k exp(lse_k),  o = sum_k exp(lse_k - lse) o_k.
// Grid: (tail units, row groups of kCombineRows); one thread per head_dim column.
constexpr int kCombineRows = 8;
__global__ void __launch_bounds__(kD) replay_fwd_tc_combine(const LsAttnArgs a, const LsSched sc,
                                                            const LsFwdOut out) {
  const int tu = blockIdx.x, T = sc.tail_units, Q = sc.pieces;
  const int u = sc.tail_unit0() + tu;
  const int tpt = kTile / a.pack, tok_per_unit = a.tiles * tpt;
  const int m = u / a.upm, ul = u - m * a.upm;  // member, unit within the member
  const int nTB = (a.rt + tok_per_unit - 1) / tok_per_unit;
  int grp, tb;
  unit_coords(ul, a.hq / a.pack, nTB, sc.tb_major != 0, &grp, &tb);
  const int t0 = tb * tok_per_unit;
  const int h0 = grp * a.pack;
  const int col = threadIdx.x;
  for (int r = blockIdx.y * kCombineRows; r < (blockIdx.y + 1) * kCombineRows; ++r) {
    const int l = r % kTile;  // row within its tile
    if (l >= a.pack * tpt || r / kTile >= a.tiles) continue;
    const int t = t0 + (r / kTile) * tpt + l / a.pack, h = h0 + l % a.pack;
    if (t >= a.rt) continue;
    float mx = -INFINITY;
    for (int k = 0; k < Q; ++k) mx = fmaxf(mx, out.part_lse[(int64_t)(k * T + tu) * kUnitRows + r]);
    float sum = 0.f;
    for (int k = 0; k < Q; ++k) sum += expf(out.part_lse[(int64_t)(k * T + tu) * kUnitRows + r] - mx);
    const float lse = mx + logf(sum);
    float acc = 0.f;
    for (int k = 0; k < Q; ++k) {
      const int64_t slot = k * T + tu;
      acc += expf(out.part_lse[slot * kUnitRows + r] - lse) * out.part_o[(slot * kUnitRows + r) * kD + col];
    }
    const int64_t row = ((int64_t)m * a.R + t) * a.hq + h;
    static_cast<__nv_bfloat16*>(out.o)[row * kD + col] = __float2bfloat16_rn(acc);
    if (col == 0) out.lse[row] = lse;
  }
}

}  // namespace

int ls_fwd_unit_rows() { return kUnitRows; }
int ls_fwd_tile() { return kTile; }
int ls_fwd_ctas_per_sm() { return 1; }
int ls_num_units(int R, int hq, int hkv, int unit_rows) {
  (void)hkv;
  return hq * ((R + unit_rows - 1) / unit_rows);
}
// Grouped-query packing.  A one-head unit of 256 tokens leaves most of its rows empty
// for short responses, so a tile may instead hold `pack` query heads of one KV head
// (pack dividing g) for floor(128 / pack) tokens: each K/V tile then serves pack heads
// at once.  Units then cover (KV head, group of pack heads, token block); a packed unit
// whose tokens all fit one tile runs as a one-tile unit (tile B would be padding).
// The pack is the one with the least work, counted in tiles with a one-tile unit
// costing 1.6 tiles (measured at P = 2,097,152, g = 6: a one-tile unit has no second tile
// to run while its softmax works, 0.17 ms against 0.11 ms per tile of two-tile units);
// on a tie the larger pack (fewer units streaming the prompt), except that one head per
// tile wins any tie.
namespace {
int64_t fwd_tiles_for(int R, int hq, int pack) {  // in tenths of a two-tile unit's tile
  const int tpt = kTile / pack;
  const int tiles = (pack > 1 && R <= tpt) ? 1 : 2;
  const int64_t units = (int64_t)(hq / pack) * ((R + tiles * tpt - 1) / (tiles * tpt));
  return units * (tiles == 1 ? 16 : 20);
}
}  // namespace
int ls_fwd_pack(int R, int hq, int hkv) {
  const int g = hq / hkv;
  int best = 1;
  int64_t bt = INT64_MAX;
  for (int p = g < 64 ? g : 64; p >= 2; --p) {
    if (g % p) continue;
    const int64_t t = fwd_tiles_for(R, hq, p);
    if (t < bt) {
      best = p;
      bt = t;
    }
  }
  return fwd_tiles_for(R, hq, 1) <= bt ? 1 : best;
}
int ls_fwd_tiles(int R, int hq, int hkv) {
  const int pack = ls_fwd_pack(R, hq, hkv);
  return (pack > 1 && R <= kTile / pack) ? 1 : 2;
}
int ls_fwd_units(int R, int hq, int hkv) {
  const int pack = ls_fwd_pack(R, hq, hkv);
  const int tok_per_unit = ls_fwd_tiles(R, hq, hkv) * (kTile / pack);
  return (hq / pack) * ((R + tok_per_unit - 1) / tok_per_unit);
}

cudaError_t ls_launch_replay_fwd(const LsAttnArgs& a, const LsSched& sc, const LsFwdOut& out,
                                 cudaStream_t st) {
  TmapSet tm;
  // Q and the response K/V are (dim, head, token) maps, with a fourth dimension for the
  // member when one launch covers several responses: a box never crosses a member, so
  // rows past a member's R read as zeros, not as the next member's rows.
  const uint32_t box_q[4] = {64, 1, kTile, 1};
  const uint64_t M = (uint64_t)a.members;
  const int mode = a.members <= 1 ? (sc.seg.n > 1 ? 3 : 0) : (a.rt > a.R ? 2 : 1);
  const int rank = (mode == 0 || mode == 3) ? 3 : 4;
  {
    // Q boxes: 128 tokens of one head, or floor(128 / pack) tokens x pack heads; in
    // kMode 2 the members' tokens are one sequence of rt tokens
    const uint32_t box_qp[4] = {64, (uint32_t)a.pack, (uint32_t)(kTile / a.pack), 1};
    const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)(mode == 2 ? a.rt : a.R), M};
    const uint64_t strides[3] = {(uint64_t)kD * 2, (uint64_t)a.hq * kD * 2,
                                 (uint64_t)a.R * a.hq * kD * 2};
    if (!ls_make_tmap_bf16(&tm.q, a.q, mode == 1 ? 4 : 3, dims, strides, box_qp))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)a.R, M};
    const uint64_t strides[3] = {(uint64_t)kD * 2, (uint64_t)a.hkv * kD * 2,
                                 (uint64_t)a.R * a.hkv * kD * 2};
    if (!ls_make_tmap_bf16(&tm.kr, a.k_resp, rank, dims, strides, box_q)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.vr, a.v_resp, rank, dims, strides, box_q)) return cudaErrorInvalidValue;
  }
  {
    const int ps = 1 << a.ps_log2;
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.num_pages * a.hkv * ps};
    const uint64_t strides[1] = {(uint64_t)kD * 2};
    const uint32_t box[2] = {64, (uint32_t)(ps < kTile ? ps : kTile)};
    if (!ls_make_tmap_bf16(&tm.kp, a.k_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tm.vp, a.v_pool, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  // token-block-major instances for the one-response layouts (the only ones whose
  // schedule can ask for it: members' launches take long responses or packed tokens)
  const bool tb = sc.tb_major != 0 && (mode == 0 || mode == 3), pk = a.pack > 1;
  const void* fn;
  if (mode == 1) {
    fn = (const void*)replay_fwd_tc_kernel<1, false, false>;
  } else if (mode == 2) {
    fn = (const void*)replay_fwd_tc_kernel<2, false, true>;
  } else if (mode == 0) {
    fn = tb ? (pk ? (const void*)replay_fwd_tc_kernel<0, true, true>
                  : (const void*)replay_fwd_tc_kernel<0, true, false>)
            : (pk ? (const void*)replay_fwd_tc_kernel<0, false, true>
                  : (const void*)replay_fwd_tc_kernel<0, false, false>);
  } else {
    fn = tb ? (pk ? (const void*)replay_fwd_tc_kernel<3, true, true>
                  : (const void*)replay_fwd_tc_kernel<3, true, false>)
            : (pk ? (const void*)replay_fwd_tc_kernel<3, false, true>
                  : (const void*)replay_fwd_tc_kernel<3, false, false>);
  }
  if ((mode == 1 && pk) || (mode == 2 && !pk)) return cudaErrorInvalidValue;
  if ((mode == 1 || mode == 2) && sc.tb_major) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&tm, (void*)&a, (void*)&sc, (void*)&out};
  e = cudaLaunchKernel(fn, dim3(sc.ctas), dim3(kThreads), args, kSmemBytes, st);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ls_note_launch();
  if (sc.has_partials()) {
    replay_fwd_tc_combine<<<dim3((unsigned)sc.tail_units, kUnitRows / kCombineRows), kD, 0, st>>>(a, sc, out);
    e = cudaGetLastError();
    if (e == cudaSuccess) ls_note_launch();
  }
  return e;
}
