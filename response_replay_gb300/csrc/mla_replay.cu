// mla_replay.cu -- replay attention over latent (MLA-style) pages, forward, on the
// 5th-generation tensor cores.
//
// The GLM path of the LongStraw explainer ("Two incompatible architectures, same
// transaction", GLM bullet) keeps multi-head latent attention state as latent pages
// held in CPU memory and replays each response over them.  The layer is multi-head
// latent attention (DeepSeek-V2, 2024) with the key up-projection absorbed into the
// query: every position j keeps one row shared by all heads, its latent c_j (512
// values) followed by its rotary key r_j (64 values), and head h of token t brings an
// absorbed query of 576 values:
//   s_{t,h,j} = scale <q_{t,h}, [c_j ; r_j]>,  j over the P prompt rows and the
//               response rows j <= t
//   lse_{t,h} = log sum_j exp(s),   o_{t,h} = sum_j exp(s - lse) c_j   (512 values)
// The value up-projection and the output projection are weights, applied by the caller.
//
// Shape.  A 128-row fp32 output of 512 columns would fill all 512 tensor-memory columns
// and leave none for the scores, so a unit is 128 query rows (token-major (t, h) rows)
// times one half of the output columns; the two halves of a row tile are separate
// units, each computing the full 576-wide scores (the price of the split: the score
// products run twice).  Latent tiles are 64 rows (72 KB) in a two-stage ring: the score
// MMA then has N = 64, and a tile's fixed costs (waits, commits, the softmax round trip)
// are paid once per 64 rows (measured: 32-row tiles ran the tensor pipe 26% busy).  The
// unit's Q tile is split between the 128 tensor-memory columns the output and the two
// score buffers leave free (values 0-255, the A operand of the first 16 score MMAs) and
// shared memory (values 256-575, 80 KB).  A stage can be refilled only once P L of its
// tile is done, so that P L is issued ahead of the next score MMAs (see the issuer) and
// the producer also prefetches prompt tiles into L2 four tiles ahead (the refills then
// hit L2).  In a stage
// the unit's output half (atoms 4h .. 4h+3) sits in the last four 8 KB slots and the
// other five atoms in the first five, loaded in slot order (measured 3% faster than the
// atoms in their own order).  Prompt tiles are gathered page by page through the page
// table, and the pages may be pinned host memory read over the host link.
//
// CTA (one per SM, persistent, 8 warps) over the same split-KV schedule as the other
// replay kernels (ls_sched.h: whole units in waves, tail units cut into pieces whose
// partial (o, lse) mla_fwd_combine merges):
//   warp 0      TMA producer: the shared-memory part of the unit's Q (5 boxes of 64
//               values x 128 rows), then the latent tiles (9 boxes of 64 values x 64
//               rows, two of 32 rows on 32-row pages), and L2 prefetches of the prompt
//               tiles four ahead; rows of a ragged last prompt tile are zeroed before the
//               hand-over.
//   warp 1      MMA issuer (one thread): O += P(g-1) L[:, half] for the tile before (four
//               TS MMAs, M=128 N=256, P from tensor memory, the latent tile as an
//               MN-major operand), then S(g) = Q L^T into one of two score buffers (16
//               TS MMAs with Q from tensor memory, then 20 SS MMAs; M=128 N=64 K=16).
//               A stage is refilled only after the P L of its tile, so issuing that P L
//               before S(g) lets the load of tile g + 1 land while S(g) computes
//               (measured 20% faster than S(g) first, which overlapped the softmax of
//               g - 1 with S(g) but left every tile waiting for its stage).  P L starts on
//               the first half of P (keys 0-31) while the softmax finishes the second
//               (measured 4% faster than waiting for all of P).  At a range
//               boundary the old range's last P L goes first, so its output can be read
//               and the next Q written into tensor memory.
//   warps 4-7   at the start of a range, the tensor-memory part of Q (each thread its
//               row's first 256 values, once the old range's score MMAs are done);
//               softmax, one query row per thread: scores of the tile, masks, running
//               max in the log2 domain (O rescaled only when the max grows by more than
//               2^8, after the previous tile's P L has finished), compensated row sum, P
//               as bf16 pairs over the score buffer, released in two halves of 32 keys;
//               at the end of a range normalises O and writes o / lse, or a partial for
//               the combine.
// Tensor memory (512 columns): O [0,256), S0 [256,320), S1 [320,384), Q values 0-255 as
// bf16 pairs [384,512).
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"
#include "ls_tmap.h"
#include "ls_umma.cuh"

namespace {

using namespace umma;

constexpr int kDc = 512;                  // latent values (output columns)
constexpr int kD = 576;                   // latent + rotary values (score length)
constexpr int kAtoms = kD / 64;           // 128-byte swizzle atoms per row
constexpr int kRows = 128;                // query rows per unit
constexpr int kKeys = 64;                 // latent rows per tile
constexpr int kHalf = kDc / 2;            // output columns per unit
constexpr int kStages = 2;
constexpr int kPrefetch = 4;              // prompt tiles prefetched into L2 ahead of the loads
constexpr int kQtAtoms = 4;               // Q atoms held in tensor memory (values 0-255)
constexpr int kThreads = 256;
constexpr uint32_t kQAtomBytes = kRows * 128;           // 16 KB
constexpr uint32_t kLAtomBytes = kKeys * 128;           // 8 KB
constexpr uint32_t kQBytes = (kAtoms - kQtAtoms) * kQAtomBytes;  // 80 KB in shared memory
constexpr uint32_t kStageBytes = kAtoms * kLAtomBytes;  // 72 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffRing = kQBytes;
constexpr uint32_t kOffBar = kOffRing + kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr uint32_t kColO = 0, kColS = kHalf, kColQ = kHalf + 2 * kKeys;
static_assert(kColQ + kQtAtoms * 32 == 512, "tensor memory columns");
constexpr int kPCols = kKeys / 2;         // P(g) as bf16 pairs over its score buffer
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

enum {
  B_KV_FULL = 0,
  B_KV_EMPTY = B_KV_FULL + kStages,
  B_Q_FULL = B_KV_EMPTY + kStages,
  B_Q_EMPTY,
  B_QT_FULL,                 // the softmax warps wrote the range's Q values 0-383
  B_S_FULL,                  // 2: scores of tile g in buffer g & 1
  B_P_FULL = B_S_FULL + 2,   // 4: P of tile g, keys [32 hf, 32 hf + 32), at 2 (g & 1) + hf
  B_PV_DONE = B_P_FULL + 4,  // P L of a tile finished (one phase per tile)
  B_O_DONE,                  // the range's last P L finished
  B_AUX,                     // producer: ragged prompt tile landed
  B_DONE,
  B_COUNT
};
static_assert(B_COUNT * 8 + 16 <= 256, "barrier area");

struct MlaTmaps {
  CUtensorMap q, lp, lr;
};

__device__ __forceinline__ uint32_t bar(uint32_t sbase, int i) { return sbase + kOffBar + 8u * i; }

// A phase that has already completed returns on a plain test; otherwise the bounded,
// sleeping wait.
__device__ __forceinline__ bool wait_fast(uint32_t b, uint32_t parity) {
  return mbar_try_wait(b, parity) || mbar_wait(b, parity);
}

// Prefetch a tensor-map box into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y)
               : "memory");
}

// Stage slot of latent atom `at` (values 64 at .. 64 at + 63) for output half h: the half's
// four atoms in slots 5-8, the others in slots 0-4; atom_in_slot is the inverse.
__device__ __forceinline__ int slot_of(int h, int at) {
  if (h == 0) return at >= 4 ? at - 4 : at + 5;
  return at < 4 ? at : (at == 8 ? 4 : at + 1);
}
__device__ __forceinline__ int atom_in_slot(int h, int sl) {
  if (h == 0) return sl < 5 ? 4 + sl : sl - 5;
  return sl < 4 ? sl : (sl == 4 ? 8 : sl - 1);
}

// One latent tile of the walk.
struct MlaTile {
  int32_t u, key0, slot;
  bool resp, first, last, complete;
};

// The tiles of one CTA in schedule order: each (unit, item) of LsWalk expanded into its
// 64-row tiles (a prompt split's tile range, or the response rows up to the row tile's
// last token).  Every item has at least one tile (non-empty splits; R >= 1), so the
// first / last flags of a range always land on a tile.
struct MlaCursor {
  LsWalk walk;
  int32_t R, H, t, t_end, u, slot;
  bool valid, resp, ifirst, ilast, complete;

  __device__ MlaCursor(const LsSched& sc, int32_t cta, int32_t R_, int32_t H_)
      : walk(sc, cta), R(R_), H(H_), t(0), t_end(0), u(0), slot(-1), valid(false),
        resp(false), ifirst(false), ilast(false), complete(false) {}

  __device__ bool open() {
    int32_t s;
    while (walk.next(&u, &s, &ifirst, &ilast, &complete, &slot)) {
      resp = s == walk.sc->nsplit;
      if (resp) {
        const int64_t rows = (int64_t)R * H;
        const int64_t end = (int64_t)(u >> 1) * kRows + kRows;
        const int32_t t_hi = (int32_t)(((end < rows ? end : rows) - 1) / H);
        t = 0;
        t_end = (t_hi + kKeys) / kKeys;
      } else {
        walk.sc->split_tiles(s, &t, &t_end);
      }
      if (t < t_end) return true;
    }
    return false;
  }

  __device__ bool next(MlaTile* r) {
    bool opened = false;
    if (!valid || t >= t_end) {
      valid = open();
      if (!valid) return false;
      opened = true;
    }
    r->u = u;
    r->key0 = t * kKeys;
    r->slot = slot;
    r->resp = resp;
    r->complete = complete;
    r->first = ifirst && opened;
    ++t;
    r->last = ilast && t >= t_end;
    return true;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
mla_fwd_kernel(const __grid_constant__ MlaTmaps tm, const LsMlaArgs a,
               const __grid_constant__ LsSched sc) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffBar + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + B_COUNT * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(sbase, B_KV_FULL + i), 1);
      mbar_init(bar(sbase, B_KV_EMPTY + i), 1);
    }
    mbar_init(bar(sbase, B_Q_FULL), 1);
    mbar_init(bar(sbase, B_Q_EMPTY), 1);
    mbar_init(bar(sbase, B_QT_FULL), kRows);
    for (int i = 0; i < 2; ++i) mbar_init(bar(sbase, B_S_FULL + i), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(sbase, B_P_FULL + i), kRows);
    mbar_init(bar(sbase, B_PV_DONE), 1);
    mbar_init(bar(sbase, B_O_DONE), 1);
    mbar_init(bar(sbase, B_AUX), 1);
    mbar_init(bar(sbase, B_DONE), 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm.q);
      tma_prefetch_desc(&tm.lp);
      tma_prefetch_desc(&tm.lr);
      MlaCursor cur(sc, blockIdx.x, a.R, a.H);
      MlaTile r;
      uint32_t ring = 0, ranges = 0, aux = 0;
      const int32_t ps = 1 << a.ps_log2;
      const int32_t box_rows = ps < kKeys ? ps : kKeys;
      const int32_t pool_rows = a.num_pages * ps;
      // a second walk kPrefetch tiles ahead: its prompt tiles are prefetched into L2, so
      // the stage loads (which may start only when a stage is released) hit L2
      MlaCursor ahead(sc, blockIdx.x, a.R, a.H);
      MlaTile ra;
      bool more = true;
      auto prefetch = [&]() {
        more = more && ahead.next(&ra);
        if (!more || ra.resp) return;
        for (int bb = 0; bb < kKeys / box_rows; ++bb) {
          const int32_t pos = ra.key0 + bb * box_rows;
          if (pos >= a.P) break;
          const int32_t phys = __ldg(a.page_table + (pos >> a.ps_log2));
          if ((uint32_t)phys >= (uint32_t)a.num_pages) continue;
          const int32_t y = phys * ps + (pos & (ps - 1));
          for (int at = 0; at < kAtoms; ++at) tma_prefetch_l2_2d(&tm.lp, at * 64, y);
        }
      };
      for (int i = 0; i < kPrefetch; ++i) prefetch();
      while (cur.next(&r)) {
        prefetch();
        if (r.first) {
          if (ranges > 0 && !mbar_wait(bar(sbase, B_Q_EMPTY), (ranges - 1) & 1)) { fail(); break; }
          const uint32_t qb = bar(sbase, B_Q_FULL);
          mbar_expect_tx(qb, kQBytes);
          for (int at = kQtAtoms; at < kAtoms; ++at)
            tma_load_2d(sbase + kOffQ + (at - kQtAtoms) * kQAtomBytes, &tm.q, at * 64,
                        (r.u >> 1) * kRows, qb);
          ++ranges;
        }
        const uint32_t st = ring % kStages;
        if (!mbar_wait(bar(sbase, B_KV_EMPTY + st), ((ring / kStages) & 1) ^ 1)) { fail(); break; }
        if (*abort_flag) break;
        // Rows past P on the last prompt page may hold stale data (even NaN); their
        // weight is 0 but 0 x NaN is not, so they are zeroed before the hand-over.
        const bool ragged = !r.resp && r.key0 + kKeys > a.P;
        const uint32_t fb = bar(sbase, ragged ? (int)B_AUX : B_KV_FULL + (int)st);
        const uint32_t dst = sbase + kOffRing + st * kStageBytes;
        mbar_expect_tx(fb, kStageBytes);
        if (r.resp) {
          for (int sl = 0; sl < kAtoms; ++sl)
            tma_load_2d(dst + sl * kLAtomBytes, &tm.lr, atom_in_slot(r.u & 1, sl) * 64, r.key0,
                        fb);
        } else {
          for (int bb = 0; bb < kKeys / box_rows; ++bb) {
            const int32_t pos = r.key0 + bb * box_rows;
            int32_t y = pool_rows;  // past P or a bad page id: reads as zeros
            if (pos < a.P) {
              const int32_t phys = __ldg(a.page_table + (pos >> a.ps_log2));
              if ((uint32_t)phys < (uint32_t)a.num_pages)
                y = phys * ps + (pos & (ps - 1));
              else
                ls_report(a.err, LS_DEVERR_CHECK);
            }
            for (int sl = 0; sl < kAtoms; ++sl)
              tma_load_2d(dst + sl * kLAtomBytes + bb * box_rows * 128, &tm.lp,
                          atom_in_slot(r.u & 1, sl) * 64, y, fb);
          }
        }
        if (ragged) {
          if (!mbar_wait(fb, aux & 1)) { fail(); break; }
          ++aux;
          const int32_t keep = (int32_t)(a.P - r.key0);
          for (int at = 0; at < kAtoms; ++at) {
            uint8_t* base = smem + kOffRing + st * kStageBytes + at * kLAtomBytes;
            for (int i = keep * 8; i < kKeys * 8; ++i)  // whole 128-byte rows
              *reinterpret_cast<uint4*>(base + i * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(sbase, B_KV_FULL + st));
        }
        ++ring;
      }
      // Do not leave while loads into this CTA's shared memory may still be in flight.
      for (uint32_t i = ring > kStages ? ring - kStages : 0; i < ring; ++i)
        mbar_wait(bar(sbase, B_KV_FULL + i % kStages), (i / kStages) & 1);
      if (ranges > 0) mbar_wait(bar(sbase, B_Q_FULL), (ranges - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(kRows, kKeys, false);
      const uint32_t idPV = idesc_bf16_f32(kRows, kHalf, true);
      const uint32_t q_lo = sdesc_lo(sbase + kOffQ, 16);
      MlaCursor cur(sc, blockIdx.x, a.R, a.H);
      MlaTile r, prev;
      uint32_t g = 0, ranges = 0, prev_stage = 0;
      RingPos<kStages> ks;
      bool have_prev = false, ok = true;
      // O += P(pg) L[:, half] for the tile before; its latent stage is free afterwards.
      auto issue_pv = [&](const MlaTile& p, uint32_t pstage, uint32_t pg) -> bool {
        const uint32_t b0 = sdesc_lo(sbase + kOffRing + pstage * kStageBytes + 5u * kLAtomBytes,
                                     kLAtomBytes);  // slots 5-8: the output half
        const uint32_t a0 = tmem + kColS + (pg & 1) * kKeys;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {  // 16 latent rows per MMA
          if ((kk & 1) == 0) {  // each half of P as soon as it is written
            if (!wait_fast(bar(sbase, B_P_FULL + 2 * (pg & 1) + (kk >> 1)), (pg >> 1) & 1))
              return false;
            tc_fence_after();
          }
          mma_ts_lo(tmem + kColO, a0 + kk * 8, b0 + ((kk * 2048u) >> 4), idPV,
                    (kk > 0 || !p.first) ? 1u : 0u);
        }
        mma_commit(bar(sbase, B_KV_EMPTY + pstage));
        mma_commit(bar(sbase, B_PV_DONE));
        if (p.last) mma_commit(bar(sbase, B_O_DONE));
        return true;
      };
      while (cur.next(&r)) {
        if (r.first) {
          // the old range's last P L first: the softmax warps read its output and only
          // then write this range's Q into tensor memory
          if (have_prev && !issue_pv(prev, prev_stage, g - 1)) { ok = false; break; }
          have_prev = false;
          if (!mbar_wait(bar(sbase, B_Q_FULL), ranges & 1)) { ok = false; break; }
          if (!mbar_wait(bar(sbase, B_QT_FULL), ranges & 1)) { ok = false; break; }
          ++ranges;
        } else if (have_prev) {
          // P L of the tile before goes first: it frees the stage that tile g + 1 is loaded
          // into, so that load lands while S(g) computes
          if (!issue_pv(prev, prev_stage, g - 1)) { ok = false; break; }
          have_prev = false;
        }
        if (!wait_fast(bar(sbase, B_KV_FULL + ks.stage), ks.phase)) { ok = false; break; }
        tc_fence_after();
        // S(g): its buffer last held P(g - 2), whose P L was issued before this
        const uint32_t b0 = sdesc_lo(sbase + kOffRing + ks.stage * kStageBytes, 16);
        const uint32_t d = tmem + kColS + (g & 1) * kKeys;
        const int h = r.u & 1;
#pragma unroll
        for (int kk = 0; kk < 4 * kQtAtoms; ++kk) {  // Q values 0-255 from tensor memory
          const uint32_t ob = (slot_of(h, kk >> 2) * kLAtomBytes + (kk & 3) * 32) >> 4;
          mma_ts_lo(d, tmem + kColQ + kk * 8, b0 + ob, idS, kk > 0);
        }
#pragma unroll
        for (int kk = 4 * kQtAtoms; kk < 4 * kAtoms; ++kk) {  // values 256-575 from shared
          const uint32_t oa = (((kk >> 2) - kQtAtoms) * kQAtomBytes + (kk & 3) * 32) >> 4;
          const uint32_t ob = (slot_of(h, kk >> 2) * kLAtomBytes + (kk & 3) * 32) >> 4;
          mma_ss_lo(d, q_lo + oa, b0 + ob, idS, 1u);
        }
        mma_commit(bar(sbase, B_S_FULL + (g & 1)));
        if (r.last) mma_commit(bar(sbase, B_Q_EMPTY));  // the range's Q is read by S only
        prev = r;
        prev_stage = ks.stage;
        have_prev = true;
        ks.advance();
        ++g;
        if ((g & 15) == 0 && *abort_flag) { ok = false; break; }
      }
      if (ok && have_prev && !issue_pv(prev, prev_stage, g - 1)) ok = false;
      if (!ok) fail();
      mma_commit(bar(sbase, B_DONE));
      mbar_wait(bar(sbase, B_DONE), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int row = (warp - 4) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp - 4) * 32) << 16);
    const float c = a.scale_log2;
    const int64_t nrows = (int64_t)a.R * a.H;
    MlaCursor cur(sc, blockIdx.x, a.R, a.H);
    MlaTile r;
    uint32_t g = 0, oc = 0, ranges = 0;
    float m = -INFINITY, l = 0.f, lcomp = 0.f;
    while (cur.next(&r)) {
      if (r.first) {
        // Q values 0-255 of this thread's row into tensor memory (bf16 pairs), once the
        // old range's score MMAs have read theirs; rows past R x H are zeros
        if (ranges > 0 && !mbar_wait(bar(sbase, B_Q_EMPTY), (ranges - 1) & 1)) { fail(); break; }
        tc_fence_after();
        const int64_t qrow = (int64_t)(r.u >> 1) * kRows + row;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                         (qrow < nrows ? qrow : 0) * kD);
#pragma unroll 1
        for (int c0 = 0; c0 < kQtAtoms * 32; c0 += 32) {
          uint32_t qv[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = qrow < nrows ? __ldg(src + c0 / 4 + i) : make_uint4(0, 0, 0, 0);
            qv[4 * i] = v.x;
            qv[4 * i + 1] = v.y;
            qv[4 * i + 2] = v.z;
            qv[4 * i + 3] = v.w;
          }
          tmem_st32(lane_base + kColQ + c0, qv);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(sbase, B_QT_FULL));
        ++ranges;
      }
      // the row's token and the tile's visible keys [0, lim), worked out before the wait
      // for the scores (the wait is on the tile's critical path)
      const int64_t grow = (int64_t)(r.u >> 1) * kRows + row;  // (t, h) row, token-major
      const int32_t tq = (int32_t)(grow / a.H);
      int32_t lim = kKeys;
      if (r.resp) {
        const int32_t lr = tq + 1 - r.key0;
        lim = lr < kKeys ? lr : kKeys;
      } else if (r.key0 + kKeys > a.P) {
        lim = (int32_t)(a.P - r.key0);
      }
      if (!mbar_wait(bar(sbase, B_S_FULL + (g & 1)), (g >> 1) & 1)) { fail(); break; }
      tc_fence_after();
      const uint32_t s_col = lane_base + kColS + (g & 1) * kKeys;
      uint32_t sr[kKeys];
      tmem_ld32(s_col, sr);
      tmem_ld32(s_col + 32, sr + 32);
      tmem_wait_ld();
      reg_fence32(sr);
      reg_fence32(sr + 32);
      if (lim < kKeys) {
#pragma unroll
        for (int j = 0; j < kKeys; ++j)
          if (j >= lim) sr[j] = __float_as_uint(-INFINITY);
      }
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[k + 8]));
#pragma unroll
      for (int j = 16; j < kKeys; j += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mx8[k] = fmax3(mx8[k], __uint_as_float(sr[j + k]), __uint_as_float(sr[j + 8 + k]));
      const float mt = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7])) * c;
      bool rescale = false;
      float alpha = 1.f;
      if (r.first) {
        m = mt;
        l = lcomp = 0.f;
      } else if (mt > m + kRescaleLog2) {
        alpha = fast_exp2(m - mt);
        m = mt;
        l *= alpha;
        lcomp *= alpha;
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // the previous tile's P L (issued after these scores) must have finished
        if (!mbar_wait(bar(sbase, B_PV_DONE), (g - 1) & 1)) { fail(); break; }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < kHalf; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(lane_base + kColO + c0, ov);
          tmem_wait_ld();
          reg_fence32(ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st32(lane_base + kColO + c0, ov);
        }
      }
      const float msub = (m == -INFINITY) ? 0.f : m;
      const float2 c2 = make_float2(c, c), nm2 = make_float2(-msub, -msub);
      float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[kPCols];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {  // each half of P released as soon as it is written
#pragma unroll
        for (int j = 16 * hf; j < 16 * hf + 16; ++j) {
          float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1])),
                                c2, nm2);
          x.x = fast_exp2(x.x);
          x.y = fast_exp2(x.y);
          ls2[j & 1] = __fadd2_rn(ls2[j & 1], x);
          pk[j] = pack_bf16(x.x, x.y);
        }
        tmem_st16(s_col + 16 * hf, pk + 16 * hf);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(sbase, B_P_FULL + 2 * (g & 1) + hf));
      }
      {
        const float2 lsa = __fadd2_rn(ls2[0], ls2[1]);
        const float ls = lsa.x + lsa.y;
        const float tsum = l + ls;
        lcomp += (l - tsum) + ls;
        l = tsum;
      }
      if (r.last) {
        if (!mbar_wait(bar(sbase, B_O_DONE), oc & 1)) { fail(); break; }
        ++oc;
        tc_fence_after();
        const float lt = l + lcomp;
        const float inv = 1.f / lt;
        const float lse = (m + log2f(lt)) * kLn2;
        const bool valid = grow < nrows;
        const int half = r.u & 1;
        if (r.complete) {
          __nv_bfloat16* orow =
              static_cast<__nv_bfloat16*>(a.o) + (valid ? grow : 0) * kDc + half * kHalf;
#pragma unroll 1
          for (int c0 = 0; c0 < kHalf; c0 += 32) {
            uint32_t ov[32];
            tmem_ld32(lane_base + kColO + c0, ov);
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
          if (valid && half == 0) a.lse[grow] = lse;
        } else {
          float* prow = a.part_o + ((int64_t)r.slot * kRows + row) * kHalf;
#pragma unroll 1
          for (int c0 = 0; c0 < kHalf; c0 += 32) {
            uint32_t ov[32];
            tmem_ld32(lane_base + kColO + c0, ov);
            tmem_wait_ld();
            reg_fence32(ov);
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(prow + c0 + i) =
                  make_float4(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv,
                              __uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
          }
          a.part_lse[(int64_t)r.slot * kRows + row] = lse;
        }
        tc_fence_before();
        m = -INFINITY;
        l = lcomp = 0.f;
      }
      ++g;
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

// Merge the partial (o, lse) of the pieces of every tail unit in fixed piece order:
//   lse = log sum_k exp(lse_k),  o = sum_k exp(lse_k - lse) o_k.
// Grid: (tail units, row groups of kCombineRows); one thread per output column of the
// unit's half.
constexpr int kCombineRows = 8;
__global__ void __launch_bounds__(kHalf) mla_fwd_combine(const LsMlaArgs a, const LsSched sc) {
  const int tu = blockIdx.x, T = sc.tail_units, Q = sc.pieces;
  const int u = sc.tail_unit0() + tu;
  const int half = u & 1, col = threadIdx.x;
  const int64_t nrows = (int64_t)a.R * a.H;
  for (int r = blockIdx.y * kCombineRows; r < (blockIdx.y + 1) * kCombineRows; ++r) {
    const int64_t grow = (int64_t)(u >> 1) * kRows + r;
    if (grow >= nrows) break;
    float mx = -INFINITY;
    for (int k = 0; k < Q; ++k) mx = fmaxf(mx, a.part_lse[(int64_t)(k * T + tu) * kRows + r]);
    float sum = 0.f;
    for (int k = 0; k < Q; ++k) sum += expf(a.part_lse[(int64_t)(k * T + tu) * kRows + r] - mx);
    const float lse = mx + logf(sum);
    float acc = 0.f;
    for (int k = 0; k < Q; ++k) {
      const int64_t slot = (int64_t)k * T + tu;
      acc += expf(a.part_lse[slot * kRows + r] - lse) * a.part_o[(slot * kRows + r) * kHalf + col];
    }
    static_cast<__nv_bfloat16*>(a.o)[grow * kDc + half * kHalf + col] = __float2bfloat16_rn(acc);
    if (col == 0 && half == 0) a.lse[grow] = lse;
  }
}

// Capture: pool[pt[p / ps]][p % ps][:] = src[p - start][:] for p in [start, start + n),
// 16-byte pieces (72 per row), grid-stride; a page id outside the pool skips the row and
// reports LS_DEVERR_CHECK.
__global__ void mla_capture_kernel(const uint4* __restrict__ src, uint4* pool,
                                   const int32_t* __restrict__ page_table, int32_t num_pages,
                                   int32_t ps_log2, int64_t start, int64_t n, uint32_t* err) {
  constexpr int kPieces = kD * 2 / 16;
  const int64_t total = n * kPieces;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rrow = i / kPieces;
    const int piece = (int)(i - rrow * kPieces);
    const int64_t p = start + rrow;
    const int32_t phys = __ldg(page_table + (p >> ps_log2));
    if ((uint32_t)phys >= (uint32_t)num_pages) {
      if (piece == 0) ls_report(err, LS_DEVERR_CHECK);
      continue;
    }
    const int64_t drow = ((int64_t)phys << ps_log2) + (p & ((1 << ps_log2) - 1));
    pool[drow * kPieces + piece] = src[rrow * kPieces + piece];
  }
}

}  // namespace

int ls_mla_tile() { return kKeys; }
int ls_mla_unit_rows() { return kRows; }
int ls_mla_half() { return kHalf; }

cudaError_t ls_launch_mla_fwd(const LsMlaArgs& a, const LsSched& sc, cudaStream_t st) {
  MlaTmaps tm;
  {
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.R * a.H};
    const uint64_t strides[1] = {(uint64_t)kD * 2};
    const uint32_t box[2] = {64, (uint32_t)kRows};
    if (!ls_make_tmap_bf16(&tm.q, a.q, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.R};
    const uint64_t strides[1] = {(uint64_t)kD * 2};
    const uint32_t box[2] = {64, (uint32_t)kKeys};
    if (!ls_make_tmap_bf16(&tm.lr, a.lat_resp, 2, dims, strides, box)) return cudaErrorInvalidValue;
    // prompt boxes never cross a page: 64 rows, or one 32-row page
    const uint64_t pdims[2] = {(uint64_t)kD, (uint64_t)a.num_pages << a.ps_log2};
    const uint32_t pbox[2] = {64, (uint32_t)((1 << a.ps_log2) < kKeys ? (1 << a.ps_log2) : kKeys)};
    if (!ls_make_tmap_bf16(&tm.lp, a.pool, 2, pdims, strides, pbox)) return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(mla_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  mla_fwd_kernel<<<sc.ctas, kThreads, kSmemBytes, st>>>(tm, a, sc);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ls_note_launch();
  if (sc.has_partials()) {
    mla_fwd_combine<<<dim3((unsigned)sc.tail_units, kRows / kCombineRows), kHalf, 0, st>>>(a, sc);
    e = cudaGetLastError();
    if (e == cudaSuccess) ls_note_launch();
  }
  return e;
}

cudaError_t ls_launch_capture_latent(const void* src, void* pool, const int32_t* page_table,
                                     int32_t num_pages, int32_t ps_log2, int64_t start,
                                     int64_t n, int sms, uint32_t* err, cudaStream_t st) {
  const int64_t total = n * (kD * 2 / 16);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  mla_capture_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4*>(src),
                                                        static_cast<uint4*>(pool), page_table,
                                                        num_pages, ps_log2, start, n, err);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ls_note_launch();
  return e;
}
