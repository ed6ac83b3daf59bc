// mla_replay_bwd.cu -- replay attention over latent (MLA-style) pages, backward, on the
// 5th-generation tensor cores.
//
// Layer as in mla_replay.cu (multi-head latent attention, DeepSeek-V2 2024, key
// up-projection absorbed into the query; the GLM bullet of the LongStraw explainer's
// "Two incompatible architectures, same transaction" keeps its state as latent pages).
// The prompt rows are stopgrad (LongStraw paper digest, Method, last paragraph), so the
// backward gives dq for every query row and a gradient only for the response's own
// latent rows.  With the forward's lse and output o, and dO (512 values per row):
//   P = exp(s - lse),  D = <dO, o>,  dP_j = <dO, c_j>,  dS = P (dP - D)
//   dq_{t,h} = scale sum_j dS_{t,h,j} [c_j ; r_j]           (576 values, every visible j)
//   d lat_j  = sum_{t >= j, h} P [dO ; 0] + scale dS q_{t,h}  (response rows j only)
// The latent c_j is both key and value, so its gradient has a value term and a key term.
//
// What fits one SM.  A 128-row tile of 576-value queries and 512-value output gradients
// is 272 KB of MMA operands, and a 576-column fp32 dq does not fit the 512 tensor-memory
// columns.  So the dq kernel stacks 64 query rows over the same 64 rows' dO on the 128
// lanes of one MMA: Q rows on lanes 0-63, dO rows on lanes 64-127 (their rotary 64
// values zero), times the latent tile, gives S on lanes 0-63 and dP on lanes 64-127 in
// one product (M = 128, N = 32 keys, K = 576).  dq then lives on both lane halves of
// the same 320 columns: values {0-255, 512-575} on lanes 64-127 and values 256-511 on
// lanes 0-63.  Each lane half is written by a product whose A operand (dS as bf16 in
// tensor memory) is dS on that half and zero on the other, so each product adds exactly
// zero to the other half's columns:
//   [0 ; dS] L[:, 0-255] and [0 ; dS] L[:, 512-575] -> lanes 64-127
//   [dS ; 0] L[:, 256-511]                          -> lanes 0-63
// The two zero-padded copies of dS fill the tile's 32-column S|dP buffer once S and dP
// have been read out, so the whole dq of a row tile takes no more tensor memory than the
// scores and one unit computes it with no recompute of S and dP.
//
// mla_bwd_dq_kernel (one CTA per SM, persistent, 8 warps; units = 64-row tiles over the
// split-KV schedule of ls_sched.h; pieces of tail units leave partial dq that
// mla_bwd_dq_combine adds in piece order):
//   warp 0      TMA producer: the shared-memory part of the stacked operand (values
//               256-575: Q rows 0-63, dO rows 64-127), then the latent tiles (9 boxes of
//               64 values x 32 rows, 3-stage ring) gathered through the page table, with
//               L2 prefetches of the prompt tiles eight ahead; rows of a ragged last prompt
//               tile are zeroed before the hand-over.
//   warp 1      MMA issuer (one thread): S|dP(g) into one of two 32-column buffers (16 TS
//               MMAs with values 0-255 from tensor memory, 20 SS), then dq += dS(g-1) L
//               (three TS MMAs per 16 keys as above, the latent tile as an MN-major
//               operand).
//   warps 4-5   lanes 0-63: P = exp2(s scale log2 e - lse log2 e) with the causal and
//               ragged masks; warps 6-7, lanes 64-127: dP.  Each pair hands its values to
//               the other through shared memory, both form dS = P (dP - D) (the same
//               bits on both sides) and write their zero-padded copy over the buffer.  At
//               the end of a range each half reads its dq columns, scales them and
//               writes dq (or a partial).
//   At the start of a range all four write the tensor-memory part of the stacked operand
//   (each thread its row's values 0-255 of Q or dO).
// Tensor memory (512 columns): stacked values 0-255 as bf16 pairs [0,128), S|dP buffers
// [128,160) and [160,192), dq [192,512).
//
// mla_bwd_dlat_kernel: the response rows' gradient, key-stationary.  A unit is one
// 128-row tile of the response's latent rows (M = 128, resident: values 0-255 in tensor
// memory, written by the key-lane warps, 256-575 in shared memory) and
// one part of the 576 output columns ({0-255, 512-575} or {256-511}, each unit computing
// S^T and dP^T for itself); it walks the query rows that see the
// tile (tokens t >= the tile's first row) 16 at a time:
//   S^T|dP^T = L [Q rows ; dO rows]^T   (SS, M = 128 keys, N = 32: 16 Q rows, 16 dO rows)
//   P^T, dS^T scale as bf16 (one key per thread)
//   d lat += P^T dO + dS^T Q             (TS, the row stage as an MN-major operand)
// The walk's iterations are cut into equal contiguous chunks, one per CTA; a unit cut by
// a chunk boundary leaves partial sums that mla_bwd_dlat_combine adds in CTA order.
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"
#include "ls_tmap.h"
#include "ls_umma.cuh"

namespace {

using namespace umma;

constexpr int kDc = 512;                  // latent values
constexpr int kD = 576;                   // latent + rotary values
constexpr int kAtoms = kD / 64;           // 128-byte swizzle atoms per row
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPartCols = 320;            // columns of part 0 (part 1: 256)

// Parts of a 576-value gradient row: part 0 = values {0-255, 512-575} (dq: lanes 64-127;
// d lat: even units), part 1 = values 256-511; accumulator column c of part h -> value.
__device__ __forceinline__ int part_value(int h, int c) {
  return h == 0 ? (c < 256 ? c : c + 256) : c + 256;
}
__device__ __forceinline__ int part_cols(int h) { return h == 0 ? kPartCols : 256; }

// ===================================================================== dq kernel
constexpr int kRows = 64;                 // query rows per unit
constexpr int kM = 128;                   // stacked MMA rows: Q rows, then dO rows
constexpr int kKeys = 32;                 // latent rows per tile
constexpr int kStages = 3;
constexpr int kPrefetch = 8;              // prompt tiles prefetched into L2 ahead
constexpr int kTAtoms = 4;                // stacked atoms held in tensor memory (0-255)
constexpr uint32_t kAAtomBytes = kM * 128;                       // 16 KB
constexpr uint32_t kLAtomBytes = kKeys * 128;                    // 4 KB
constexpr uint32_t kABytes = (kAtoms - kTAtoms) * kAAtomBytes;   // 80 KB
constexpr uint32_t kAFill = (kAtoms - kTAtoms) * kRows * 128 + (8 - kTAtoms) * kRows * 128;
constexpr uint32_t kStageBytes = kAtoms * kLAtomBytes;           // 36 KB
constexpr uint32_t kXBytes = kRows * kKeys * 4;                  // 8 KB: one side's values
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffRing = kABytes;
constexpr uint32_t kOffX = kOffRing + kStages * kStageBytes;     // [tile & 1][P, dP]
constexpr uint32_t kOffBar = kOffX + 4 * kXBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr uint32_t kColA = 0, kColS = kTAtoms * 32, kColDq = kColS + 2 * kKeys;
static_assert(kColDq + kPartCols == 512, "tensor memory columns");

enum {
  B_KV_FULL = 0,
  B_KV_EMPTY = B_KV_FULL + kStages,
  B_Q_FULL = B_KV_EMPTY + kStages,
  B_Q_EMPTY,
  B_QT_FULL,                  // the four softmax warps wrote values 0-255 of the range
  B_S_FULL,                   // 2: S|dP of tile g in buffer g & 1
  B_X_FULL = B_S_FULL + 2,    // 2: P and dP of tile g in exchange buffer g & 1
  B_X_EMPTY = B_X_FULL + 2,   // 2: exchange buffer read by both sides
  B_DS_FULL = B_X_EMPTY + 2,  // 2: dS of tile g over buffer g & 1
  B_DQ_DONE = B_DS_FULL + 2,  // the range's last dq MMA finished
  B_AUX,                      // producer: ragged prompt tile landed
  B_DONE,
  B_COUNT
};
static_assert(B_COUNT * 8 + 16 <= 256, "barrier area");

struct DqTmaps {
  CUtensorMap q, d_o, lp, lr;
};

__device__ __forceinline__ uint32_t bar(uint32_t sbase, int i) { return sbase + kOffBar + 8u * i; }

// A phase that has already completed returns on a plain test; otherwise the bounded,
// sleeping wait.
__device__ __forceinline__ bool wait_fast(uint32_t b, uint32_t parity) {
  return mbar_try_wait(b, parity) || mbar_wait(b, parity);
}

__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y)
               : "memory");
}

struct DqTile {
  int32_t u, key0, slot;
  bool resp, first, last, complete;
};

// Tiles of one CTA in schedule order: each (unit, item) of LsWalk expanded into its
// 32-row latent tiles (a prompt split's range, or the response rows up to the row
// tile's last token).
struct DqCursor {
  LsWalk walk;
  int32_t R, H, t, t_end, u, slot;
  bool valid, resp, ifirst, ilast, complete;

  __device__ DqCursor(const LsSched& sc, int32_t cta, int32_t R_, int32_t H_)
      : walk(sc, cta), R(R_), H(H_), t(0), t_end(0), u(0), slot(-1), valid(false),
        resp(false), ifirst(false), ilast(false), complete(false) {}

  __device__ bool open() {
    int32_t s;
    while (walk.next(&u, &s, &ifirst, &ilast, &complete, &slot)) {
      resp = s == walk.sc->nsplit;
      if (resp) {
        const int64_t rows = (int64_t)R * H;
        const int64_t end = (int64_t)u * kRows + kRows;
        const int32_t t_hi = (int32_t)(((end < rows ? end : rows) - 1) / H);
        t = 0;
        t_end = t_hi / kKeys + 1;
      } else {
        walk.sc->split_tiles(s, &t, &t_end);
      }
      if (t < t_end) return true;
    }
    return false;
  }

  __device__ bool next(DqTile* r) {
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
mla_bwd_dq_kernel(const __grid_constant__ DqTmaps tm, const LsMlaBwdArgs a,
                  const __grid_constant__ LsSched sc) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffBar + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + B_COUNT * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // The dO rows of the last stacked atom (values 512-575) are zero for good: no load
  // writes them.
  {
    uint4* z = reinterpret_cast<uint4*>(smem + kOffA + (kAtoms - 1 - kTAtoms) * kAAtomBytes +
                                        kRows * 128);
    for (int i = tid; i < kRows * 128 / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(sbase, B_KV_FULL + i), 1);
      mbar_init(bar(sbase, B_KV_EMPTY + i), 1);
    }
    mbar_init(bar(sbase, B_Q_FULL), 1);
    mbar_init(bar(sbase, B_Q_EMPTY), 1);
    mbar_init(bar(sbase, B_QT_FULL), kM);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(sbase, B_S_FULL + i), 1);
      mbar_init(bar(sbase, B_X_FULL + i), kM);
      mbar_init(bar(sbase, B_X_EMPTY + i), kM);
      mbar_init(bar(sbase, B_DS_FULL + i), kM);
    }
    mbar_init(bar(sbase, B_DQ_DONE), 1);
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
      tma_prefetch_desc(&tm.d_o);
      tma_prefetch_desc(&tm.lp);
      tma_prefetch_desc(&tm.lr);
      DqCursor cur(sc, blockIdx.x, a.R, a.H);
      DqTile r;
      uint32_t ring = 0, ranges = 0, aux = 0;
      const int32_t ps = 1 << a.ps_log2;
      const int32_t pool_rows = a.num_pages * ps;
      DqCursor ahead(sc, blockIdx.x, a.R, a.H);
      DqTile ra;
      bool more = true;
      auto prefetch = [&]() {
        more = more && ahead.next(&ra);
        if (!more || ra.resp || ra.key0 >= a.P) return;
        const int32_t phys = __ldg(a.page_table + (ra.key0 >> a.ps_log2));
        if ((uint32_t)phys >= (uint32_t)a.num_pages) return;
        const int32_t y = phys * ps + (ra.key0 & (ps - 1));
        for (int at = 0; at < kAtoms; ++at) tma_prefetch_l2_2d(&tm.lp, at * 64, y);
      };
      for (int i = 0; i < kPrefetch; ++i) prefetch();
      while (cur.next(&r)) {
        prefetch();
        if (r.first) {
          if (ranges > 0 && !mbar_wait(bar(sbase, B_Q_EMPTY), (ranges - 1) & 1)) { fail(); break; }
          const uint32_t qb = bar(sbase, B_Q_FULL);
          const int32_t row0 = r.u * kRows;
          mbar_expect_tx(qb, kAFill);
          for (int at = kTAtoms; at < kAtoms; ++at)
            tma_load_2d(sbase + kOffA + (at - kTAtoms) * kAAtomBytes, &tm.q, at * 64, row0, qb);
          for (int at = kTAtoms; at < 8; ++at)
            tma_load_2d(sbase + kOffA + (at - kTAtoms) * kAAtomBytes + kRows * 128, &tm.d_o,
                        at * 64, row0, qb);
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
          for (int at = 0; at < kAtoms; ++at)
            tma_load_2d(dst + at * kLAtomBytes, &tm.lr, at * 64, r.key0, fb);
        } else {
          // a tile is one box: tiles are 32-row aligned and pages at least 32 rows
          int32_t y = pool_rows;  // a bad page id: reads as zeros
          const int32_t phys = __ldg(a.page_table + (r.key0 >> a.ps_log2));
          if ((uint32_t)phys < (uint32_t)a.num_pages)
            y = phys * ps + (r.key0 & (ps - 1));
          else
            ls_report(a.err, LS_DEVERR_CHECK);
          for (int at = 0; at < kAtoms; ++at)
            tma_load_2d(dst + at * kLAtomBytes, &tm.lp, at * 64, y, fb);
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
      const uint32_t idS = idesc_bf16_f32(kM, kKeys, false);
      const uint32_t id256 = idesc_bf16_f32(kM, 256, true);
      const uint32_t id64 = idesc_bf16_f32(kM, 64, true);
      const uint32_t a_lo = sdesc_lo(sbase + kOffA, 16);
      DqCursor cur(sc, blockIdx.x, a.R, a.H);
      DqTile r, prev;
      uint32_t g = 0, ranges = 0, prev_stage = 0;
      RingPos<kStages> ks;
      bool have_prev = false, ok = true;
      // dq += dS(pg) L for the tile before; its latent stage is free afterwards.
      auto issue_dq = [&](const DqTile& p, uint32_t pstage, uint32_t pg) -> bool {
        if (!wait_fast(bar(sbase, B_DS_FULL + (pg & 1)), (pg >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t sb = sbase + kOffRing + pstage * kStageBytes;
        // [0 ; dS] in the buffer's first 16 columns, [dS ; 0] in the next 16
        const uint32_t a_hi = tmem + kColS + (pg & 1) * kKeys, a_lo = a_hi + kKeys / 2;
        const uint32_t b_lat = sdesc_lo(sb, kLAtomBytes);                    // values 0-255
        const uint32_t b_mid = sdesc_lo(sb + 4u * kLAtomBytes, kLAtomBytes);  // 256-511
        const uint32_t b_rot = sdesc_lo(sb + 8u * kLAtomBytes, kLAtomBytes);  // 512-575
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {  // 16 latent rows per MMA
          const uint32_t acc = (kk > 0 || !p.first) ? 1u : 0u;
          const uint32_t ob = (kk * 2048u) >> 4;
          // the first product of a range sets all 128 lanes (zero on lanes 0-63), so the
          // lanes 0-63 product accumulates from the start
          mma_ts_lo(tmem + kColDq, a_hi + kk * 8, b_lat + ob, id256, acc);
          mma_ts_lo(tmem + kColDq + 256, a_hi + kk * 8, b_rot + ob, id64, acc);
          mma_ts_lo(tmem + kColDq, a_lo + kk * 8, b_mid + ob, id256, 1u);
        }
        mma_commit(bar(sbase, B_KV_EMPTY + pstage));
        if (p.last) mma_commit(bar(sbase, B_DQ_DONE));
        return true;
      };
      while (cur.next(&r)) {
        if (r.first) {
          // the old range's last dq first: the dS warps read it and only then write this
          // range's rows into tensor memory
          if (have_prev && !issue_dq(prev, prev_stage, g - 1)) { ok = false; break; }
          have_prev = false;
          if (!mbar_wait(bar(sbase, B_Q_FULL), ranges & 1)) { ok = false; break; }
          if (!mbar_wait(bar(sbase, B_QT_FULL), ranges & 1)) { ok = false; break; }
          ++ranges;
        }
        if (!wait_fast(bar(sbase, B_KV_FULL + ks.stage), ks.phase)) { ok = false; break; }
        tc_fence_after();
        // S|dP(g): its buffer last held dS(g - 2), whose dq MMA was issued before this
        const uint32_t b0 = sdesc_lo(sbase + kOffRing + ks.stage * kStageBytes, 16);
        const uint32_t d = tmem + kColS + (g & 1) * kKeys;
#pragma unroll
        for (int kk = 0; kk < 4 * kTAtoms; ++kk) {  // values 0-255 from tensor memory
          const uint32_t ob = ((kk >> 2) * kLAtomBytes + (kk & 3) * 32) >> 4;
          mma_ts_lo(d, tmem + kColA + kk * 8, b0 + ob, idS, kk > 0);
        }
#pragma unroll
        for (int kk = 4 * kTAtoms; kk < 4 * kAtoms; ++kk) {  // values 256-575 from shared
          const uint32_t oa = (((kk >> 2) - kTAtoms) * kAAtomBytes + (kk & 3) * 32) >> 4;
          const uint32_t ob = ((kk >> 2) * kLAtomBytes + (kk & 3) * 32) >> 4;
          mma_ss_lo(d, a_lo + oa, b0 + ob, idS, 1u);
        }
        mma_commit(bar(sbase, B_S_FULL + (g & 1)));
        if (r.last) mma_commit(bar(sbase, B_Q_EMPTY));  // the stacked rows are read by S only
        if (have_prev && !issue_dq(prev, prev_stage, g - 1)) { ok = false; break; }
        prev = r;
        prev_stage = ks.stage;
        have_prev = true;
        ks.advance();
        ++g;
        if ((g & 15) == 0 && *abort_flag) { ok = false; break; }
      }
      if (ok && have_prev && !issue_dq(prev, prev_stage, g - 1)) ok = false;
      if (!ok) fail();
      mma_commit(bar(sbase, B_DONE));
      mbar_wait(bar(sbase, B_DONE), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P / dP / dS warps
    const int row = (warp - 4) * 32 + lane;  // tensor-memory lane
    const bool is_s = row < kRows;           // lanes 0-63: S and P; 64-127: dP
    const int rr = row & (kRows - 1);
    const uint32_t lane_base = tmem + ((uint32_t)((warp - 4) * 32) << 16);
    const float c = a.scale_log2;
    const int64_t nrows = (int64_t)a.R * a.H;
    DqCursor cur(sc, blockIdx.x, a.R, a.H);
    DqTile r;
    uint32_t g = 0, oc = 0, ranges = 0;
    float lse2 = 0.f, dd = 0.f;  // the row's lse log2(e) (lanes 0-63) and D
    while (cur.next(&r)) {
      const int64_t grow = (int64_t)r.u * kRows + rr;  // (t, h) row, token-major
      const bool valid = grow < nrows;
      if (r.first) {
        // values 0-255 of this thread's row (Q on lanes 0-63, dO on 64-127) into tensor
        // memory, once the old range's S|dP MMAs have read theirs; rows past R x H zero
        if (ranges > 0 && !mbar_wait(bar(sbase, B_Q_EMPTY), (ranges - 1) & 1)) { fail(); break; }
        tc_fence_after();
        const uint4* src =
            is_s ? reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                  (valid ? grow : 0) * kD)
                 : reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.d_o) +
                                                  (valid ? grow : 0) * kDc);
#pragma unroll 1
        for (int c0 = 0; c0 < kTAtoms * 32; c0 += 32) {
          uint32_t v[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 w = valid ? __ldg(src + c0 / 4 + i) : make_uint4(0, 0, 0, 0);
            v[4 * i] = w.x;
            v[4 * i + 1] = w.y;
            v[4 * i + 2] = w.z;
            v[4 * i + 3] = w.w;
          }
          tmem_st32(lane_base + kColA + c0, v);
        }
        lse2 = valid && is_s ? __ldg(a.lse + grow) * kLog2e : 0.f;
        dd = valid ? __ldg(a.delta + grow) : 0.f;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(sbase, B_QT_FULL));
        ++ranges;
      }
      // the tile's visible keys [0, lim) for this row, worked out before the wait
      int32_t lim = kKeys;
      if (is_s) {
        const int32_t tq = (int32_t)(grow / a.H);
        if (r.resp) {
          const int32_t lr = tq + 1 - r.key0;
          lim = lr < kKeys ? lr : kKeys;
        } else if (r.key0 + kKeys > a.P) {
          lim = (int32_t)(a.P - r.key0);
        }
        if (!valid) lim = 0;
      }
      if (!mbar_wait(bar(sbase, B_S_FULL + (g & 1)), (g >> 1) & 1)) { fail(); break; }
      tc_fence_after();
      const uint32_t s_col = lane_base + kColS + (g & 1) * kKeys;
      uint32_t x[kKeys];
      tmem_ld32(s_col, x);
      tmem_wait_ld();
      reg_fence32(x);
      // lanes 0-63 turn S into P; lanes 64-127 keep dP as it is
      float mine[kKeys];
      if (is_s) {
#pragma unroll
        for (int j = 0; j < kKeys; ++j)
          mine[j] = j < lim ? fast_exp2(__uint_as_float(x[j]) * c - lse2) : 0.f;
      } else {
#pragma unroll
        for (int j = 0; j < kKeys; ++j) mine[j] = __uint_as_float(x[j]);
      }
      tc_fence_before();
      // Exchange: P rows at side 0, dP rows at side 1 of buffer g & 1; 16-byte chunk k
      // of a row at position k ^ (row & 7), so a quarter-warp's accesses touch every bank
      // once.
      uint8_t* xb = smem + kOffX + (g & 1) * 2 * kXBytes;
      float4* own = reinterpret_cast<float4*>(xb + (is_s ? 0 : kXBytes) + rr * kKeys * 4);
      const float4* other =
          reinterpret_cast<const float4*>(xb + (is_s ? kXBytes : 0) + rr * kKeys * 4);
      if (!mbar_wait(bar(sbase, B_X_EMPTY + (g & 1)), ((g >> 1) & 1) ^ 1)) { fail(); break; }
#pragma unroll
      for (int k = 0; k < kKeys / 4; ++k)
        own[k ^ (rr & 7)] = make_float4(mine[4 * k], mine[4 * k + 1], mine[4 * k + 2], mine[4 * k + 3]);
      mbar_arrive(bar(sbase, B_X_FULL + (g & 1)));
      if (!mbar_wait(bar(sbase, B_X_FULL + (g & 1)), (g >> 1) & 1)) { fail(); break; }
      float theirs[kKeys];
#pragma unroll
      for (int k = 0; k < kKeys / 4; ++k) {
        const float4 w = other[k ^ (rr & 7)];
        theirs[4 * k] = w.x;
        theirs[4 * k + 1] = w.y;
        theirs[4 * k + 2] = w.z;
        theirs[4 * k + 3] = w.w;
      }
      mbar_arrive(bar(sbase, B_X_EMPTY + (g & 1)));
      // dS = P (dP - D), the same operands and operations on both sides; lanes 64-127
      // write [dS, 0] and lanes 0-63 [0, dS] over the buffer's 32 columns
      uint32_t pk[kKeys];
#pragma unroll
      for (int j = 0; j < kKeys / 2; ++j) {
        const float p0 = is_s ? mine[2 * j] : theirs[2 * j];
        const float p1 = is_s ? mine[2 * j + 1] : theirs[2 * j + 1];
        const float q0 = is_s ? theirs[2 * j] : mine[2 * j];
        const float q1 = is_s ? theirs[2 * j + 1] : mine[2 * j + 1];
        const uint32_t w = pack_bf16(p0 * (q0 - dd), p1 * (q1 - dd));
        pk[j] = is_s ? 0u : w;
        pk[kKeys / 2 + j] = is_s ? w : 0u;
      }
      tmem_st32(s_col, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(sbase, B_DS_FULL + (g & 1)));
      if (r.last) {
        if (!mbar_wait(bar(sbase, B_DQ_DONE), oc & 1)) { fail(); break; }
        ++oc;
        tc_fence_after();
        // lanes 64-127: values 0-255 and 512-575 (320 columns); lanes 0-63: 256-511 (256)
        const int h = is_s ? 1 : 0;
        const int nc = part_cols(h);
        float* drow = r.complete ? a.dq + (valid ? grow : 0) * kD
                                 : a.part_dq + ((int64_t)r.slot * kRows + rr) * kD;
#pragma unroll 1
        for (int c0 = 0; c0 < kPartCols; c0 += 32) {
          if (c0 >= nc) break;
          uint32_t v[32];
          tmem_ld32(lane_base + kColDq + c0, v);
          tmem_wait_ld();
          reg_fence32(v);
          if (valid || !r.complete) {
            float* dst = drow + part_value(h, c0);
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + i) =
                  make_float4(__uint_as_float(v[i]) * a.scale, __uint_as_float(v[i + 1]) * a.scale,
                              __uint_as_float(v[i + 2]) * a.scale, __uint_as_float(v[i + 3]) * a.scale);
          }
        }
        tc_fence_before();
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

// Partial dq of the pieces of every tail unit, added in fixed piece order.
// Grid: (tail units, row groups of 8); one thread per dq value.
constexpr int kCombineRows = 8;
__global__ void __launch_bounds__(kD) mla_bwd_dq_combine(const LsMlaBwdArgs a, const LsSched sc) {
  const int tu = blockIdx.x, T = sc.tail_units, Q = sc.pieces;
  const int u = sc.tail_unit0() + tu;
  const int col = threadIdx.x;
  const int64_t nrows = (int64_t)a.R * a.H;
  for (int r = blockIdx.y * kCombineRows; r < (blockIdx.y + 1) * kCombineRows; ++r) {
    const int64_t grow = (int64_t)u * kRows + r;
    if (grow >= nrows) break;
    float acc = 0.f;
    for (int k = 0; k < Q; ++k) acc += a.part_dq[((int64_t)(k * T + tu) * kRows + r) * kD + col];
    a.dq[grow * kD + col] = acc;
  }
}

// D = <dO, o> per (t, h) row (512 bf16 values each, fp32 sum): one warp per row.
__global__ void __launch_bounds__(256) mla_bwd_delta(const LsMlaBwdArgs a) {
  const int64_t nrows = (int64_t)a.R * a.H;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;
  const uint4* go = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.d_o) + row * kDc);
  const uint4* oo = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.o) + row * kDc);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 x = __ldg(go + lane + 32 * i), y = __ldg(oo + lane + 32 * i);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[k]));
      const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[k]));
      acc = fmaf(xf.x, yf.x, acc);
      acc = fmaf(xf.y, yf.y, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) a.delta[row] = acc;
}

// ===================================================================== d lat kernel
constexpr int kKT = 128;                  // response latent rows per unit (M)
constexpr int kNB = 16;                   // query rows per iteration
constexpr int kN2 = 2 * kNB;              // stacked: Q rows 0-15, dO rows 16-31
constexpr int kRStages = 4;
constexpr int kLtAtoms = 4;               // latent values 0-255 of the tile in tensor memory
constexpr int kMinIters = 16;             // fewest iterations a CTA of the walk takes
constexpr uint32_t kLTAtomBytes = kKT * 128;                     // 16 KB
constexpr uint32_t kLTBytes = (kAtoms - kLtAtoms) * kLTAtomBytes;  // 80 KB: values 256-575
constexpr uint32_t kRAtomBytes = kN2 * 128;                      // 4 KB
constexpr uint32_t kRStageBytes = kAtoms * kRAtomBytes;          // 36 KB
constexpr uint32_t kRFill = kAtoms * kNB * 128 + 8 * kNB * 128;  // Q 9 atoms, dO 8 atoms
constexpr uint32_t kOffL = 0;
constexpr uint32_t kOffR = kLTBytes;
constexpr uint32_t kOffBar2 = kOffR + kRStages * kRStageBytes;
constexpr uint32_t kSmemBytes2 = kOffBar2 + 256 + 1024;
static_assert(kSmemBytes2 <= 232448, "shared memory per CTA");
// S^T|dP^T buffers [0,64), d lat [64,384), latent values 0-255 as bf16 pairs [384,512)
constexpr uint32_t kColB = 0, kColAcc = 2 * kN2, kColL = kColAcc + kPartCols;
static_assert(kColL + kLtAtoms * 32 == 512, "tensor memory columns");

enum {
  C_L_FULL = 0,
  C_L_EMPTY,
  C_LT_FULL,                    // the key-lane warps wrote the tile's values 0-255
  C_R_FULL,                     // 2 row stages
  C_R_EMPTY = C_R_FULL + kRStages,
  C_S_FULL = C_R_EMPTY + kRStages,  // 2: S^T|dP^T of iteration g in buffer g & 1
  C_PD_FULL = C_S_FULL + 2,     // 2: P^T, dS^T of iteration g written over buffer g & 1
  C_ACC_DONE = C_PD_FULL + 2,   // the unit's last d lat MMA finished
  C_DONE,
  C_COUNT
};
static_assert(C_COUNT * 8 + 16 <= 256, "barrier area");

struct DlatTmaps {
  CUtensorMap q, d_o, lr;
};

// The walk of the d lat kernel.  Unit u = (key tile kt = u >> 1, part u & 1); its
// iterations are the 16-row blocks rb from 8 kt H (token 128 kt, the tile's first row)
// up to ceil(R H / 16).  Units follow one another in u order, and CTA c takes the
// iterations [total c / C, total (c + 1) / C).
struct DlatGeom {
  int32_t H, nkt, ctas;
  int64_t rb_hi, total;
  __host__ __device__ int64_t n_it(int64_t kt) const { return rb_hi - 8 * kt * H; }
  __host__ __device__ int64_t unit_begin(int32_t u) const {
    const int64_t kt = u >> 1;
    return 2 * (kt * rb_hi - 4ll * H * kt * (kt - 1)) + (u & 1) * n_it(kt);
  }
  __host__ __device__ int64_t chunk_begin(int32_t c) const { return total * c / ctas; }
  // Partial-sum slot of unit u in CTA c (u not whole in c): 2c for the unit the chunk
  // starts in, 2c + 1 for one that starts inside the chunk.
  __host__ __device__ int32_t slot(int32_t c, int64_t ub) const {
    return 2 * c + (ub > chunk_begin(c) ? 1 : 0);
  }
};

DlatGeom make_dlat_geom(int32_t R, int32_t H, int sms) {
  DlatGeom g;
  g.H = H;
  g.nkt = (R + kKT - 1) / kKT;
  g.rb_hi = ((int64_t)R * H + kNB - 1) / kNB;
  g.ctas = 1;
  g.total = 0;
  g.total = g.unit_begin(2 * g.nkt);
  // at least kMinIters iterations per CTA: a thinner slice costs more in its latent tile
  // load and in the partial sums it leaves than it saves
  int64_t c = sms;
  if (c > g.total / kMinIters) c = g.total / kMinIters;
  g.ctas = c < 1 ? 1 : (int32_t)c;
  return g;
}

struct DlatIt {
  int32_t u, rb, slot;
  bool first, last, complete;
};

struct DlatCursor {
  const DlatGeom* gm;
  int32_t c, u;
  int64_t x, x0, x1, ub, ue;

  __device__ DlatCursor(const DlatGeom& g, int32_t cta) : gm(&g), c(cta) {
    x0 = x = g.chunk_begin(cta);
    x1 = g.chunk_begin(cta + 1);
    int32_t lo = 0, hi = 2 * g.nkt;  // last u with unit_begin(u) <= x
    while (hi - lo > 1) {
      const int32_t m = (lo + hi) >> 1;
      if (g.unit_begin(m) <= x) lo = m; else hi = m;
    }
    u = lo;
    ub = g.unit_begin(u);
    ue = g.unit_begin(u + 1);
  }

  __device__ bool next(DlatIt* it) {
    if (x >= x1) return false;
    while (x >= ue) {
      ++u;
      ub = ue;
      ue = gm->unit_begin(u + 1);
    }
    it->u = u;
    it->rb = (int32_t)(8ll * (u >> 1) * gm->H + (x - ub));
    it->first = x == (ub > x0 ? ub : x0);
    it->last = x + 1 == (ue < x1 ? ue : x1);
    it->complete = ub >= x0 && ue <= x1;
    it->slot = gm->slot(c, ub);
    ++x;
    return true;
  }
};

__device__ __forceinline__ uint32_t bar2(uint32_t sbase, int i) { return sbase + kOffBar2 + 8u * i; }

__global__ void __launch_bounds__(kThreads, 1)
mla_bwd_dlat_kernel(const __grid_constant__ DlatTmaps tm, const LsMlaBwdArgs a,
                    const __grid_constant__ DlatGeom gm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffBar2 + C_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar2 + C_COUNT * 8 + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // The dO rows of each row stage's last atom (values 512-575) are zero for good.
  for (int s = 0; s < kRStages; ++s) {
    uint4* z = reinterpret_cast<uint4*>(smem + kOffR + s * kRStageBytes + 8 * kRAtomBytes +
                                        kNB * 128);
    for (int i = tid; i < kNB * 128 / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(bar2(sbase, C_L_FULL), 1);
    mbar_init(bar2(sbase, C_L_EMPTY), 1);
    mbar_init(bar2(sbase, C_LT_FULL), kKT);
    for (int i = 0; i < kRStages; ++i) {
      mbar_init(bar2(sbase, C_R_FULL + i), 1);
      mbar_init(bar2(sbase, C_R_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar2(sbase, C_S_FULL + i), 1);
      mbar_init(bar2(sbase, C_PD_FULL + i), kKT);
    }
    mbar_init(bar2(sbase, C_ACC_DONE), 1);
    mbar_init(bar2(sbase, C_DONE), 1);
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
      tma_prefetch_desc(&tm.d_o);
      tma_prefetch_desc(&tm.lr);
      DlatCursor cur(gm, blockIdx.x);
      DlatIt it;
      uint32_t ring = 0, units = 0;
      while (cur.next(&it)) {
        if (it.first) {
          if (units > 0 && !mbar_wait(bar2(sbase, C_L_EMPTY), (units - 1) & 1)) { fail(); break; }
          const uint32_t lb = bar2(sbase, C_L_FULL);
          mbar_expect_tx(lb, kLTBytes);
          for (int at = kLtAtoms; at < kAtoms; ++at)
            tma_load_2d(sbase + kOffL + (at - kLtAtoms) * kLTAtomBytes, &tm.lr, at * 64,
                        (it.u >> 1) * kKT, lb);
          ++units;
        }
        const uint32_t st = ring % kRStages;
        if (!mbar_wait(bar2(sbase, C_R_EMPTY + st), ((ring / kRStages) & 1) ^ 1)) { fail(); break; }
        if (*abort_flag) break;
        const uint32_t fb = bar2(sbase, C_R_FULL + st);
        const uint32_t dst = sbase + kOffR + st * kRStageBytes;
        mbar_expect_tx(fb, kRFill);
        for (int at = 0; at < kAtoms; ++at)
          tma_load_2d(dst + at * kRAtomBytes, &tm.q, at * 64, it.rb * kNB, fb);
        for (int at = 0; at < 8; ++at)
          tma_load_2d(dst + at * kRAtomBytes + kNB * 128, &tm.d_o, at * 64, it.rb * kNB, fb);
        ++ring;
      }
      for (uint32_t i = ring > kRStages ? ring - kRStages : 0; i < ring; ++i)
        mbar_wait(bar2(sbase, C_R_FULL + i % kRStages), (i / kRStages) & 1);
      if (units > 0) mbar_wait(bar2(sbase, C_L_FULL), (units - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(kKT, kN2, false);
      const uint32_t id256 = idesc_bf16_f32(kKT, 256, true);
      const uint32_t id64 = idesc_bf16_f32(kKT, 64, true);
      const uint32_t l_lo = sdesc_lo(sbase + kOffL, 16);
      DlatCursor cur(gm, blockIdx.x);
      DlatIt it, prev;
      uint32_t g = 0, units = 0, prev_stage = 0;
      RingPos<kRStages> ks;
      bool have_prev = false, ok = true;
      // d lat += P^T dO + dS^T Q of the iteration before; its row stage is free afterwards.
      auto issue_dlat = [&](const DlatIt& p, uint32_t pstage, uint32_t pg) -> bool {
        if (!wait_fast(bar2(sbase, C_PD_FULL + (pg & 1)), (pg >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t sb = sbase + kOffR + pstage * kRStageBytes;
        const uint32_t aP = tmem + kColB + (pg & 1) * kN2;  // P^T: 16 rows as 8 columns
        const uint32_t aS = aP + 8;                          // dS^T scale
        const uint32_t acc0 = p.first ? 0u : 1u;
        const uint32_t at0 = (p.u & 1) ? 4u : 0u;
        mma_ts_lo(tmem + kColAcc, aP, sdesc_lo(sb + at0 * kRAtomBytes + kNB * 128, kRAtomBytes),
                  id256, acc0);
        mma_ts_lo(tmem + kColAcc, aS, sdesc_lo(sb + at0 * kRAtomBytes, kRAtomBytes), id256, 1u);
        if ((p.u & 1) == 0)
          mma_ts_lo(tmem + kColAcc + 256, aS, sdesc_lo(sb + 8 * kRAtomBytes, kRAtomBytes), id64,
                    acc0);
        mma_commit(bar2(sbase, C_R_EMPTY + pstage));
        if (p.last) mma_commit(bar2(sbase, C_ACC_DONE));
        return true;
      };
      while (cur.next(&it)) {
        if (it.first) {
          if (have_prev && !issue_dlat(prev, prev_stage, g - 1)) { ok = false; break; }
          have_prev = false;
          if (!mbar_wait(bar2(sbase, C_L_FULL), units & 1)) { ok = false; break; }
          if (!mbar_wait(bar2(sbase, C_LT_FULL), units & 1)) { ok = false; break; }
          ++units;
        } else if (have_prev) {
          // the product of the iteration before goes first: it frees the row stage that
          // iteration g + 1 is loaded into, so that load lands while S^T(g) computes
          if (!issue_dlat(prev, prev_stage, g - 1)) { ok = false; break; }
          have_prev = false;
        }
        if (!wait_fast(bar2(sbase, C_R_FULL + ks.stage), ks.phase)) { ok = false; break; }
        tc_fence_after();
        const uint32_t b0 = sdesc_lo(sbase + kOffR + ks.stage * kRStageBytes, 16);
        const uint32_t d = tmem + kColB + (g & 1) * kN2;
#pragma unroll
        for (int kk = 0; kk < 4 * kLtAtoms; ++kk) {  // values 0-255 from tensor memory
          const uint32_t ob = ((kk >> 2) * kRAtomBytes + (kk & 3) * 32) >> 4;
          mma_ts_lo(d, tmem + kColL + kk * 8, b0 + ob, idS, kk > 0);
        }
#pragma unroll
        for (int kk = 4 * kLtAtoms; kk < 4 * kAtoms; ++kk) {  // values 256-575 from shared
          const uint32_t oa = (((kk >> 2) - kLtAtoms) * kLTAtomBytes + (kk & 3) * 32) >> 4;
          const uint32_t ob = ((kk >> 2) * kRAtomBytes + (kk & 3) * 32) >> 4;
          mma_ss_lo(d, l_lo + oa, b0 + ob, idS, 1u);
        }
        mma_commit(bar2(sbase, C_S_FULL + (g & 1)));
        if (it.last) mma_commit(bar2(sbase, C_L_EMPTY));  // the latent tile is read by S only
        prev = it;
        prev_stage = ks.stage;
        have_prev = true;
        ks.advance();
        ++g;
        if ((g & 15) == 0 && *abort_flag) { ok = false; break; }
      }
      if (ok && have_prev && !issue_dlat(prev, prev_stage, g - 1)) ok = false;
      if (!ok) fail();
      mma_commit(bar2(sbase, C_DONE));
      mbar_wait(bar2(sbase, C_DONE), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P^T / dS^T warps
    const int k = (warp - 4) * 32 + lane;  // key of the tile on this lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp - 4) * 32) << 16);
    const float c = a.scale_log2;
    const int64_t nrows = (int64_t)a.R * a.H;
    DlatCursor cur(gm, blockIdx.x);
    DlatIt it;
    uint32_t g = 0, oc = 0, units = 0;
    while (cur.next(&it)) {
      const int32_t j = (it.u >> 1) * kKT + k;  // response row
      if (it.first) {
        // values 0-255 of this lane's latent row into tensor memory, once the old unit's
        // score MMAs have read theirs; rows past R are zeros
        if (units > 0 && !mbar_wait(bar2(sbase, C_L_EMPTY), (units - 1) & 1)) { fail(); break; }
        tc_fence_after();
        const bool in = j < a.R;
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(a.lat_resp) + (int64_t)(in ? j : 0) * kD);
#pragma unroll 1
        for (int c0 = 0; c0 < kLtAtoms * 32; c0 += 32) {
          uint32_t v[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 w = in ? __ldg(src + c0 / 4 + i) : make_uint4(0, 0, 0, 0);
            v[4 * i] = w.x;
            v[4 * i + 1] = w.y;
            v[4 * i + 2] = w.z;
            v[4 * i + 3] = w.w;
          }
          tmem_st32(lane_base + kColL + c0, v);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar2(sbase, C_LT_FULL));
        ++units;
      }
      // the block's 16 lse and D values (the same for every thread), loaded before the
      // wait so their latency hides behind it
      float lse2[kNB], dd[kNB];
#pragma unroll
      for (int n = 0; n < kNB; ++n) {
        const int64_t row = (int64_t)it.rb * kNB + n;
        const bool in = row < nrows;
        lse2[n] = in ? __ldg(a.lse + row) * kLog2e : 0.f;
        dd[n] = in ? __ldg(a.delta + row) : 0.f;
      }
      if (!mbar_wait(bar2(sbase, C_S_FULL + (g & 1)), (g >> 1) & 1)) { fail(); break; }
      tc_fence_after();
      const uint32_t b_col = lane_base + kColB + (g & 1) * kN2;
      uint32_t x[kN2];
      tmem_ld32(b_col, x);
      tmem_wait_ld();
      reg_fence32(x);
      uint32_t pk[kNB];
#pragma unroll
      for (int n = 0; n < kNB; n += 2) {
        float pv[2], dv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t row = (int64_t)it.rb * kNB + n + e;
          const bool vis = row < nrows && j < a.R && (int64_t)j * a.H <= row;  // j <= t
          float p = 0.f, ds = 0.f;
          if (vis) {
            p = fast_exp2(__uint_as_float(x[n + e]) * c - lse2[n + e]);
            ds = p * (__uint_as_float(x[kNB + n + e]) - dd[n + e]) * a.scale;
          }
          pv[e] = p;
          dv[e] = ds;
        }
        pk[n / 2] = pack_bf16(pv[0], pv[1]);
        pk[kNB / 2 + n / 2] = pack_bf16(dv[0], dv[1]);
      }
      tmem_st16(b_col, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar2(sbase, C_PD_FULL + (g & 1)));
      if (it.last) {
        if (!mbar_wait(bar2(sbase, C_ACC_DONE), oc & 1)) { fail(); break; }
        ++oc;
        tc_fence_after();
        const int h = it.u & 1;
        const int nc = part_cols(h);
        const bool keep = j < a.R;
        float* drow = it.complete ? a.dlat + (int64_t)(keep ? j : 0) * kD
                                  : a.part_dlat + ((int64_t)it.slot * kKT + k) * kPartCols;
#pragma unroll 1
        for (int c0 = 0; c0 < nc; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(lane_base + kColAcc + c0, v);
          tmem_wait_ld();
          reg_fence32(v);
          if (keep || !it.complete) {
            float* dst = drow + (it.complete ? part_value(h, c0) : c0);
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + i) =
                  make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                              __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
          }
        }
        tc_fence_before();
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

// Units cut by a chunk boundary: their partial sums added in CTA order.  Grid: (units,
// key groups of 2); one thread per accumulator column of the part.  Whole units were
// written by the kernel itself.
__global__ void __launch_bounds__(kPartCols) mla_bwd_dlat_combine(const LsMlaBwdArgs a,
                                                                  const DlatGeom gm) {
  const int32_t u = blockIdx.x, h = u & 1, col = threadIdx.x;
  if (col >= part_cols(h)) return;
  const int64_t ub = gm.unit_begin(u), ue = gm.unit_begin(u + 1);
  int32_t c0 = -1, c1 = -1;  // CTAs whose chunks meet [ub, ue)
  for (int32_t c = 0; c < gm.ctas; ++c) {
    const int64_t b = gm.chunk_begin(c), e = gm.chunk_begin(c + 1);
    if (b < e && b < ue && e > ub) {
      if (c0 < 0) c0 = c;
      c1 = c;
    }
  }
  if (c0 < 0 || (c0 == c1 && gm.chunk_begin(c0) <= ub && gm.chunk_begin(c0 + 1) >= ue)) return;
  for (int kk = blockIdx.y * 2; kk < blockIdx.y * 2 + 2; ++kk) {
    const int32_t j = (u >> 1) * kKT + kk;
    if (j >= a.R) break;
    float acc = 0.f;
    for (int32_t c = c0; c <= c1; ++c) {
      const int64_t b = gm.chunk_begin(c), e = gm.chunk_begin(c + 1);
      if (b >= e) continue;
      acc += a.part_dlat[((int64_t)gm.slot(c, ub) * kKT + kk) * kPartCols + col];
    }
    a.dlat[(int64_t)j * kD + part_value(h, col)] = acc;
  }
}

}  // namespace

int ls_mla_bwd_tile() { return kKeys; }
int ls_mla_bwd_unit_rows() { return kRows; }
int ls_mla_bwd_part_cols() { return kPartCols; }
int ls_mla_bwd_dlat_ctas(int32_t R, int32_t H, int sms) {
  return R > 0 ? make_dlat_geom(R, H, sms).ctas : 0;
}

cudaError_t ls_launch_mla_bwd(const LsMlaBwdArgs& a, const LsSched& sc, int sms, cudaStream_t st) {
  const int64_t nrows = (int64_t)a.R * a.H;
  DqTmaps tq;
  DlatTmaps tl;
  {
    const uint64_t qdims[2] = {(uint64_t)kD, (uint64_t)nrows};
    const uint64_t qstr[1] = {(uint64_t)kD * 2};
    const uint64_t odims[2] = {(uint64_t)kDc, (uint64_t)nrows};
    const uint64_t ostr[1] = {(uint64_t)kDc * 2};
    const uint32_t box64[2] = {64, (uint32_t)kRows};
    const uint32_t box16[2] = {64, (uint32_t)kNB};
    if (!ls_make_tmap_bf16(&tq.q, a.q, 2, qdims, qstr, box64)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tq.d_o, a.d_o, 2, odims, ostr, box64)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tl.q, a.q, 2, qdims, qstr, box16)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tl.d_o, a.d_o, 2, odims, ostr, box16)) return cudaErrorInvalidValue;
    const uint64_t rdims[2] = {(uint64_t)kD, (uint64_t)a.R};
    const uint32_t rbox[2] = {64, (uint32_t)kKeys};
    const uint32_t rbox128[2] = {64, (uint32_t)kKT};
    if (!ls_make_tmap_bf16(&tq.lr, a.lat_resp, 2, rdims, qstr, rbox)) return cudaErrorInvalidValue;
    if (!ls_make_tmap_bf16(&tl.lr, a.lat_resp, 2, rdims, qstr, rbox128)) return cudaErrorInvalidValue;
    const uint64_t pdims[2] = {(uint64_t)kD, (uint64_t)a.num_pages << a.ps_log2};
    if (!ls_make_tmap_bf16(&tq.lp, a.pool, 2, pdims, qstr, rbox)) return cudaErrorInvalidValue;
  }
  cudaError_t e;
  mla_bwd_delta<<<(unsigned)((nrows + 7) / 8), 256, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ls_note_launch();
  e = cudaFuncSetAttribute(mla_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e != cudaSuccess) return e;
  mla_bwd_dq_kernel<<<sc.ctas, kThreads, kSmemBytes, st>>>(tq, a, sc);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ls_note_launch();
  if (sc.has_partials()) {
    mla_bwd_dq_combine<<<dim3((unsigned)sc.tail_units, kRows / kCombineRows), kD, 0, st>>>(a, sc);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ls_note_launch();
  }
  const DlatGeom gm = make_dlat_geom(a.R, a.H, sms);
  e = cudaFuncSetAttribute(mla_bwd_dlat_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes2);
  if (e != cudaSuccess) return e;
  mla_bwd_dlat_kernel<<<gm.ctas, kThreads, kSmemBytes2, st>>>(tl, a, gm);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ls_note_launch();
  mla_bwd_dlat_combine<<<dim3((unsigned)(2 * gm.nkt), kKT / 2), kPartCols, 0, st>>>(a, gm);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ls_note_launch();
  return cudaSuccess;
}
