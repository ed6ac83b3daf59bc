// ls_sched.h -- how replay-attention work is spread over a persistent grid.
//
// Work is a grid of (unit, item) pairs.  A unit is a block of query rows that share a
// key/value head (a few query heads x a block of response tokens); its items are the
// prompt splits 0..S-1 (contiguous ranges of KV tiles) followed by one item for the
// response's own causal keys.  Items of one unit that the same CTA processes back to
// back are merged on chip by the online-softmax rescaling; items of one unit that land
// in different CTAs leave partial results that a combine kernel merges by log-sum-exp
// (the on-chip counterpart of the cross-rank LSE/output merge the LongStraw explainer
// describes in "Two incompatible architectures", Qwen bullet).
//
// Schedule ("full waves + aligned tail pieces"): with C persistent CTAs and U units,
// the first W = floor(U / C) waves give each CTA whole units (unit w*C + c in wave w),
// so every CTA of a wave starts at prompt position 0 at the same time and walks the
// prompt in lockstep: CTAs that share a KV head read each KV tile from HBM once and
// from L2 after that.  The T = U - W*C remaining units are each cut at the same Q item
// boundaries into pieces, and piece k of tail unit t (number p = k*T + t) goes to CTA
// p mod C in round p div C.  In a round, the CTAs holding piece k of different units
// walk the same key range together, so the tail shares L2 the way the waves do; Q is
// the smallest count whose rounds balance the tail to within 2% of T / C units of work
// per CTA.  Each piece leaves a partial result (slot p) that the combine merges in
// piece order (when Q = 1 the tail units are processed whole and need no combine).
//
// Included by host and device code.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define LS_HD __host__ __device__ __forceinline__
#else
#define LS_HD inline
#endif

// Segments of a concatenated response (ragged members replayed in one launch):
// segment s holds tokens [off[s], off[s + 1]).  Every token sees the whole prompt and
// the response keys of its own segment up to itself, so members never see each other.
// A single response is one segment [0, R).
constexpr int kLsMaxSegs = 64;
struct LsSegs {
  int32_t n;
  int32_t off[kLsMaxSegs + 1];
};

// Bounds [lo, hi) of the segment holding token t (t past the end: the last segment).
LS_HD void ls_seg_bounds(const LsSegs& s, int32_t t, int32_t* lo, int32_t* hi) {
  int32_t a = 0, b = s.n;  // off[a] <= t < off[b]
  while (b - a > 1) {
    const int32_t m = (a + b) >> 1;
    if (s.off[m] <= t) a = m; else b = m;
  }
  *lo = s.off[a];
  *hi = s.off[a + 1];
}

struct LsSched {
  int32_t units;       // U
  int32_t ctas;        // C (grid size)
  int32_t waves;       // W full waves
  int32_t ntiles;      // prompt KV tiles per unit: ceil(P / tile)
  int32_t tps;         // prompt tiles per split
  int32_t nsplit;      // non-empty prompt splits S (0 when P == 0)
  int32_t tail_units;  // T = U - W*C
  int32_t pieces;      // Q pieces per tail unit (1: tail units are processed whole)
  int32_t tb_major;    // unit numbering (ls_tiles.cuh, unit_coords): token block major when
                       // the response's causal keys are a large share of a unit's work
  LsSegs seg;          // segments of the response tokens (one: a single response)

  LS_HD int32_t items_per_unit() const { return nsplit + 1; }
  LS_HD int32_t tail_unit0() const { return waves * ctas; }
  LS_HD int32_t num_pieces() const { return tail_units * pieces; }
  LS_HD bool has_partials() const { return tail_units > 0 && pieces > 1; }
  // First item of piece k of a tail unit (k = pieces gives items_per_unit()).
  LS_HD int32_t piece_begin(int32_t k) const {
    return (int32_t)((int64_t)k * items_per_unit() / pieces);
  }
  // True when CTA c has any work (some CTAs get no piece when T*Q < C and W = 0).
  LS_HD bool cta_has_work(int32_t c) const { return waves > 0 || c < num_pieces(); }
  // Prompt tile range [t0, t1) of split s.
  LS_HD void split_tiles(int32_t s, int32_t* t0, int32_t* t1) const {
    int32_t a = s * tps, b = a + tps;
    *t0 = a < ntiles ? a : ntiles;
    *t1 = b < ntiles ? b : ntiles;
  }
};

// Tail time, in units of work per CTA, of T tail units cut into q pieces over C CTAs:
// ceil(T*q / C) rounds of 1/q unit each.
inline double ls_tail_cost(int32_t T, int32_t q, int32_t C) {
  return (double)((T * (int64_t)q + C - 1) / C) / q;
}

// Host: build the schedule for U units, a prompt of `ntiles` tiles, the caller's split
// request and a grid of at most `max_ctas` CTAs; a tail unit is cut into at most
// `max_pieces` pieces.
inline LsSched ls_make_sched(int32_t units, int32_t ntiles, int32_t num_splits, int32_t max_ctas,
                             int32_t max_pieces = 64) {
  LsSched s;
  s.units = units;
  s.ntiles = ntiles;
  if (ntiles > 0) {
    int32_t sp = num_splits < ntiles ? num_splits : ntiles;
    if (sp < 1) sp = 1;
    s.tps = (ntiles + sp - 1) / sp;
    s.nsplit = (ntiles + s.tps - 1) / s.tps;
  } else {
    s.tps = 1;
    s.nsplit = 0;
  }
  const int32_t ipu = s.nsplit + 1;
  int64_t total = (int64_t)units * ipu;
  int32_t c = max_ctas;
  if ((int64_t)c > total) c = (int32_t)total;
  if (c < 1) c = 1;
  s.ctas = c;
  s.waves = units / c;
  s.tail_units = units - s.waves * c;
  s.pieces = 1;
  s.tb_major = 0;
  s.seg.n = 1;
  s.seg.off[0] = 0;
  s.seg.off[1] = 0;
  if (s.tail_units > 0) {
    const int32_t qmax = ipu < max_pieces ? ipu : max_pieces;  // a piece holds at least one item
    double best = ls_tail_cost(s.tail_units, 1, c);
    for (int32_t q = 2; q <= qmax; ++q) {
      const double cq = ls_tail_cost(s.tail_units, q, c);
      if (cq < best) best = cq;
    }
    for (int32_t q = 1; q <= qmax; ++q)
      if (ls_tail_cost(s.tail_units, q, c) <= best * 1.02) {
        s.pieces = q;
        break;
      }
  }
  return s;
}

// Walks the item ranges of one CTA: W whole units, then its tail pieces in round order.
// Usage:  LsWalk w(sched, c); int32_t u, s, slot; bool first, last, complete;
//         while (w.next(&u, &s, &first, &last, &complete, &slot)) { ... }
// first/last: this item is the first/last of the current range (a whole unit or a
// piece); complete: the range is the whole unit u; slot: the partial-result slot of a
// range that is not complete (-1 otherwise).
struct LsWalk {
  const LsSched* sc;   // the schedule (the kernel's __grid_constant__ parameter on the
                       // device, so the walk holds a pointer, not a register copy)
  int32_t cta;
  int32_t range;       // -1 before the first; < waves: whole units; then piece rounds
  int32_t u, it0, it, it_end, slot;
  bool complete;

  LS_HD LsWalk(const LsSched& s, int32_t c)
      : sc(&s), cta(c), range(-1), u(0), it0(0), it(0), it_end(0), slot(-1), complete(false) {}

  LS_HD bool open_range(int32_t r) {
    if (r < sc->waves) {
      u = r * sc->ctas + cta;
      it0 = 0;
      it_end = sc->items_per_unit();
      slot = -1;
      complete = true;
    } else {
      const int64_t p = (int64_t)cta + (int64_t)(r - sc->waves) * sc->ctas;
      if (p >= sc->num_pieces()) return false;
      const int32_t T = sc->tail_units;
      const int32_t k = (int32_t)(p / T);
      u = sc->tail_unit0() + (int32_t)(p - (int64_t)k * T);
      it0 = sc->piece_begin(k);
      it_end = sc->piece_begin(k + 1);
      complete = sc->pieces == 1;
      slot = complete ? -1 : (int32_t)p;
    }
    it = it0;
    range = r;
    return true;
  }

  LS_HD bool next(int32_t* uo, int32_t* s, bool* first, bool* last, bool* cpl, int32_t* sl) {
    while (range < 0 || it >= it_end) {
      if (!open_range(range + 1)) return false;
    }
    *uo = u;
    *s = it;
    *first = it == it0;
    *last = it + 1 == it_end;
    *cpl = complete;
    *sl = slot;
    ++it;
    return true;
  }
};
