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
// Schedule ("full waves + split tail"): with C persistent CTAs and U units, the first
// W = floor(U / C) waves give each CTA whole units (unit w*C + c in wave w), so every
// CTA of a wave starts at prompt position 0 at the same time and walks the prompt in
// lockstep: CTAs that share a KV head read each KV tile from HBM once and from L2
// after that.  The remaining U - W*C units are cut into their items and the items are
// shared out evenly (a contiguous range per CTA), which balances the last wave; those
// are the only units that need the combine.
//
// Included by host and device code.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define LS_HD __host__ __device__ __forceinline__
#else
#define LS_HD inline
#endif

struct LsSched {
  int32_t units;       // U
  int32_t ctas;        // C (grid size)
  int32_t waves;       // W full waves
  int32_t ntiles;      // prompt KV tiles per unit: ceil(P / tile)
  int32_t tps;         // prompt tiles per split
  int32_t nsplit;      // non-empty prompt splits S (0 when P == 0)
  int64_t tail_items;  // (U - W*C) * (S + 1)

  LS_HD int32_t items_per_unit() const { return nsplit + 1; }
  LS_HD int32_t tail_unit0() const { return waves * ctas; }
  // Contiguous tail item range of CTA c, relative to the first tail item.
  LS_HD int64_t tail_begin(int32_t c) const { return (int64_t)c * tail_items / ctas; }
  // True when CTA c has tail items (with fewer tail items than CTAs, some ranges are
  // empty; those CTAs write no partial results and the combine skips them).
  LS_HD bool tail_nonempty(int32_t c) const { return tail_begin(c + 1) > tail_begin(c); }
  // CTA whose tail range holds tail item i (the last CTA whose range starts at or
  // before i, so CTAs with empty ranges are never returned).
  LS_HD int32_t tail_cta_of(int64_t i) const {
    return (int32_t)(((i + 1) * ctas + tail_items - 1) / tail_items - 1);
  }
  // Partial-result slot of unit u in CTA c (tail units only): slot 2c for the first
  // unit of c's tail range, 2c+1 for its last unit when that differs.
  LS_HD int32_t slot_of(int32_t c, int32_t u) const {
    int32_t first_u = tail_unit0() + (int32_t)(tail_begin(c) / items_per_unit());
    return 2 * c + (u == first_u ? 0 : 1);
  }
  // Prompt tile range [t0, t1) of split s.
  LS_HD void split_tiles(int32_t s, int32_t* t0, int32_t* t1) const {
    int32_t a = s * tps, b = a + tps;
    *t0 = a < ntiles ? a : ntiles;
    *t1 = b < ntiles ? b : ntiles;
  }
};

// Host: build the schedule for U units, a prompt of `ntiles` tiles, the caller's split
// request and a grid of at most `max_ctas` CTAs.
inline LsSched ls_make_sched(int32_t units, int32_t ntiles, int32_t num_splits, int32_t max_ctas) {
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
  int64_t total = (int64_t)units * (s.nsplit + 1);
  int32_t c = max_ctas;
  if ((int64_t)c > total) c = (int32_t)total;
  if (c < 1) c = 1;
  s.ctas = c;
  s.waves = units / c;
  s.tail_items = (int64_t)(units - s.waves * c) * (s.nsplit + 1);
  return s;
}

// Walks the item ranges of one CTA: W whole units, then its tail range.
// Usage:  LsWalk w(sched, c); int32_t u, s; bool first, last, complete;
//         while (w.next(&u, &s, &first, &last, &complete)) { ... }
// first/last: this item is the first/last of unit u that this CTA processes;
// complete: this CTA processes every item of u (only meaningful when last is set).
struct LsWalk {
  const LsSched* sc;   // the schedule (the kernel's __grid_constant__ parameter on the
                       // device, so the walk holds a pointer, not a register copy)
  int32_t cta;
  int32_t range;       // 0..waves-1 whole units, waves = tail
  int64_t item, end;   // current / end item (global item index u*(S+1)+s)
  int64_t range_begin;

  LS_HD LsWalk(const LsSched& s, int32_t c) : sc(&s), cta(c), range(-1), item(0), end(0), range_begin(0) {}

  LS_HD bool open_range(int32_t r) {
    const int64_t ipu = sc->items_per_unit();
    if (r < sc->waves) {
      range_begin = (int64_t)(r * sc->ctas + cta) * ipu;
      end = range_begin + ipu;
    } else if (r == sc->waves && sc->tail_items > 0) {
      int64_t base = (int64_t)sc->tail_unit0() * ipu;
      range_begin = base + sc->tail_begin(cta);
      end = base + sc->tail_begin(cta + 1);
    } else {
      return false;
    }
    item = range_begin;
    range = r;
    return true;
  }

  LS_HD bool next(int32_t* u, int32_t* s, bool* first, bool* last, bool* complete) {
    while (range < 0 || item >= end) {
      if (!open_range(range + 1)) return false;
    }
    const int64_t ipu = sc->items_per_unit();
    *u = (int32_t)(item / ipu);
    *s = (int32_t)(item % ipu);
    *first = (item == range_begin) || (*s == 0);
    *last = (item + 1 == end) || (*s == ipu - 1);
    int64_t ub = (int64_t)(*u) * ipu;
    *complete = (ub >= range_begin) && (ub + ipu <= end);
    ++item;
    return true;
  }
};
