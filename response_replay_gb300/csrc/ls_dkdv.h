// ls_dkdv.h -- how the backward's response-key work (dK, dV of the response's own keys)
// is spread over the grid.
//
// The work of KV head c is the set of (key tile kt, query head h of the group, query
// tile tt >= kt) iterations: a 128-key tile of the response meets every later 128-token
// query tile of each of the g query heads of its group (the causal R x R triangle), so
// key tile kt has n_kt = g (nT - kt) iterations.  All iterations are numbered in one
// sequence (KV head, then key tile, then query head, then query tile) and CTA b takes the
// contiguous range [b c, (b + 1) c) with c = ceil(total / C): every CTA gets the same
// number of iterations even though key tile 0 has nT times the work of the last one.
//
// A CTA's range cuts it into segments, one per key tile it touches.  A segment that holds
// a whole key tile writes dK/dV directly; the segments of a key tile that spans several
// CTAs write partial sums, into slot 2b when the segment is its CTA's first and 2b + 1
// when it is the CTA's last, and a combine launch adds them in CTA order (fixed order:
// deterministic).  A CTA range has at most one segment of each kind, so the slots are
// unique.
//
// Ragged members replayed in one launch form one response of several segments
// (ls_sched.h, LsSegs); a key then meets only the query tiles up to the end of its own
// segment, so key tile kt's span of query tiles comes from a table instead of nT - kt.
//
// Included by host and device code.
#pragma once
#include <stdint.h>

#include "ls_sched.h"

#ifdef __CUDACC__
#define LS_DK_HD __host__ __device__ __forceinline__
#else
#define LS_DK_HD inline
#endif

constexpr int kLsMaxDkTiles = 1024;  // key tiles of a segmented response (131,072 tokens)

struct LsDkdvGeom {
  int32_t nT;       // key (and query) tiles of 128 tokens: ceil(R / 128)
  int32_t g;        // query heads per KV head
  int32_t hkv;      // KV heads
  int64_t ikv;      // iterations per KV head: g nT (nT + 1) / 2 (one segment)
  int64_t total;    // hkv * ikv
  int64_t per_cta;  // c
  int32_t ctas;     // ceil(total / c)
  int32_t ragged;   // spans from pre[] (several segments)
  int32_t pre[kLsMaxDkTiles + 1];  // ragged: query tiles met by key tiles 0 .. kt-1

  // Query tiles key tile kt meets, the first iteration of key tile kt of KV head c, and
  // its iteration count.
  LS_DK_HD int32_t span(int32_t kt) const { return ragged ? pre[kt + 1] - pre[kt] : nT - kt; }
  LS_DK_HD int64_t tile_begin(int32_t c, int32_t kt) const {
    const int64_t before = ragged ? (int64_t)pre[kt]
                                  : (int64_t)kt * nT - (int64_t)kt * (kt - 1) / 2;
    return (int64_t)c * ikv + (int64_t)g * before;
  }
  LS_DK_HD int64_t tile_iters(int32_t kt) const { return (int64_t)g * span(kt); }
  // Partial-sum slot of CTA b's segment of a key tile that starts at iteration s.
  LS_DK_HD int32_t slot(int32_t b, int64_t s) const {
    return s <= (int64_t)b * per_cta ? 2 * b : 2 * b + 1;
  }
};

// segs: the response's segments (NULL or one segment: a single response); with several
// segments nT must not exceed kLsMaxDkTiles (the caller checks).
inline LsDkdvGeom ls_make_dkdv_geom(int32_t R, int32_t g, int32_t hkv, int32_t max_ctas,
                                    const LsSegs* segs = nullptr) {
  LsDkdvGeom d;
  d.nT = (R + 127) / 128;
  d.g = g;
  d.hkv = hkv;
  d.ragged = segs && segs->n > 1 && d.nT <= kLsMaxDkTiles ? 1 : 0;
  d.pre[0] = 0;
  if (d.ragged) {
    for (int32_t kt = 0; kt < d.nT; ++kt) {
      const int32_t last = (kt + 1) * 128 < R ? (kt + 1) * 128 - 1 : R - 1;
      int32_t lo, hi;
      ls_seg_bounds(*segs, last, &lo, &hi);  // the last key's segment ends latest
      d.pre[kt + 1] = d.pre[kt] + ((hi + 127) / 128 - kt);
    }
    d.ikv = (int64_t)g * d.pre[d.nT];
  } else {
    d.ikv = (int64_t)g * d.nT * (d.nT + 1) / 2;
  }
  d.total = d.ikv * hkv;
  const int32_t C = max_ctas > 0 ? max_ctas : 1;
  d.per_cta = d.total > 0 ? (d.total + C - 1) / C : 1;
  d.ctas = (int32_t)((d.total + d.per_cta - 1) / d.per_cta);
  return d;
}

// One iteration of a CTA's range.
struct LsDkdvIter {
  int32_t kvh, kt, h, tt;  // KV head, key tile, query head, query tile
  bool first, last;        // first / last iteration of its segment
  bool complete;           // the segment is the whole key tile
  int32_t slot;            // partial-sum slot when not complete
};

// Walks CTA b's iterations in order.
struct LsDkdvWalk {
  const LsDkdvGeom* gm;
  int32_t b;
  int64_t i, r0, r1;        // current iteration, CTA range [r0, r1)
  int32_t kvh, kt, hh, tt;  // position of iteration i
  int64_t ts, te;           // range of the current key tile

  LS_DK_HD LsDkdvWalk(const LsDkdvGeom& g_, int32_t b_) : gm(&g_), b(b_) {
    r0 = (int64_t)b * gm->per_cta;
    r1 = r0 + gm->per_cta < gm->total ? r0 + gm->per_cta : gm->total;
    i = r0;
    kvh = kt = hh = tt = 0;
    ts = te = 0;
    if (i < r1) {
      kvh = (int32_t)(i / gm->ikv);
      int64_t r = i - (int64_t)kvh * gm->ikv;
      kt = 0;
      while (r >= gm->tile_iters(kt)) {
        r -= gm->tile_iters(kt);
        ++kt;
      }
      const int32_t span = gm->span(kt);
      hh = (int32_t)(r / span);
      tt = kt + (int32_t)(r - (int64_t)hh * span);
      ts = gm->tile_begin(kvh, kt);
      te = ts + gm->tile_iters(kt);
    }
  }

  LS_DK_HD bool next(LsDkdvIter* it) {
    if (i >= r1) return false;
    it->kvh = kvh;
    it->kt = kt;
    it->h = kvh * gm->g + hh;
    it->tt = tt;
    const int64_t seg0 = ts > r0 ? ts : r0, seg1 = te < r1 ? te : r1;
    it->first = i == seg0;
    it->last = i + 1 == seg1;
    it->complete = ts >= r0 && te <= r1;
    it->slot = it->complete ? -1 : gm->slot(b, ts);
    ++i;
    if (++tt == kt + gm->span(kt)) {  // next query head, or next key tile
      if (++hh == gm->g) {
        hh = 0;
        if (++kt == gm->nT) {
          kt = 0;
          ++kvh;
        }
        ts = te;
        te = ts + gm->tile_iters(kt);
      }
      tt = kt;
    }
    return true;
  }
};
