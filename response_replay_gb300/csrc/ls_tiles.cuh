// ls_tiles.cuh -- the sequence of KV tiles one persistent CTA processes, derived from
// the work walk of ls_sched.h.  A unit is UnitRows consecutive response tokens of one
// query head; its items are the prompt splits (tile ranges of Tile keys) followed by
// the response's own keys (tiles 0 .. ceil(last token of the unit / Tile)).
#pragma once
#include <stdint.h>

#include "ls_sched.h"

struct TileRec {
  int32_t u;           // unit
  int32_t h, kvh, t0;  // query head, kv head, first token of the unit
  int32_t key0;        // first key of the tile (prompt position or response index)
  int32_t slot;        // partial-result slot of the tile's range (-1: complete unit)
  bool resp;           // response keys (causal) vs prompt keys
  bool first_of_unit, last_of_unit, complete;
};

template <int UnitRows, int Tile>
struct TileCursor {
  LsWalk walk;
  int32_t u, s, t, t_end, slot;
  bool item_first, item_last, item_complete, valid;
  int32_t R, g, nTB;
  int32_t h, kvh, t0;  // derived from u once per item, not per tile
  bool resp;

  __device__ TileCursor(const LsSched& sc, int cta, int32_t R_, int32_t g_)
      : walk(sc, cta), u(0), s(0), t(0), t_end(0), slot(-1), item_first(false), item_last(false),
        item_complete(false), valid(false), R(R_), g(g_), h(0), kvh(0), t0(0), resp(false) {
    nTB = (R + UnitRows - 1) / UnitRows;
  }

  __device__ bool open_item() {
    while (walk.next(&u, &s, &item_first, &item_last, &item_complete, &slot)) {
      h = u / nTB;
      t0 = (u - h * nTB) * UnitRows;
      kvh = h / g;
      resp = (s == walk.sc->nsplit);
      if (resp) {
        const int32_t qe = t0 + UnitRows < R ? t0 + UnitRows : R;
        t = 0;
        t_end = (qe + Tile - 1) / Tile;
      } else {
        walk.sc->split_tiles(s, &t, &t_end);
      }
      if (t < t_end) return true;
    }
    return false;
  }

  // The same walk as next(), reporting only whether the tile is the first / last of
  // its unit in this CTA (what an MMA issuer needs), so the common step is a compare
  // and an increment.
  __device__ bool next_flags(bool* first, bool* last) {
    if (!valid || t >= t_end) {
      valid = open_item();
      if (!valid) return false;
      *first = item_first;
    } else {
      *first = false;
    }
    ++t;
    *last = item_last && t >= t_end;
    return true;
  }

  __device__ bool next(TileRec* r) {
    if (!valid || t >= t_end) {
      valid = open_item();
      if (!valid) return false;
      r->first_of_unit = item_first;
    } else {
      r->first_of_unit = false;
    }
    r->u = u;
    r->h = h;
    r->t0 = t0;
    r->kvh = kvh;
    r->resp = resp;
    r->key0 = t * Tile;
    r->slot = slot;
    ++t;
    r->last_of_unit = item_last && t >= t_end;
    r->complete = item_complete;
    return true;
  }
};
