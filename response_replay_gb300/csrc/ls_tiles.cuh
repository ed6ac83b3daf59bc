// ls_tiles.cuh -- the sequence of KV tiles one persistent CTA processes, derived from
// the work walk of ls_sched.h.  A unit is UnitRows query rows that share a KV head:
// with pack = 1, UnitRows consecutive response tokens of one query head; with pack = g
// (grouped-query packing, for short responses), the rows of consecutive tokens for all
// g query heads of one KV head, a tile holding floor(Tile / g) whole tokens.  Its items
// are the prompt splits (tile ranges of Tile keys) followed by the response's own keys
// (tiles 0 .. ceil(last token of the unit / Tile)).
#pragma once
#include <stdint.h>

#include "ls_sched.h"

struct TileRec {
  int32_t u;           // unit
  int32_t h, kvh, t0;  // first query head, kv head, first token of the unit
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
  int32_t R, g, pack, tok_per_unit, nTB;
  int32_t h, kvh, t0;  // derived from u once per item, not per tile
  bool resp;

  __device__ TileCursor(const LsSched& sc, int cta, int32_t R_, int32_t g_, int32_t pack_ = 1,
                        int32_t tiles_ = UnitRows / Tile)
      : walk(sc, cta), u(0), s(0), t(0), t_end(0), slot(-1), item_first(false), item_last(false),
        item_complete(false), valid(false), R(R_), g(g_), pack(pack_), h(0), kvh(0), t0(0),
        resp(false) {
    tok_per_unit = tiles_ * (Tile / pack);
    nTB = (R + tok_per_unit - 1) / tok_per_unit;
  }

  __device__ bool open_item() {
    while (walk.next(&u, &s, &item_first, &item_last, &item_complete, &slot)) {
      const int32_t grp = u / nTB;  // query head (pack 1) or kv head (packed)
      t0 = (u - grp * nTB) * tok_per_unit;
      kvh = pack == 1 ? grp / g : grp;
      h = pack == 1 ? grp : grp * g;
      resp = (s == walk.sc->nsplit);
      if (resp) {
        const int32_t qe = t0 + tok_per_unit < R ? t0 + tok_per_unit : R;
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
