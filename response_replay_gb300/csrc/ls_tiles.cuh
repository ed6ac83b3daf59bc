// ls_tiles.cuh -- the sequence of KV tiles one persistent CTA processes, derived from
// the work walk of ls_sched.h.  A unit is UnitRows query rows that share a KV head:
// with pack = 1, UnitRows consecutive response tokens of one query head; with pack > 1
// (grouped-query packing, for short responses; pack divides g), the rows of consecutive
// tokens for a group of pack query heads of one KV head, a tile holding floor(Tile /
// pack) whole tokens.  Unit groups are numbered grp = h / pack.  Its items
// are the prompt splits (tile ranges of Tile keys) followed by the response's own keys
// (tiles 0 .. ceil(last token of the unit / Tile)).
//
// A forward launch over several responses of equal length R ("members") runs in one of
// two layouts (kMode):
//   1  units of one member each: member m's units follow those of members 0 .. m-1
//      (upm units per member); used when tiles hold one head's tokens (pack = 1).
//   2  members packed: the members' tokens are numbered back to back (member m's token t
//      is number m R + t of RT = members R) and units cover that sequence, so a tile may
//      hold rows of several members, all sharing each prompt K/V tile.  The response
//      item of a unit then walks the response keys of every member it holds, member by
//      member; the softmax masks the rows of the other members.
// kMode 0 is the one-response walk; kMode 3 the same for one response cut into segments
// (ragged members back to back, ls_sched.h LsSegs): a unit's response walk starts at the
// key tile of its first token's segment.
#pragma once
#include <stdint.h>

#include "ls_sched.h"

// Compiled for the device and, by the schedule checker, for the host.
#ifdef __CUDACC__
#define LS_TILE_HD __host__ __device__
#else
#define LS_TILE_HD
#endif

// Unit numbering.  Group grp is a query head (pack = 1, ngrp = Hq groups) or a KV head
// (packed, ngrp = Hkv), tb the unit's token block (nTB blocks).  Group major (unit = grp
// nTB + tb) puts the units of one head next to each other, so a persistent wave holds
// few KV heads and each prompt K/V tile serves many CTAs from L2.  Token block major
// (unit = tb ngrp + grp) puts units of neighbouring token blocks in a wave, whose
// response items (causal keys up to the block) are about as long as each other: used
// when those items are a large share of the work (short prompts), where group major
// would leave every wave waiting on its one longest unit.
LS_TILE_HD inline void unit_coords(int32_t ul, int32_t ngrp, int32_t nTB, bool tb_major,
                                   int32_t* grp, int32_t* tb) {
  if (tb_major) {
    *tb = ul / ngrp;
    *grp = ul - *tb * ngrp;
  } else {
    *grp = ul / nTB;
    *tb = ul - *grp * nTB;
  }
}

struct TileRec {
  int32_t u;           // unit
  int32_t m;           // member (response) of the unit
  int32_t h, kvh, t0;  // first query head, kv head, first token of the unit (in its member)
  int32_t key0;        // first key of the tile (prompt position or response index)
  int32_t slot;        // partial-result slot of the tile's range (-1: complete unit)
  bool resp;           // response keys (causal) vs prompt keys
  bool first_of_unit, last_of_unit, complete;
};

// kMode 2: the member and key tile of response tile `key0` (as TileCursor reports it:
// the tile's index in the unit's response walk, times Tile) of the unit whose first
// member is rm; the members' responses have R < 2 Tile tokens (packing is for short
// responses), so each has rnt = 1 or 2 key tiles.
template <int Tile>
LS_HD void packed_resp_tile(int32_t key0, int32_t rm, int32_t R, int32_t* m,
                                                 int32_t* key) {
  const int32_t t = key0 / Tile, rnt = R > Tile ? 2 : 1;
  const int32_t dm = rnt == 1 ? t : t >> 1;
  *m = rm + dm;
  *key = (t - dm * rnt) * Tile;
}

// kTbMajor: units numbered token block major (unit_coords); kPacked: tiles hold pack > 1
// heads (grouped-query packing).  Template parameters, so that the one-head, group-major
// walk of long responses compiles to the plainest decode (it sits in every role's inner
// loop, and measured slower by 1% with the general forms compiled in).
template <int UnitRows, int Tile, int kMode = 0, bool kTbMajor = false, bool kPacked = true>
struct TileCursor {
  LsWalk walk;
  int32_t u, s, t, t_end, slot;
  bool item_first, item_last, item_complete, valid;
  int32_t R, g, pack, tok_per_unit, nTB, upm, RT;
  int32_t m, h, kvh, t0;  // derived from u once per item, not per tile
  bool resp;

  // RT_: tokens the units cover (R, or members x R in kMode 2; 0 means R).
  LS_TILE_HD TileCursor(const LsSched& sc, int cta, int32_t R_, int32_t g_, int32_t pack_ = 1,
                        int32_t tiles_ = UnitRows / Tile, int32_t upm_ = INT32_MAX,
                        int32_t RT_ = 0)
      : walk(sc, cta), u(0), s(0), t(0), t_end(0), slot(-1), item_first(false), item_last(false),
        item_complete(false), valid(false), R(R_), g(g_), pack(pack_), upm(upm_),
        RT(RT_ > 0 ? RT_ : R_), m(0), h(0), kvh(0), t0(0), resp(false) {
    tok_per_unit = tiles_ * (Tile / pack);
    nTB = (RT + tok_per_unit - 1) / tok_per_unit;

  }



  LS_TILE_HD bool open_item() {
    while (walk.next(&u, &s, &item_first, &item_last, &item_complete, &slot)) {
      int32_t ul = u;  // unit within its member
      if constexpr (kMode == 1) {
        m = u / upm;
        ul = u - m * upm;
      }
      int32_t grp;                     // query head (pack 1) or kv head (packed)
      if constexpr (kTbMajor) {
        int32_t ngrp = (kMode == 1 ? upm : walk.sc->units) / nTB, tb;
        unit_coords(ul, ngrp, nTB, true, &grp, &tb);
        t0 = tb * tok_per_unit;
      } else {
        grp = ul / nTB;
        t0 = (ul - grp * nTB) * tok_per_unit;
      }
      if constexpr (kPacked) {         // first query head of the unit's group, KV head
        h = grp * pack;
        kvh = h / g;
      } else {                         // pack is 1 here; this form measured fastest
        kvh = pack == 1 ? grp / g : grp;
        h = pack == 1 ? grp : grp * g;
      }
      resp = (s == walk.sc->nsplit);
      if (resp) {
        t = 0;
        if constexpr (kMode == 2) {
          // Members rm .. ml have rows in the unit.  Each sees keys up to its last row in
          // the unit: all rnt key tiles of its response, except member ml, whose rows may
          // stop early.  Tile t (key0 = t Tile) is key tile t % rnt of member
          // rm + t / rnt (packed_resp_tile).
          const int32_t ve = t0 + tok_per_unit < RT ? t0 + tok_per_unit : RT;
          const int32_t rm = t0 / R, ml = (ve - 1) / R;
          const int32_t rnt = (R + Tile - 1) / Tile;
          t_end = (ml - rm) * rnt + (ve - ml * R + Tile - 1) / Tile;
        } else {
          const int32_t qe = t0 + tok_per_unit < R ? t0 + tok_per_unit : R;
          t_end = (qe + Tile - 1) / Tile;
          if constexpr (kMode == 3) {  // keys before the first token's segment: unseen
            int32_t lo, hi;
            ls_seg_bounds(walk.sc->seg, t0, &lo, &hi);
            t = lo / Tile;
          }
        }
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
  LS_TILE_HD bool next_flags(bool* first, bool* last) {
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

  LS_TILE_HD bool next(TileRec* r) {
    if (!valid || t >= t_end) {
      valid = open_item();
      if (!valid) return false;
      r->first_of_unit = item_first;
    } else {
      r->first_of_unit = false;
    }
    r->u = u;
    r->m = m;
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
