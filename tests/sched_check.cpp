// Host check of the replay-attention work schedule (ls_sched.h): for many shapes,
// every (unit, item) is processed exactly once, ranges carry consistent first/last
// flags, "complete" is set exactly for units one CTA processes whole, every partial
// slot has exactly one writer and the combine's slots k*T + t of a tail unit are
// exactly the slots written for it, the waves keep their lockstep assignment, and the
// tail pieces balance the work to within 2% of the best piece count.  A second check
// walks the forward's tile cursor (ls_tiles.cuh) in its packed-members layout: every
// unit visits exactly the response key tiles its members' rows can see (member by
// member, each once), and the MMA issuer's flag walk sees the same tiles.  A third
// check walks the response-key backward's iteration ranges (ls_dkdv.h): every (KV head,
// key tile, query head, query tile >= key tile) once, segments flagged first/last at
// key-tile and range boundaries, "complete" exactly for key tiles one CTA holds whole,
// every partial slot written once, the combine's slot list of each split key tile equal
// to the slots written for it, and at most ceil(total / C) iterations per CTA.
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>
#include <vector>

#include "ls_dkdv.h"
#include "ls_sched.h"
#include "ls_tiles.cuh"

static int fail(const char* what, int U, int nt, int sp, int C) {
  std::printf("FAIL %s U=%d ntiles=%d splits=%d ctas=%d\n", what, U, nt, sp, C);
  return 1;
}

static int check(int U, int nt, int sp, int C, int max_pieces = 64) {
  LsSched s = ls_make_sched(U, nt, sp, C, max_pieces);
  const int ipu = s.items_per_unit();
  if (s.tail_units != U - s.waves * s.ctas || s.tail_units < 0 || s.tail_units >= s.ctas)
    return fail("tail units", U, nt, sp, C);
  if (s.pieces < 1 || s.pieces > ipu || s.pieces > max_pieces) return fail("piece count", U, nt, sp, C);
  std::vector<int> seen((size_t)U * ipu, 0);
  std::map<int, int> complete_of_unit;         // unit -> cta that completed it
  std::map<int, std::set<int>> slots_of_unit;  // unit -> partial slots written
  std::map<int, int> writers_of_slot;
  for (int c = 0; c < s.ctas; ++c) {
    LsWalk w(s, c);
    int u, it, slot, cur = -1, cur_slot = -2;
    bool first, last, complete;
    bool expect_first = true;
    int n = 0;
    while (w.next(&u, &it, &first, &last, &complete, &slot)) {
      ++n;
      if (u < 0 || u >= U || it < 0 || it >= ipu) return fail("range", U, nt, sp, C);
      seen[(size_t)u * ipu + it]++;
      if (first != expect_first) return fail("first flag", U, nt, sp, C);
      if (!first && (u != cur || slot != cur_slot)) return fail("range change without first", U, nt, sp, C);
      cur = u;
      cur_slot = slot;
      expect_first = last;
      if (complete != (slot < 0)) return fail("complete vs slot", U, nt, sp, C);
      if (last) {
        if (complete) {
          if (complete_of_unit.count(u)) return fail("completed twice", U, nt, sp, C);
          complete_of_unit[u] = c;
        } else {
          if (u < s.tail_unit0()) return fail("partial outside tail", U, nt, sp, C);
          if (writers_of_slot[slot]++) return fail("slot written twice", U, nt, sp, C);
          slots_of_unit[u].insert(slot);
        }
      }
    }
    if ((n > 0) != s.cta_has_work(c)) return fail("cta_has_work", U, nt, sp, C);
  }
  for (size_t i = 0; i < seen.size(); ++i)
    if (seen[i] != 1) return fail("item not processed exactly once", U, nt, sp, C);
  for (int u = 0; u < U; ++u) {
    if (complete_of_unit.count(u)) {
      if (slots_of_unit.count(u)) return fail("complete unit with partials", U, nt, sp, C);
      continue;
    }
    if (!s.has_partials() || u < s.tail_unit0()) return fail("unit neither complete nor split", U, nt, sp, C);
    std::set<int> expect;
    for (int k = 0; k < s.pieces; ++k) expect.insert(k * s.tail_units + (u - s.tail_unit0()));
    if (expect != slots_of_unit[u]) return fail("combine slots", U, nt, sp, C);
  }
  // full waves: wave w gives unit w*C + c to CTA c (lockstep order)
  for (int u = 0; u < s.tail_unit0(); ++u)
    if (complete_of_unit[u] != u % s.ctas) return fail("wave assignment", U, nt, sp, C);
  // the chosen piece count is within 2% of the best one
  if (s.tail_units > 0) {
    double best = 1e30;
    for (int q = 1; q <= ipu && q <= 64; ++q) {
      const double cq = ls_tail_cost(s.tail_units, q, s.ctas);
      if (cq < best) best = cq;
    }
    if (ls_tail_cost(s.tail_units, s.pieces, s.ctas) > best * 1.02 + 1e-12)
      return fail("tail balance", U, nt, sp, C);
  }
  return 0;
}

// Packed members: `members` responses of R tokens numbered back to back (RT tokens), a
// tile holding 128 / pack tokens of one KV head, `tiles` tiles per unit.
template <bool kTb>
static int check_packed(int R, int members, int pack, int hkv, int nt, int sp, int C) {
  const int tb_major = kTb ? 1 : 0;
  constexpr int kTile = 128, kUnitRows = 256;
  const int RT = R * members, tpt = kTile / pack;
  const int tiles = RT <= tpt ? 1 : 2, tpu = tiles * tpt;
  const int nTB = (RT + tpu - 1) / tpu, U = hkv * nTB;
  LsSched s = ls_make_sched(U, nt, sp, C);
  s.tb_major = tb_major;
  // the unit's KV head and first token under either numbering
  auto kvh_of = [&](int u) { return tb_major ? u % hkv : u / nTB; };
  auto t0_of = [&](int u) { return (tb_major ? u / hkv : u % nTB) * tpu; };
  std::map<int, std::multiset<std::pair<int, int>>> got;  // unit -> (member, first key)
  for (int c = 0; c < s.ctas; ++c) {
    TileCursor<kUnitRows, kTile, 2, kTb, true> cur(s, c, R, pack, pack, tiles, INT32_MAX, RT);
    TileCursor<kUnitRows, kTile, 2, kTb, true> flags(s, c, R, pack, pack, tiles, INT32_MAX, RT);
    TileRec r;
    bool f0, l0;
    int n = 0, nf = 0;
    while (cur.next(&r)) {
      ++n;
      if (!flags.next_flags(&f0, &l0) || f0 != r.first_of_unit || l0 != r.last_of_unit) {
        std::printf("FAIL packed flag walk R=%d members=%d pack=%d\n", R, members, pack);
        return 1;
      }
      ++nf;
      if (r.t0 != t0_of(r.u) || r.kvh != kvh_of(r.u)) {
        std::printf("FAIL packed unit decode R=%d members=%d pack=%d\n", R, members, pack);
        return 1;
      }
      if (r.resp) {
        int m, key;
        packed_resp_tile<kTile>(r.key0, r.t0 / R, R, &m, &key);
        got[r.u].insert({m, key});
      }
    }
    if (flags.next_flags(&f0, &l0)) {
      std::printf("FAIL packed flag walk longer R=%d members=%d pack=%d\n", R, members, pack);
      return 1;
    }
    (void)nf;
  }
  for (int u = 0; u < U; ++u) {
    std::multiset<std::pair<int, int>> want;
    const int t0 = t0_of(u), ve = t0 + tpu < RT ? t0 + tpu : RT;
    for (int m = t0 / R; m * R < ve; ++m) {
      const int e = (ve < (m + 1) * R ? ve : (m + 1) * R) - m * R;  // last row's token + 1
      for (int k = 0; k * kTile < e; ++k) want.insert({m, k * kTile});
    }
    if (got[u] != want) {
      std::printf("FAIL packed response tiles R=%d members=%d pack=%d hkv=%d unit=%d\n", R,
                  members, pack, hkv, u);
      return 1;
    }
  }
  return 0;
}

// lens: ragged members (segments of one response), empty for a single response
static int check_dkdv(int R, int g, int hkv, int C, const std::vector<int>& lens = {}) {
  LsSegs seg;
  seg.n = 1;
  seg.off[0] = 0;
  seg.off[1] = R;
  if (!lens.empty()) {
    seg.n = (int)lens.size();
    R = 0;
    for (int i = 0; i < seg.n; ++i) {
      R += lens[i];
      seg.off[i + 1] = R;
    }
  }
  const LsDkdvGeom gm = ls_make_dkdv_geom(R, g, hkv, C, &seg);
  auto bad = [&](const char* what) {
    std::printf("FAIL dkdv %s R=%d g=%d hkv=%d C=%d segments=%d\n", what, R, g, hkv, C, seg.n);
    return 1;
  };
  // the query tiles key tile kt must meet: up to the end of its last key's segment
  auto want_span = [&](int kt) {
    const int last = (kt + 1) * 128 < R ? (kt + 1) * 128 - 1 : R - 1;
    int k = 0;
    while (seg.off[k + 1] <= last) ++k;
    return (seg.off[k + 1] + 127) / 128 - kt;
  };
  if (gm.ctas > C || gm.ctas < (gm.total > 0 ? 1 : 0)) return bad("grid");
  const int nT = gm.nT;
  std::map<std::vector<int>, int> seen;                // (kvh, kt, h, tt) -> count
  std::map<std::pair<int, int>, std::vector<int>> written;  // key tile -> slots (cta order)
  std::map<std::pair<int, int>, int> complete_by;
  std::set<int> slots;
  for (int b = 0; b < gm.ctas; ++b) {
    LsDkdvWalk w(gm, b);
    LsDkdvIter it;
    int n = 0;
    bool open = false;
    int ckvh = -1, ckt = -1;
    while (w.next(&it)) {
      ++n;
      if (it.tt < it.kt || it.tt >= it.kt + want_span(it.kt) || it.h / g != it.kvh)
        return bad("iteration");
      if (++seen[{it.kvh, it.kt, it.h, it.tt}] != 1) return bad("visited twice");
      const bool new_tile = it.kvh != ckvh || it.kt != ckt;
      if (it.first != new_tile) return bad("first flag");
      if (new_tile && open) return bad("segment not closed");
      open = true;
      ckvh = it.kvh;
      ckt = it.kt;
      if (it.last) {
        open = false;
        const auto key = std::make_pair(it.kvh, it.kt);
        if (it.complete) {
          if (complete_by.count(key) || written.count(key)) return bad("complete twice");
          complete_by[key] = b;
        } else {
          if (it.slot != 2 * b && it.slot != 2 * b + 1) return bad("slot range");
          if (!slots.insert(it.slot).second) return bad("slot reused");
          written[key].push_back(it.slot);
        }
      }
    }
    if (open) return bad("range ends inside a segment");
    if (n > gm.per_cta) return bad("balance");
  }
  long long want = 0;
  for (int kt = 0; kt < nT; ++kt) want += (long long)hkv * g * want_span(kt);
  if ((long long)seen.size() != want) return bad("coverage");
  // the combine's view of each split key tile
  for (int c = 0; c < hkv; ++c)
    for (int kt = 0; kt < nT; ++kt) {
      const auto key = std::make_pair(c, kt);
      const long long s = gm.tile_begin(c, kt), e = s + gm.tile_iters(kt);
      const int b0 = (int)(s / gm.per_cta), b1 = (int)((e - 1) / gm.per_cta);
      if (b0 == b1) {
        if (!complete_by.count(key) || complete_by[key] != b0) return bad("complete owner");
        continue;
      }
      std::vector<int> expect;
      for (int b = b0; b <= b1; ++b) expect.push_back(gm.slot(b, s));
      if (written[key] != expect) return bad("combine slots");
    }
  return 0;
}

int main() {
  int bad = 0, n = 0;
  int dn = 0, dbad = 0;
  for (int R : {1, 100, 128, 129, 1000, 4096, 8192})
    for (int g : {1, 6, 8})
      for (int hkv : {1, 4})
        for (int C : {1, 3, 148, 152}) {
          dbad += check_dkdv(R, g, hkv, C);
          ++dn;
        }
  // ragged members: a cycle of the 4,194,304-position workload's lengths, short and
  // empty members, members ending inside and on tile boundaries
  const std::vector<std::vector<int>> raggeds = {
      {6012, 5295, 2370, 5318, 2053, 7773, 3591, 959}, {1, 0, 5, 300, 0, 128, 127, 129},
      {128, 128, 256}, {7, 1000, 3}, {4096, 1}};
  for (const auto& l : raggeds)
    for (int g : {1, 6})
      for (int C : {1, 7, 152}) {
        dbad += check_dkdv(0, g, 4, C, l);
        ++dn;
      }
  std::printf("%d/%d response-key walks ok\n", dn - dbad, dn);
  bad += dbad;
  const int Us[] = {1, 2, 3, 7, 8, 96, 151, 152, 153, 304, 384, 768, 1000};
  const int nts[] = {0, 1, 2, 5, 32, 64, 257, 16384};
  const int sps[] = {1, 2, 3, 4, 32, 256, 1000};
  const int Cs[] = {1, 2, 5, 148, 152, 304};
  for (int U : Us)
    for (int nt : nts)
      for (int sp : sps)
        for (int C : Cs) {
          bad += check(U, nt, sp, C);
          ++n;
        }
  // the latent backward's cap of 256 pieces (a lone unit spread over every CTA)
  for (int U : {1, 2, 3, 152, 153})
    for (int nt : {0, 5, 257, 65536})
      for (int sp : {1, 256, 1000})
        for (int C : {1, 152, 304}) {
          bad += check(U, nt, sp, C, 256);
          ++n;
        }
  // the two launches of the 2,097,152-position workload: 384 forward and 768 backward
  // units over 152 CTAs, 256 splits of 64 tiles
  for (int U : {4, 384, 768}) {
    LsSched s = ls_make_sched(U, 16384, 256, 152);
    std::printf("U=%d: %d waves, %d tail units in %d pieces\n", U, s.waves, s.tail_units, s.pieces);
  }
  int pn = 0, pbad = 0;
  for (int R : {1, 2, 5, 16, 21, 22, 77, 127, 128, 129, 255})
    for (int members : {2, 3, 8, 100})
      for (int pack : {2, 6, 8})
        for (int hkv : {1, 4})
          for (int C : {1, 7, 152})
            for (int nt : {0, 7}) {
              pbad += check_packed<false>(R, members, pack, hkv, nt, 3, C);
              pbad += check_packed<true>(R, members, pack, hkv, nt, 3, C);
              pn += 2;
            }
  bad += pbad;
  std::printf("%d/%d packed-member walks ok\n", pn - pbad, pn);
  std::printf("%d/%d schedules ok\n", n - bad + pbad + dbad, n);
  return bad ? 1 : 0;
}
