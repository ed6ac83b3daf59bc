// Host check of the replay-attention work schedule (ls_sched.h): for many shapes,
// every (unit, item) is processed exactly once, "complete" is set exactly for units one
// CTA processes whole, the combine's CTA range for a split unit is exactly the set of
// CTAs that touched it, and partial-result slots never collide.
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>
#include <vector>

#include "ls_sched.h"

static int fail(const char* what, int U, int nt, int sp, int C) {
  std::printf("FAIL %s U=%d ntiles=%d splits=%d ctas=%d\n", what, U, nt, sp, C);
  return 1;
}

static int check(int U, int nt, int sp, int C) {
  LsSched s = ls_make_sched(U, nt, sp, C);
  const int ipu = s.items_per_unit();
  std::vector<int> seen((size_t)U * ipu, 0);
  std::map<int, std::set<int>> ctas_of_unit;
  std::map<int, int> complete_of_unit;   // unit -> cta that completed it
  std::map<int, std::set<int>> slot_writers;  // slot -> units
  for (int c = 0; c < s.ctas; ++c) {
    LsWalk w(s, c);
    int u, it, cur = -1;
    bool first, last, complete;
    bool expect_first = true;
    while (w.next(&u, &it, &first, &last, &complete)) {
      if (u < 0 || u >= U || it < 0 || it >= ipu) return fail("range", U, nt, sp, C);
      seen[(size_t)u * ipu + it]++;
      ctas_of_unit[u].insert(c);
      if (first != expect_first) return fail("first flag", U, nt, sp, C);
      if (!first && u != cur) return fail("unit change without first", U, nt, sp, C);
      cur = u;
      expect_first = last;
      if (last) {
        if (complete) {
          if (complete_of_unit.count(u)) return fail("completed twice", U, nt, sp, C);
          complete_of_unit[u] = c;
        } else {
          if (u < s.tail_unit0()) return fail("partial outside tail", U, nt, sp, C);
          slot_writers[s.slot_of(c, u)].insert(u);
        }
      }
    }
  }
  for (size_t i = 0; i < seen.size(); ++i)
    if (seen[i] != 1) return fail("item not processed exactly once", U, nt, sp, C);
  for (auto& kv : slot_writers)
    if (kv.second.size() != 1) return fail("slot collision", U, nt, sp, C);
  for (int u = 0; u < U; ++u) {
    const std::set<int>& cs = ctas_of_unit[u];
    if (cs.size() == 1) {
      if (!complete_of_unit.count(u)) return fail("single-CTA unit not complete", U, nt, sp, C);
      continue;
    }
    if (complete_of_unit.count(u)) return fail("split unit marked complete", U, nt, sp, C);
    if (u < s.tail_unit0()) return fail("wave unit split", U, nt, sp, C);
    const long long i0 = (long long)(u - s.tail_unit0()) * ipu;
    const int lo = s.tail_cta_of(i0), hi = s.tail_cta_of(i0 + ipu - 1);
    std::set<int> expect;
    for (int c = lo; c <= hi; ++c)
      if (s.tail_nonempty(c)) expect.insert(c);
    if (expect != cs) return fail("combine CTA range", U, nt, sp, C);
    for (int c = lo; c <= hi; ++c)
      if (s.tail_nonempty(c) &&
          (!slot_writers.count(s.slot_of(c, u)) || !slot_writers[s.slot_of(c, u)].count(u)))
        return fail("combine slot not written", U, nt, sp, C);
  }
  // full waves: wave w gives unit w*C + c to CTA c (lockstep order)
  for (int u = 0; u < s.tail_unit0(); ++u)
    if (complete_of_unit[u] != u % s.ctas) return fail("wave assignment", U, nt, sp, C);
  return 0;
}

int main() {
  int bad = 0, n = 0;
  const int Us[] = {1, 2, 3, 7, 8, 96, 151, 152, 153, 304, 384, 1000};
  const int nts[] = {0, 1, 2, 5, 32, 64, 257};
  const int sps[] = {1, 2, 3, 4, 32, 256, 1000};
  const int Cs[] = {1, 2, 5, 148, 152, 304};
  for (int U : Us)
    for (int nt : nts)
      for (int sp : sps)
        for (int C : Cs) {
          bad += check(U, nt, sp, C);
          ++n;
        }
  std::printf("%d/%d schedules ok\n", n - bad, n);
  return bad ? 1 : 0;
}
