// Brute-force check of the work partition in xsymv_plan.h (host logic of the
// CUDA library): simulates the main kernel's per-warp loop and verifies that
// every column segment of the stored triangle is owned exactly once, that the
// row-partial slots of each block row have no holes, that the finaliser's
// block-row ranges are exactly the rows holding each column, and that the
// ordered-ticket chains visit exactly the contributors of every output chunk,
// in increasing warp order.  The same holds for a column window (the shard
// of a block-column split): only the window's stored columns are owned, the
// rows they miss hold nothing, and the closed-form row starts equal the sums
// of the row costs.
#include <cstdio>
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <set>
#include <vector>

#include "xsymv_plan.h"

using namespace xsymv;

static int g_G = 1;   // warps per block of the case being checked
static int g_c0 = 0, g_c1 = 0;   // column window of the case being checked

static int fail(const char* what, int n, int NB, int upper, long long W, int cd, int cg) {
  std::printf("FAIL %s n=%d NB=%d upper=%d W=%lld cd=%d cg=%d G=%d window=[%d,%d)\n", what, n, NB,
              upper, W, cd, cg, g_G, g_c0, g_c1);
  return 1;
}

// the warp table: rows Ia..Ib, first column ja in row Ia, end jb in row Ib,
// whole rows between; read this way it gives exactly the owned columns
static int check_warp_table(const Plan& p, const std::vector<std::vector<int>>& own,
                            const std::vector<std::vector<int>>& row_warps, long long Wmax, int cd,
                            int cg) {
  const int n = p.n, NB = p.NB, upper = p.upper, nb = p.nb;
  for (int w = 0; w < p.W; ++w) {
    int Ia, Ib;
    long long ja, jb;
    plan_warp_entry(p, w, &Ia, &Ib, &ja, &jb);
    for (int I = 0; I < nb; ++I) {
      const long long cb = plan_colbase(p, I), len = plan_rowlen(p, I);
      const long long a = I == Ia ? ja : cb, b = I == Ib ? jb : cb + len;
      for (long long c = 0; c < len; ++c) {
        const bool mine = I >= Ia && I <= Ib && cb + c >= a && cb + c < b;
        if (mine != (own[I][c] == w)) return fail("warp table", n, NB, upper, Wmax, cd, cg);
      }
    }
    if (ja > INT32_MAX || jb > INT32_MAX) return fail("warp table range", n, NB, upper, Wmax, cd, cg);
    // a row strictly between the warp's first and last rows is its alone:
    // the kernel writes that row partial straight to the block's slot
    for (int I = Ia + 1; I < Ib; ++I)
      if (row_warps[I].size() != 1 || row_warps[I][0] != w)
        return fail("middle row shared", n, NB, upper, Wmax, cd, cg);
  }
  return 0;
}

static int check(int n, int NB, int upper, long long Wmax, int cd, int cg, int c0 = 0,
                 int c1 = -1) {
  const Plan p = plan_make(n, NB, upper, Wmax, cd, cg, g_G, c0, c1);
  g_c0 = p.c0;
  g_c1 = p.c1;
  const bool full = p.c0 == 0 && p.c1 == n;
  const int G = p.G;
  const int nb = p.nb;
  // the window's columns of each block row, from the definition
  long long acc = 0;
  for (int I = 0; I < nb; ++I) {
    long long first = -1, count = 0;
    for (long long j = p.c0; j < p.c1; ++j) {
      const bool stored = upper ? j >= (long long)I * NB : j < std::min<long long>(n, (long long)(I + 1) * NB);
      if (!stored) continue;
      if (first < 0) first = j;
      if (j != first + count) return fail("row columns not contiguous", n, NB, upper, Wmax, cd, cg);
      ++count;
    }
    if (plan_rowlen(p, I) != count || (count > 0 && plan_colbase(p, I) != first))
      return fail("row columns", n, NB, upper, Wmax, cd, cg);
    // closed-form row start = the costs of the rows before
    if (plan_rowstart(p, I) != acc) return fail("row start", n, NB, upper, Wmax, cd, cg);
    acc += plan_rowcost(p, I);
  }
  if (plan_rowstart(p, nb) != acc || p.SC != acc) return fail("total cost", n, NB, upper, Wmax, cd, cg);
  // owners[I][c] = warp owning column c of block row I, from the kernel loop
  std::vector<std::vector<int>> own(nb);
  for (int I = 0; I < nb; ++I) own[I].assign((size_t)plan_rowlen(p, I), -1);
  std::vector<std::vector<int>> row_warps(nb);
  for (int w = 0; w < p.W; ++w) {
    const long long ce = plan_wstart(p, w + 1);
    long long cs = plan_wstart(p, w);
    int I = plan_row_of(p, cs);
    for (; cs < ce && I < nb; ++I) {
      const long long rcs = plan_rowstart(p, I);
      const long long rce = rcs + plan_rowcost(p, I);
      if (cs < rcs) return fail("range starts before row", n, NB, upper, Wmax, cd, cg);
      const long long c0 = plan_cols_before(p, I, cs - rcs);
      const long long c1 = plan_cols_before(p, I, (ce < rce ? ce : rce) - rcs);
      cs = rce;
      if (c0 >= c1) continue;
      for (long long c = c0; c < c1; ++c) {
        if (own[I][c] != -1) return fail("column owned twice", n, NB, upper, Wmax, cd, cg);
        own[I][c] = w;
        // the owner is the warp whose range holds the column's first cost unit
        if (plan_owner(p, rcs + plan_col_cost(p, I, c)) != w)
          return fail("owner rule", n, NB, upper, Wmax, cd, cg);
      }
      // the row-partial slot of the warp's block
      const int q = w / G - plan_first_owner(p, I) / G;
      if (q < 0 || q >= plan_nq(p, I) || q >= p.qmax)
        return fail("slot index", n, NB, upper, Wmax, cd, cg);
      row_warps[I].push_back(w);
    }
  }
  long long total = 0;
  for (int I = 0; I < nb; ++I) {
    for (int o : own[I])
      if (o < 0) return fail("column not owned", n, NB, upper, Wmax, cd, cg);
    total += (long long)own[I].size();
    if (row_warps[I].empty()) {
      // a row outside the window: no columns, no slots
      if (plan_rowlen(p, I) != 0 || plan_nq(p, I) != 0)
        return fail("empty row", n, NB, upper, Wmax, cd, cg);
      continue;
    }
    // the warps of a row are exactly first_owner .. last_owner, each once, so
    // its blocks are exactly first_owner/G .. last_owner/G: the slots have
    // no holes
    const int f = plan_first_owner(p, I), l = plan_last_owner(p, I);
    if ((int)row_warps[I].size() != l - f + 1) return fail("slot holes", n, NB, upper, Wmax, cd, cg);
    for (int k = 0; k <= l - f; ++k)
      if (row_warps[I][k] != f + k) return fail("slot order", n, NB, upper, Wmax, cd, cg);
    if (plan_nq(p, I) != l / G - f / G + 1) return fail("slot count", n, NB, upper, Wmax, cd, cg);
  }
  // total segments = stored columns per block row, as the report's triangle
  long long want = 0;
  for (long long j = p.c0; j < p.c1; ++j) want += upper ? j / NB + 1 : nb - j / NB;
  if (total != want) return fail("segment count", n, NB, upper, Wmax, cd, cg);
  // finaliser: column j gets column partials from block rows I0..I1
  for (int j = 0; j < n; ++j) {
    const int K = j / NB;
    const int I0 = upper ? 0 : K, I1 = upper ? K : nb - 1;
    for (int I = 0; I < nb; ++I) {
      const long long cb = plan_colbase(p, I), len = plan_rowlen(p, I);
      const bool has = j >= cb && j < cb + len;
      const bool in_window = j >= p.c0 && j < p.c1;
      if (has != (in_window && I >= I0 && I <= I1))
        return fail("finaliser rows", n, NB, upper, Wmax, cd, cg);
    }
  }
  // the diagonal-tile columns are the ones costed cg
  for (int I = 0; I < nb; ++I) {
    const long long d = plan_dlen(p, I), len = plan_rowlen(p, I), cb = plan_colbase(p, I);
    for (long long c = 0; c < len; ++c) {
      const long long j = cb + c;
      const bool diag = j >= (long long)I * NB && j < (long long)I * NB + NB;
      const long long next = c + 1 < len ? plan_col_cost(p, I, c + 1) : plan_rowcost(p, I);
      if (next - plan_col_cost(p, I, c) != (diag ? cg : cd))
        return fail("column cost", n, NB, upper, Wmax, cd, cg);
    }
    const long long ds = std::max<long long>((long long)I * NB, p.c0);
    const long long de = std::min<long long>({(long long)I * NB + NB, (long long)n, (long long)p.c1});
    if (d != std::max<long long>(0, de - ds)) return fail("dlen", n, NB, upper, Wmax, cd, cg);
  }
  if (p.W >= (1 << 24)) return fail("warp bits", n, NB, upper, Wmax, cd, cg);
  // the warp table (below) holds for any window; the ordered tickets are
  // used on the whole triangle only
  if (!full) return check_warp_table(p, own, row_warps, Wmax, cd, cg);
  // ordered tickets: contributors of chunk K = owners of its columns in any
  // row, plus the warps holding row K's partial slots
  std::vector<std::set<int>> contrib(nb);
  std::vector<std::set<int>> chunks_of(p.W);
  for (int I = 0; I < nb; ++I) {
    const long long cb = plan_colbase(p, I);
    for (size_t c = 0; c < own[I].size(); ++c) {
      const int K = (int)((cb + (long long)c) / NB);
      contrib[K].insert(own[I][c]);
      chunks_of[own[I][c]].insert(K);
    }
    for (int w : row_warps[I]) {
      contrib[I].insert(w);
      chunks_of[w].insert(I);
    }
  }
  for (int K = 0; K < nb; ++K) {
    const std::vector<int> v(contrib[K].begin(), contrib[K].end());
    if (v.empty() || plan_chain_first(p, K) != v[0])
      return fail("chain first", n, NB, upper, Wmax, cd, cg);
    for (size_t k = 0; k < v.size(); ++k) {
      const int want_next = k + 1 < v.size() ? v[k + 1] : -1;
      if (plan_chain_next(p, K, v[k]) != want_next)
        return fail("chain next", n, NB, upper, Wmax, cd, cg);
    }
    // link ranges sorted by first and last warp
    int pa = -1, pb = -1;
    for (int t = 0; t < plan_links(p, K); ++t) {
      int wa, wb;
      plan_link_range(p, K, t, &wa, &wb);
      if (wa < pa || wb < pb || wa > wb) return fail("link ranges", n, NB, upper, Wmax, cd, cg);
      pa = wa;
      pb = wb;
    }
  }
  if (check_warp_table(p, own, row_warps, Wmax, cd, cg)) return 1;
  // the same chains between groups of G consecutive warps (thread blocks)
  for (int G : {1, 3, 8}) {
    const int ng = (p.W + G - 1) / G;
    for (int K = 0; K < nb; ++K) {
      std::set<int> gs;
      for (int w : contrib[K]) gs.insert(w / G);
      const std::vector<int> v(gs.begin(), gs.end());
      if (plan_group_first(p, K, G) != v[0]) return fail("group first", n, NB, upper, Wmax, cd, cg);
      for (size_t k = 0; k < v.size(); ++k) {
        const int want_next = k + 1 < v.size() ? v[k + 1] : -1;
        if (plan_group_next(p, K, v[k], G) != want_next)
          return fail("group next", n, NB, upper, Wmax, cd, cg);
      }
    }
    for (int g = 0; g < ng; ++g) {
      const int w0 = g * G, w1 = std::min(p.W, w0 + G);
      const int Ia = plan_row_of(p, plan_wstart(p, w0));
      const int Ib = plan_row_of(p, plan_wstart(p, w1) - 1);
      std::set<int> want;
      for (int w = w0; w < w1; ++w) want.insert(chunks_of[w].begin(), chunks_of[w].end());
      std::vector<int> got;
      for (int K = plan_group_next_chunk(p, w0, w1, Ia, Ib, -1); K < nb;
           K = plan_group_next_chunk(p, w0, w1, Ia, Ib, K))
        got.push_back(K);
      if (got != std::vector<int>(want.begin(), want.end()))
        return fail("group chunks", n, NB, upper, Wmax, cd, cg);
      for (int I = Ia; I <= Ib; ++I) {
        long long ja, jb;
        const bool has = plan_group_cols(p, w0, w1, I, &ja, &jb);
        // the group's columns are the union of the columns of its warps that
        // own columns there (a contiguous run of warps)
        std::vector<int> slots;
        for (int w : row_warps[I])
          if (w >= w0 && w < w1) slots.push_back(w - plan_first_owner(p, I));
        if (has != !slots.empty()) return fail("group cols", n, NB, upper, Wmax, cd, cg);
        if (!has) continue;
        if ((int)slots.size() != slots.back() - slots.front() + 1)
          return fail("group warps", n, NB, upper, Wmax, cd, cg);
        for (long long c = 0; c < (long long)own[I].size(); ++c) {
          const long long j = plan_colbase(p, I) + c;
          const bool mine = own[I][c] >= w0 && own[I][c] < w1;
          if (mine != (j >= ja && j < jb)) return fail("group cols range", n, NB, upper, Wmax, cd, cg);
        }
      }
    }
  }
  return 0;
}

int main() {
  int bad = 0, cases = 0;
  const int sizes[] = {1, 2, 3, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 511, 700, 1025};
  const int edges[] = {32, 64, 128, 256, 512};
  const long long warps[] = {1, 2, 3, 7, 64, 300, 1000, 7296, 1000000};
  const int costs[][2] = {{1, 1}, {4, 6}, {4, 3}, {2, 7}, {5, 1}};
  for (int n : sizes)
    for (int NB : edges)
      for (int upper = 0; upper < 2; ++upper)
        for (long long W : warps)
          for (auto& c : costs)
            for (int G : {1, 8}) {
              g_G = G;
              bad += check(n, NB, upper, W, c[0], c[1]);
              ++cases;
            }
  // column windows (shards of a block-column split), every boundary kind:
  // at 0 / n, inside a diagonal tile, on a tile edge, a single column
  const long long wwarps[] = {1, 3, 64, 1000, 7296};
  for (int n : sizes)
    for (int NB : edges)
      for (int upper = 0; upper < 2; ++upper)
        for (long long W : wwarps)
          for (auto& c : costs)
            for (int G : {1, 8}) {
              const int wins[][2] = {{n / 3, n}, {0, (2 * n + 2) / 3}, {n / 4, (3 * n + 3) / 4},
                                     {1, n}, {0, n - 1}, {n / 2, n / 2 + 1},
                                     {std::min(n, NB), n}, {0, std::min(n, 2 * NB)}};
              for (auto& w : wins) {
                if (w[0] < 0 || w[0] >= w[1] || w[1] > n) continue;
                g_G = G;
                bad += check(n, NB, upper, W, c[0], c[1], w[0], w[1]);
                ++cases;
              }
            }
  std::printf("%d cases, %d failures\n", cases, bad);
  return bad ? 1 : 0;
}
