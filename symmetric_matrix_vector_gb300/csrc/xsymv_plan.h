// Work partition of one xSYMV call, shared by host dispatch and the kernels.
//
// The stored triangle is cut into block rows of NB rows (NB = the tile edge).
// Block row I owns one "column segment" per matrix column j that meets the
// stored triangle inside its rows:
//   upper ('U'): j = I*NB .. n-1        (diagonal tile first, then the rest)
//   lower ('L'): j = 0 .. min(n, I*NB+NB)-1   (off-diagonal first, diagonal last)
// Columns of the diagonal tile cost more than dense ones (masked loads), so
// the warps do not get equal column counts but equal cost: a dense column
// costs cd units, a diagonal-tile column cg units.  Costs are laid out row
// after row (block row 0 first); warp w takes the cost range
// [w*SC/W, (w+1)*SC/W) and owns the columns whose first cost unit falls in
// it, so every column has exactly one owner.
//
// Deterministic cross-warp accumulation (the role the report's ordered
// tickets play, "CUDA-xSYMV の実装と評価" §2.1, figure "Atomic"):
//   * a warp writes one column partial per column it owns, to Wc[I*n + j];
//   * the G warps of a thread block (warps b*G .. b*G+G-1) add their row
//     partials of block row I in warp order, and the block writes the sum to
//     slot q of that row, Wr[(I*qmax + q)*NB + r], q = b - (block of the
//     owner of the row's first column);
// a second kernel then sums those slots for every output element in a fixed
// order, so results are bit-identical from run to run.  Warp ranges are at
// least max(cd, cg) units long, so every warp between the owners of a row's
// first and last columns owns columns in that row, hence every block between
// their blocks does: no slot a finaliser reads is left unwritten.
#pragma once

#ifdef __CUDACC__
#define XSYMV_HD __host__ __device__ __forceinline__
#else
#define XSYMV_HD inline
#endif

namespace xsymv {

struct Plan {
  int n;            // matrix order
  int NB;           // tile edge (rows per block row)
  int nb;           // number of block rows, ceil(n / NB)
  int upper;        // 1: upper triangle stored, 0: lower
  int cd;           // cost of a dense column
  int cg;           // cost of a diagonal-tile column
  long long SC;     // total cost
  int W;            // warps sharing the cost (1 <= W <= SC / max(cd, cg))
  int G;            // warps per thread block: row partials are written per block
  int qmax;         // most blocks that touch one block row
  int c0, c1;       // column window: only the stored columns c0 <= j < c1
                    // are streamed (0, n: the whole triangle)
};

// The window: block row I holds the stored columns of its rows that lie in
// [c0, c1).  Upper: [max(I*NB, c0), c1); lower: [c0, min((I+1)*NB, n, c1)).
// Rows with no such column hold nothing and cost nothing; they are the last
// rows (upper) or the first ones (lower), so the rows that hold columns are
// consecutive.  With the whole triangle (c0 = 0, c1 = n) every row holds
// columns.

// first column (matrix index) of block row I's columns
XSYMV_HD long long plan_colbase(const Plan& p, int I) {
  if (!p.upper) return p.c0;
  const long long s = (long long)I * p.NB;
  return s > p.c0 ? s : (long long)p.c0;
}

XSYMV_HD long long plan_rowlen(const Plan& p, int I) {
  if (p.upper) {
    const long long s = plan_colbase(p, I);
    return p.c1 > s ? p.c1 - s : 0;
  }
  long long e = ((long long)I + 1) * p.NB;
  if (e > p.n) e = p.n;
  if (e > p.c1) e = p.c1;
  return e > p.c0 ? e - p.c0 : 0;
}

// columns of block row I that lie in its diagonal tile
XSYMV_HD long long plan_dlen(const Plan& p, int I) {
  long long s = (long long)I * p.NB, e = s + p.NB;
  if (e > p.n) e = p.n;
  if (e > p.c1) e = p.c1;
  if (s < p.c0) s = p.c0;
  return e > s ? e - s : 0;
}

// sum of floor(j / NB) over 0 <= j < m
XSYMV_HD long long plan_floor_sum(long long m, int NB) {
  const long long q = m / NB, r = m % NB;
  return (long long)NB * q * (q - 1) / 2 + q * r;
}

// column segments in block rows before I (0 <= I <= nb).  Column j of the
// window lies in block rows I' <= j/NB (upper) or I' >= j/NB (lower), so
// this is the sum over the window of min(I, j/NB + 1) (upper) or
// max(0, I - j/NB) (lower), in closed form.
XSYMV_HD long long plan_segstart(const Plan& p, int I) {
  const long long a = p.c0, b = p.c1;
  long long m = (long long)I * p.NB;   // columns below m lie in a row's diagonal tile or later
  m = m < a ? a : (m > b ? b : m);
  const long long fs = plan_floor_sum(m, p.NB) - plan_floor_sum(a, p.NB);
  if (p.upper) return (m - a) + fs + (long long)I * (b - m);
  return (long long)I * (m - a) - fs;
}

// diagonal-tile columns in block rows before I: the window's columns below
// min(I*NB, n) (each column lies in exactly one diagonal tile)
XSYMV_HD long long plan_diag_before(const Plan& p, int I) {
  long long e = (long long)I * p.NB;
  if (e > p.n) e = p.n;
  if (e > p.c1) e = p.c1;
  return e > p.c0 ? e - p.c0 : 0;
}

// first cost unit of block row I (0 <= I <= nb; I = nb gives the total)
XSYMV_HD long long plan_rowstart(const Plan& p, int I) {
  return (long long)p.cd * plan_segstart(p, I) + (long long)(p.cg - p.cd) * plan_diag_before(p, I);
}

XSYMV_HD long long plan_rowcost(const Plan& p, int I) {
  const long long d = plan_dlen(p, I);
  return (long long)p.cd * (plan_rowlen(p, I) - d) + (long long)p.cg * d;
}

// the row's columns come in two runs: upper = diagonal tile then dense,
// lower = dense then diagonal tile; (len1, unit1) describes the first run
XSYMV_HD void plan_runs(const Plan& p, int I, long long* len1, int* unit1, int* unit2) {
  const long long d = plan_dlen(p, I);
  if (p.upper) {
    *len1 = d;
    *unit1 = p.cg;
    *unit2 = p.cd;
  } else {
    *len1 = plan_rowlen(p, I) - d;
    *unit1 = p.cd;
    *unit2 = p.cg;
  }
}

// number of columns of block row I whose first cost unit lies before
// offset o (0 <= o <= rowcost) from the row's start
XSYMV_HD long long plan_cols_before(const Plan& p, int I, long long o) {
  long long len1;
  int u1, u2;
  plan_runs(p, I, &len1, &u1, &u2);
  if (o <= (long long)u1 * len1) return (o + u1 - 1) / u1;
  return len1 + (o - (long long)u1 * len1 + u2 - 1) / u2;
}

// cost offset of column c (0 <= c < rowlen) within block row I
XSYMV_HD long long plan_col_cost(const Plan& p, int I, long long c) {
  long long len1;
  int u1, u2;
  plan_runs(p, I, &len1, &u1, &u2);
  return c < len1 ? (long long)u1 * c : (long long)u1 * len1 + (long long)u2 * (c - len1);
}

// first cost unit of warp w (w = W gives SC)
XSYMV_HD long long plan_wstart(const Plan& p, int w) { return (long long)w * p.SC / p.W; }

// the warp whose range contains cost unit s
XSYMV_HD int plan_owner(const Plan& p, long long s) { return (int)(((s + 1) * p.W - 1) / p.SC); }

// warps owning the first and the last column of block row I (a row that
// holds columns)
XSYMV_HD int plan_first_owner(const Plan& p, int I) { return plan_owner(p, plan_rowstart(p, I)); }
XSYMV_HD int plan_last_owner(const Plan& p, int I) {
  return plan_owner(p, plan_rowstart(p, I) + plan_col_cost(p, I, plan_rowlen(p, I) - 1));
}
// row-partial slots of block row I: the blocks owning its columns (none for
// a row outside the window)
XSYMV_HD int plan_nq(const Plan& p, int I) {
  if (plan_rowlen(p, I) == 0) return 0;
  return plan_last_owner(p, I) / p.G - plan_first_owner(p, I) / p.G + 1;
}

// block row containing cost unit s (binary search: the last row starting at
// or before s, which holds columns when 0 <= s < SC)
XSYMV_HD int plan_row_of(const Plan& p, long long s) {
  int lo = 0, hi = p.nb - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (plan_rowstart(p, mid) <= s) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Build the plan for n, NB, uplo with at most Wmax warps in blocks of G; a
// dense column costs cd units and a diagonal-tile column cg units (cd, cg >=
// 1).  Only the stored columns c0 <= j < c1 are streamed (c1 < 0: n); the
// window must not be empty (0 <= c0 < c1 <= n).
inline Plan plan_make(int n, int NB, int upper, long long Wmax, int cd = 1, int cg = 1,
                      int G = 1, int c0 = 0, int c1 = -1) {
  Plan p{};
  p.n = n;
  p.NB = NB;
  p.nb = (n + NB - 1) / NB;
  p.upper = upper;
  p.cd = cd;
  p.cg = cg;
  p.c0 = c0;
  p.c1 = c1 < 0 ? n : c1;
  p.SC = n > 0 ? plan_rowstart(p, p.nb) : 0;
  const long long unit = cd > cg ? cd : cg;
  long long W = Wmax < p.SC / unit ? Wmax : p.SC / unit;
  p.W = (int)(W < 1 ? 1 : W);
  p.G = G < 1 ? 1 : G;
  p.qmax = 1;
  for (int I = 0; I < p.nb; ++I) {
    int q = plan_nq(p, I);
    if (q > p.qmax) p.qmax = q;
  }
  return p;
}

// columns [ja, jb) of block row I whose first cost unit lies in [cs, ce);
// false if there are none
XSYMV_HD bool plan_cost_cols(const Plan& p, long long cs, long long ce, int I, long long* ja,
                             long long* jb) {
  const long long rcs = plan_rowstart(p, I), rce = rcs + plan_rowcost(p, I);
  const long long lo = cs > rcs ? cs : rcs, hi = ce < rce ? ce : rce;
  if (lo >= hi) return false;
  const long long c0 = plan_cols_before(p, I, lo - rcs), c1 = plan_cols_before(p, I, hi - rcs);
  if (c0 >= c1) return false;
  *ja = plan_colbase(p, I) + c0;
  *jb = plan_colbase(p, I) + c1;
  return true;
}

// The warp and row tables of a plan: built once per plan on the device (by
// symv_plan_tables) and kept with the workspace, so that the kernels find
// their work without 64-bit divisions.
//   warp table, one int4 per warp w: x, y = the first and last block row its
//     cost range touches; z = its first column in row x; w = the end of its
//     columns in row y (rows strictly between are wholly its own).  A row
//     whose share holds no column start gets an empty range (z or w at the
//     row's other end).
//   row table, one int2 per block row I: x = the thread block of the owner
//     of its first column (block b's row-partial slot in the row is b - x),
//     y = the number of blocks that own columns of the row (slots 0 .. y-1).
XSYMV_HD void plan_warp_entry(const Plan& p, int w, int* Ia, int* Ib, long long* ja, long long* jb) {
  const long long cs = plan_wstart(p, w), ce = plan_wstart(p, w + 1);
  *Ia = plan_row_of(p, cs);
  *Ib = plan_row_of(p, ce - 1);
  long long a, b;
  *ja = plan_cost_cols(p, cs, ce, *Ia, &a, &b) ? a : plan_colbase(p, *Ia) + plan_rowlen(p, *Ia);
  *jb = plan_cost_cols(p, cs, ce, *Ib, &a, &b) ? b : plan_colbase(p, *Ib);
}

// workspace elements: Wc (nb*n) followed by Wr (nb*qmax*NB)
inline long long plan_wc_elems(const Plan& p) { return (long long)p.nb * p.n; }
inline long long plan_wr_elems(const Plan& p) { return (long long)p.nb * p.qmax * p.NB; }

// ---------------------------------------------------------------------------
// Ordered tickets (the report's own accumulation, "CUDA-xSYMV の実装と評価"
// §2.1, figures "kernel" and "Atomic"): the partial sums of output chunk K
// (outputs K*NB .. K*NB+NB-1) are added into one vector in a fixed order,
// one contributing warp at a time, each handing a ticket to the next.
//
// Contributors of chunk K are the warps that wrote a column partial of one
// of its columns or a row partial of block row K.  In row I they form the
// contiguous warp range "link range t" below:
//   upper: t = I = 0 .. K (column partials of rows I < K; all owners of row
//          K, whose first columns are chunk K's diagonal tile),
//   lower: t = I - K = 0 .. nb-1-K (all owners of row K, whose last columns
//          are the diagonal tile; then column partials of rows I > K).
// The ranges are sorted (their first and last warps never decrease with t),
// so ordering the contributors by warp index orders them by block row, and a
// warp waits only for warps with smaller indices.

// columns [ja, jb) of block row I owned by warp w; false if it owns none
XSYMV_HD bool plan_warp_cols(const Plan& p, int w, int I, long long* ja, long long* jb) {
  return plan_cost_cols(p, plan_wstart(p, w), plan_wstart(p, w + 1), I, ja, jb);
}

// columns of block row I owned by warps w0 .. w1-1 (a contiguous run,
// their union)
XSYMV_HD bool plan_group_cols(const Plan& p, int w0, int w1, int I, long long* ja, long long* jb) {
  return plan_cost_cols(p, plan_wstart(p, w0), plan_wstart(p, w1), I, ja, jb);
}

// number of link ranges of chunk K
XSYMV_HD int plan_links(const Plan& p, int K) { return p.upper ? K + 1 : p.nb - K; }

// first and last warp of link range t of chunk K
XSYMV_HD void plan_link_range(const Plan& p, int K, int t, int* wa, int* wb) {
  const int I = p.upper ? t : K + t;
  if (I == K) {
    *wa = plan_first_owner(p, K);
    *wb = plan_last_owner(p, K);
    return;
  }
  const long long cb = plan_colbase(p, I), rs = plan_rowstart(p, I);
  const long long j0 = (long long)K * p.NB;
  const long long j1 = ((long long)K + 1) * p.NB < p.n ? ((long long)K + 1) * p.NB : (long long)p.n;
  *wa = plan_owner(p, rs + plan_col_cost(p, I, j0 - cb));
  *wb = plan_owner(p, rs + plan_col_cost(p, I, j1 - 1 - cb));
}

// the first contributor of chunk K (it starts the chain without waiting)
XSYMV_HD int plan_chain_first(const Plan& p, int K) {
  int wa, wb;
  plan_link_range(p, K, 0, &wa, &wb);
  return wa;
}

// the contributor of chunk K that follows warp w, or -1 if w is the last
// (binary search for the first link range that ends after w)
XSYMV_HD int plan_chain_next(const Plan& p, int K, int w) {
  int lo = 0, hi = plan_links(p, K);   // answer in [lo, hi]; hi = none
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    int wa, wb;
    plan_link_range(p, K, mid, &wa, &wb);
    if (wb > w) hi = mid; else lo = mid + 1;
  }
  if (lo == plan_links(p, K)) return -1;
  int wa, wb;
  plan_link_range(p, K, lo, &wa, &wb);
  return wa > w + 1 ? wa : w + 1;
}

// The same chains between groups of G consecutive warps (group g = warps
// g*G .. g*G+G-1, e.g. the warps of one thread block): a group contributes
// to chunk K if any of its warps does, and groups follow each other in
// increasing order.  The first group of chunk K:
XSYMV_HD int plan_group_first(const Plan& p, int K, int G) { return plan_chain_first(p, K) / G; }

// the group after group g in chunk K's chain, or -1 if g is the last
XSYMV_HD int plan_group_next(const Plan& p, int K, int g, int G) {
  const long long e = ((long long)g + 1) * G;
  const int last = (int)((e < p.W ? e : (long long)p.W) - 1);   // g's last warp
  const int nx = plan_chain_next(p, K, last);
  return nx < 0 ? -1 : nx / G;
}

// the smallest chunk > after that a warp owning columns [ja, jb) of block
// row I contributes to from that row (its row partial goes to chunk I, its
// column partials to the chunks of its columns); a large value if none
XSYMV_HD int plan_row_next_chunk(const Plan& p, int I, long long ja, long long jb, int after) {
  int best = I > after ? I : 0x7fffffff;
  const int a = (int)(ja / p.NB), b = (int)((jb - 1) / p.NB);
  const int c = after + 1 > a ? after + 1 : a;
  return (c <= b && c < best) ? c : best;
}

// the smallest chunk > after that warps w0 .. w1-1 contribute to, with
// their rows [Ia, Ib] (a large value if there is none)
XSYMV_HD int plan_group_next_chunk(const Plan& p, int w0, int w1, int Ia, int Ib, int after) {
  int best = 0x7fffffff;
  for (int I = Ia; I <= Ib; ++I) {
    long long ja, jb;
    if (!plan_cost_cols(p, plan_wstart(p, w0), plan_wstart(p, w1), I, &ja, &jb)) continue;
    const int c = plan_row_next_chunk(p, I, ja, jb, after);
    if (c < best) best = c;
  }
  return best;
}

// ---------------------------------------------------------------------------
// Partition of the general product y := alpha*A*x + beta*y (all n*n elements
// of A read), the comparison the report makes in §1.  Block row I (rows
// I*NB ..) holds n columns of equal cost; the nb*n (block row, column) units
// are laid out row after row and warp w takes [w*T/W, (w+1)*T/W), T = nb*n.
// Row partials go to slot q = w - (owner of the row's first column) of the
// row, as for SYMV; there are no column partials.
struct GemvPlan {
  int n;
  int NB;
  int nb;
  int W;      // 1 <= W <= nb*n, so every warp owns at least one unit
  int qmax;
};

XSYMV_HD long long gemv_units(const GemvPlan& p) { return (long long)p.nb * p.n; }
XSYMV_HD long long gemv_wstart(const GemvPlan& p, int w) { return (long long)w * gemv_units(p) / p.W; }
XSYMV_HD int gemv_owner(const GemvPlan& p, long long s) {
  return (int)(((s + 1) * p.W - 1) / gemv_units(p));
}
XSYMV_HD int gemv_first_owner(const GemvPlan& p, int I) { return gemv_owner(p, (long long)I * p.n); }
XSYMV_HD int gemv_nq(const GemvPlan& p, int I) {
  return gemv_owner(p, (long long)I * p.n + p.n - 1) - gemv_first_owner(p, I) + 1;
}

inline GemvPlan gemv_plan_make(int n, int NB, long long Wmax) {
  GemvPlan p{};
  p.n = n;
  p.NB = NB;
  p.nb = (n + NB - 1) / NB;
  const long long units = (long long)p.nb * n;
  const long long W = Wmax < units ? Wmax : units;
  p.W = (int)(W < 1 ? 1 : W);
  p.qmax = 1;
  for (int I = 0; I < p.nb; ++I) {
    const int q = gemv_nq(p, I);
    if (q > p.qmax) p.qmax = q;
  }
  return p;
}

}  // namespace xsymv
