// Work partition of one xSYMV call, shared by host dispatch and the kernels.
//
// The stored triangle is cut into block rows of NB rows (NB = the tile edge).
// Block row I owns one "column segment" per matrix column j that meets the
// stored triangle inside its rows:
//   upper ('U'): j = I*NB .. n-1        (diagonal tile first, then the rest)
//   lower ('L'): j = 0 .. min(n, I*NB+NB)-1   (off-diagonal first, diagonal last)
// Segments are numbered row after row (block row 0 first), S in total, and
// each of the W warps takes one contiguous run of ceil or floor S/W of them,
// so every warp streams the same number of column segments from HBM.
//
// Deterministic cross-warp accumulation (the role the report's ordered
// tickets play, "CUDA-xSYMV の実装と評価" §2.1, figure "Atomic"): a warp
// writes
//   * one column partial per segment it processes, to Wc[I*n + j], and
//   * one row partial per block row it touches, to slot q of that row,
//     Wr[(I*qmax + q)*NB + r], q = its index among the warps touching row I;
// a second kernel then sums those slots for every output element in a fixed
// order, so results are bit-identical from run to run.  W <= S guarantees
// that every warp owns at least one segment, so every slot a finaliser reads
// has been written.
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
  long long S;      // total column segments
  int W;            // warps sharing the segments (1 <= W <= S)
  int qmax;         // most warps that touch one block row
};

XSYMV_HD long long plan_rowlen(const Plan& p, int I) {
  if (p.upper) return (long long)p.n - (long long)I * p.NB;
  long long e = (long long)(I + 1) * p.NB;
  return e < p.n ? e : (long long)p.n;
}

// first segment of block row I (0 <= I <= nb-1; and I == nb for upper)
XSYMV_HD long long plan_rowstart(const Plan& p, int I) {
  if (p.upper) return (long long)I * p.n - (long long)p.NB * I * (I - 1) / 2;
  return (long long)p.NB * I * (I + 1) / 2;
}

XSYMV_HD long long plan_total(int n, int NB, int upper) {
  if (n <= 0) return 0;
  Plan p{n, NB, (n + NB - 1) / NB, upper, 0, 1, 1};
  return plan_rowstart(p, p.nb - 1) + plan_rowlen(p, p.nb - 1);
}

// first column (matrix index) of block row I's segments
XSYMV_HD long long plan_colbase(const Plan& p, int I) { return p.upper ? (long long)I * p.NB : 0; }

// first segment of warp w (w = W gives S)
XSYMV_HD long long plan_wstart(const Plan& p, int w) { return (long long)w * p.S / p.W; }

// the warp whose run contains segment s
XSYMV_HD int plan_owner(const Plan& p, long long s) { return (int)(((s + 1) * p.W - 1) / p.S); }

// number of warps whose runs meet block row I
XSYMV_HD int plan_nq(const Plan& p, int I) {
  long long rs = plan_rowstart(p, I);
  return plan_owner(p, rs + plan_rowlen(p, I) - 1) - plan_owner(p, rs) + 1;
}

// block row containing segment s (binary search)
XSYMV_HD int plan_row_of(const Plan& p, long long s) {
  int lo = 0, hi = p.nb - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (plan_rowstart(p, mid) <= s) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Build the plan for n, NB, uplo with at most Wmax warps.
inline Plan plan_make(int n, int NB, int upper, long long Wmax) {
  Plan p{};
  p.n = n;
  p.NB = NB;
  p.nb = (n + NB - 1) / NB;
  p.upper = upper;
  p.S = plan_total(n, NB, upper);
  long long W = Wmax < p.S ? Wmax : p.S;
  p.W = (int)(W < 1 ? 1 : W);
  p.qmax = 1;
  for (int I = 0; I < p.nb; ++I) {
    int q = plan_nq(p, I);
    if (q > p.qmax) p.qmax = q;
  }
  return p;
}

// workspace elements: Wc (nb*n) followed by Wr (nb*qmax*NB)
inline long long plan_wc_elems(const Plan& p) { return (long long)p.nb * p.n; }
inline long long plan_wr_elems(const Plan& p) { return (long long)p.nb * p.qmax * p.NB; }

}  // namespace xsymv
