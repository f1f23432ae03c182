// xSYMV / xHEMV kernels for sm_103a: y := alpha*A*x + beta*y with A symmetric
// (Hermitian for complex types), only the upper or lower triangle stored in
// column-major order with leading dimension lda.
//
// Method ("CUDA-xSYMV の実装と評価", IPSJ 2014-HPC-146, §2.1): every stored
// element A(i,j), i != j, is read from memory once and used twice, for the
// row term A(i,j)*x(j) of y(i) and the column term conj(A(i,j))*x(i) of y(j);
// this halves the memory traffic of GEMV.  The report's kernels are the
// preprocess (y *= beta, v = 0), main (parts one and two) and postprocess
// (y += alpha*v) of figure "kernel", with ordered tickets for the updates of
// v.  Here the same arithmetic is organised for GB300:
//
//   symv_main      Each warp streams an equal share of the triangle's column
//                  segments (see xsymv_plan.h).  A column segment is the
//                  NB-row piece of one matrix column inside one block row:
//                  the 32 lanes cover its NB rows with 16-byte loads
//                  (VR vectors per lane), U columns in flight at a time.
//                  Row terms stay in the lane's registers for the whole block
//                  row (no reduction needed: each lane owns its rows); column
//                  terms are summed across the 32 lanes with a butterfly
//                  reduce-scatter of the U columns and written to the
//                  workspace.  The diagonal tile is handled by the same loop
//                  with a triangle mask: its stored part is read once and
//                  contributes to both sides, which is what the report's
//                  mirrored copy in shared memory (part two) achieves.
//   symv_finalize  One thread per output element sums the workspace slots of
//                  its row in a fixed order and applies y = alpha*s + beta*y
//                  (the report's parts three and the beta scaling).  No atomic
//                  operation touches data, so results are bit-identical from
//                  run to run.
#pragma once

#include "xsymv_plan.h"
#include "xsymv_scalar.cuh"

namespace xsymv {

template <int U> struct Log2;
template <> struct Log2<1> { static constexpr int v = 0; };
template <> struct Log2<2> { static constexpr int v = 1; };
template <> struct Log2<4> { static constexpr int v = 2; };
template <> struct Log2<8> { static constexpr int v = 3; };
template <> struct Log2<16> { static constexpr int v = 4; };
template <> struct Log2<32> { static constexpr int v = 5; };

// Sum v[0..U) over the 32 lanes of the warp.  On return lane l holds the
// total of column u = l >> (5 - log2 U); the additions happen in a fixed
// pattern, independent of timing.
template <class T, int U>
__device__ __forceinline__ T reduce_scatter(T (&v)[U], int lane) {
  constexpr int H = Log2<U>::v;
  int off = 16;
#pragma unroll
  for (int h = 0; h < H; ++h) {
    const int half = U >> (h + 1);
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      T send = up ? v[i] : v[i + half];
      T keep = up ? v[i + half] : v[i];
      v[i] = Ops<T>::add(keep, Ops<T>::shfl_xor(send, off));
    }
    off >>= 1;
  }
#pragma unroll
  for (int o = 16 >> H; o >= 1; o >>= 1) v[0] = Ops<T>::add(v[0], Ops<T>::shfl_xor(v[0], o));
  return v[0];
}

template <class T, int VR, int U>
struct WarpTile {
  static constexpr int VPL = Ops<T>::VPL;
  static constexpr int NB = 32 * VPL * VR;
  static constexpr int H = Log2<U>::v;

  // one block row's state for this lane
  T xi[VR][VPL];
  T racc[VR][VPL];

  __device__ __forceinline__ static long long row_of(long long r0, int v, int lane, int k) {
    return r0 + (long long)(v * 32 + lane) * VPL + k;
  }

  // write the U reduced column sums of one chunk (cnt valid columns)
  __device__ __forceinline__ static void emit_columns(T (&cp)[U], int lane, int cnt, T* wc_row,
                                                      long long j0) {
    T red = reduce_scatter<T, U>(cp, lane);
    const int uo = lane >> (5 - H);
    if ((lane & ((32 >> H) - 1)) == 0 && uo < cnt) wc_row[j0 + uo] = red;
  }

  // Columns [ja, jb) of block row starting at row r0, all NB rows stored
  // (off-diagonal, complete block row).  ALIGNED: 16-byte vector loads.
  template <bool ALIGNED>
  __device__ __forceinline__ void dense_cols(const T* __restrict__ A, long long lda,
                                             const T* __restrict__ x, long long incx, long long r0,
                                             long long ja, long long jb, T* wc_row, int lane) {
    long long j0 = ja;
    for (; j0 + U <= jb; j0 += U) {
      const T xl = (lane < U) ? Ops<T>::load(x + (j0 + lane) * incx) : Ops<T>::zero();
      T a[U][VR][VPL];
      if (ALIGNED) {
        uint4 raw[U][VR];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int v = 0; v < VR; ++v)
            raw[u][v] = ldg_stream16(A + (j0 + u) * lda + row_of(r0, v, lane, 0));
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int v = 0; v < VR; ++v) Unpack<T>::run(raw[u][v], a[u][v]);
      } else {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int v = 0; v < VR; ++v)
#pragma unroll
            for (int k = 0; k < VPL; ++k)
              a[u][v][k] = Ops<T>::load(A + (j0 + u) * lda + row_of(r0, v, lane, k));
      }
      T cp[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const T xj = Ops<T>::shfl(xl, u);
        T c = Ops<T>::zero();
#pragma unroll
        for (int v = 0; v < VR; ++v)
#pragma unroll
          for (int k = 0; k < VPL; ++k) {
            racc[v][k] = Ops<T>::madd(racc[v][k], a[u][v][k], xj);
            c = Ops<T>::maddc(c, a[u][v][k], xi[v][k]);
          }
        cp[u] = c;
      }
      emit_columns(cp, lane, U, wc_row, j0);
    }
    if (j0 < jb) masked_cols<false>(A, lda, x, incx, r0, j0, jb, wc_row, lane, 0, 0);
  }

  // Columns [ja, jb) with per-element masks: rows must be < n and, when
  // DIAG, inside the stored triangle (upper: row <= col; lower: row >= col).
  // On the diagonal only the row term is taken (and for a Hermitian matrix
  // only the real part of the element).  Elements outside the mask are
  // never read.
  template <bool DIAG>
  __device__ __forceinline__ void masked_cols(const T* __restrict__ A, long long lda,
                                              const T* __restrict__ x, long long incx,
                                              long long r0, long long ja, long long jb,
                                              T* wc_row, int lane, long long n, int upper) {
    for (long long j0 = ja; j0 < jb; j0 += U) {
      const int cnt = (int)((jb - j0) < U ? (jb - j0) : U);
      const T xl = (lane < cnt) ? Ops<T>::load(x + (j0 + lane) * incx) : Ops<T>::zero();
      T cp[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long j = j0 + u;
        const T xj = Ops<T>::shfl(xl, u);
        T c = Ops<T>::zero();
#pragma unroll
        for (int v = 0; v < VR; ++v)
#pragma unroll
          for (int k = 0; k < VPL; ++k) {
            const long long r = row_of(r0, v, lane, k);
            bool valid = u < cnt;
            if (DIAG) valid = valid && r < n && (upper ? r <= j : r >= j);
            if (valid) {
              T a = Ops<T>::load(A + j * lda + r);
              if (DIAG && r == j) {
                racc[v][k] = Ops<T>::madd(racc[v][k], Ops<T>::diag(a), xj);
              } else {
                racc[v][k] = Ops<T>::madd(racc[v][k], a, xj);
                c = Ops<T>::maddc(c, a, xi[v][k]);
              }
            }
          }
        cp[u] = c;
      }
      emit_columns(cp, lane, cnt, wc_row, j0);
    }
  }
};

// ----------------------------------------------------------------------------
// main kernel
// ----------------------------------------------------------------------------
template <class T, int VR, int U, int WARPS, bool ALIGNED>
__global__ void __launch_bounds__(WARPS * 32)
symv_main(Plan p, const T* __restrict__ A, long long lda, const T* __restrict__ x, long long incx,
          T* __restrict__ Wc, T* __restrict__ Wr) {
  using Tile = WarpTile<T, VR, U>;
  constexpr int VPL = Tile::VPL;
  constexpr int NB = Tile::NB;
  const int lane = threadIdx.x & 31;
  const int w = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  if (w >= p.W) return;

  long long s = plan_wstart(p, w);
  const long long send = plan_wstart(p, w + 1);
  int I = plan_row_of(p, s);
  const long long n = p.n;
  Tile t;

  while (s < send) {
    const long long rs = plan_rowstart(p, I);
    const long long rl = plan_rowlen(p, I);
    const long long cb = plan_colbase(p, I);
    const long long ja = cb + (s - rs);
    const long long jb = cb + ((send - rs) < rl ? (send - rs) : rl);
    const int q = w - plan_owner(p, rs);
    const long long r0 = (long long)I * NB;

#pragma unroll
    for (int v = 0; v < VR; ++v)
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        const long long r = Tile::row_of(r0, v, lane, k);
        t.xi[v][k] = (r < n) ? Ops<T>::load(x + r * incx) : Ops<T>::zero();
        t.racc[v][k] = Ops<T>::zero();
      }

    T* wc_row = Wc + (long long)I * n;
    const long long dA = r0;
    const long long dB = (r0 + NB < n) ? r0 + NB : n;   // diagonal tile columns [dA, dB)
    const bool complete = (r0 + NB <= n);               // all NB rows exist
    if (p.upper) {
      // diagonal tile first, then the off-diagonal columns (rows all stored)
      const long long a0 = ja > dA ? ja : dA, a1 = jb < dB ? jb : dB;
      if (a0 < a1) t.template masked_cols<true>(A, lda, x, incx, r0, a0, a1, wc_row, lane, n, 1);
      const long long b0 = ja > dB ? ja : dB;
      if (b0 < jb) t.template dense_cols<ALIGNED>(A, lda, x, incx, r0, b0, jb, wc_row, lane);
    } else {
      // off-diagonal columns first, then the diagonal tile
      const long long b1 = jb < dA ? jb : dA;
      if (ja < b1) {
        if (complete)
          t.template dense_cols<ALIGNED>(A, lda, x, incx, r0, ja, b1, wc_row, lane);
        else
          t.template masked_cols<true>(A, lda, x, incx, r0, ja, b1, wc_row, lane, n, 0);
      }
      const long long a0 = ja > dA ? ja : dA;
      if (a0 < jb) t.template masked_cols<true>(A, lda, x, incx, r0, a0, jb, wc_row, lane, n, 0);
    }

    T* wr = Wr + ((long long)I * p.qmax + q) * NB;
#pragma unroll
    for (int v = 0; v < VR; ++v)
#pragma unroll
      for (int k = 0; k < VPL; ++k) wr[(v * 32 + lane) * VPL + k] = t.racc[v][k];

    s = rs + (jb - cb);
    ++I;
  }
}

// ----------------------------------------------------------------------------
// finalize: y := alpha * (fixed-order sum of the workspace slots) + beta * y
// ----------------------------------------------------------------------------
enum FinalMode { kFull = 0, kBetaZero = 1, kAlphaZero = 2, kZero = 3 };

template <class T>
__global__ void __launch_bounds__(256)
symv_finalize(Plan p, const T* __restrict__ Wc, const T* __restrict__ Wr, T alpha, T beta,
              int mode, T* __restrict__ y, long long incy) {
  const long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= p.n) return;
  T* yj = y + j * incy;
  T s = Ops<T>::zero();
  if (mode == kFull || mode == kBetaZero) {
    const int K = (int)(j / p.NB);
    const int jj = (int)(j - (long long)K * p.NB);
    const int I0 = p.upper ? 0 : K;
    const int I1 = p.upper ? K : p.nb - 1;
    const T* wc = Wc + j;
#pragma unroll 8
    for (int I = I0; I <= I1; ++I) s = Ops<T>::add(s, wc[(long long)I * p.n]);
    const long long rs = plan_rowstart(p, K);
    const int q0 = plan_owner(p, rs);
    const int nq = plan_owner(p, rs + plan_rowlen(p, K) - 1) - q0 + 1;
    const T* wr = Wr + (long long)K * p.qmax * p.NB + jj;
    for (int q = 0; q < nq; ++q) s = Ops<T>::add(s, wr[(long long)q * p.NB]);
  }
  T out;
  if (mode == kFull)
    out = Ops<T>::add(Ops<T>::mul(alpha, s), Ops<T>::mul(beta, *yj));
  else if (mode == kBetaZero)
    out = Ops<T>::mul(alpha, s);
  else if (mode == kAlphaZero)
    out = Ops<T>::mul(beta, *yj);
  else
    out = Ops<T>::zero();
  *yj = out;
}

}  // namespace xsymv
