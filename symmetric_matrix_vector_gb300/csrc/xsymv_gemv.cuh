// The general matrix-vector product y := alpha*A*x + beta*y (A n-by-n,
// column-major, all n*n elements read), built from the SYMV kernels' warp
// loader so that the two can be compared on the same hardware.
//
// "CUDA-xSYMV の実装と評価" (IPSJ 2014-HPC-146) motivates SYMV by this
// comparison (§1 and the abstract): SYMV needs half the memory traffic of
// GEMV, so a bandwidth-bound SYMV should run at about twice GEMV's speed.
// gemv_main streams every column of every block row exactly as symv_main
// streams the off-diagonal columns (same tile edge NB, U columns per step,
// same 16-byte loads), but keeps only the row terms; there is no diagonal
// tile and no column partial.  gemv_finalize sums the row-partial slots of
// each output element in a fixed order, so results are bit-identical from
// run to run.
#pragma once

#include "xsymv_kernels.cuh"

namespace xsymv {

template <class T, int VR, int U, int WARPS, bool ALIGNED, int MINB>
__global__ void __launch_bounds__(WARPS * 32, MINB)
gemv_main(GemvPlan p, const T* __restrict__ A, long long lda, const T* __restrict__ x, int incx,
          T* __restrict__ Wr) {
  using Tile = WarpTile<T, VR, U>;
  constexpr int VPL = Tile::VPL;
  constexpr int NB = Tile::NB;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int w = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  if (w >= p.W) return;

  const long long n = p.n;
  const long long se = gemv_wstart(p, w + 1);
  long long s = gemv_wstart(p, w);
  Tile t;
  while (s < se) {
    const int I = (int)(s / n);
    const long long ja = s - (long long)I * n;
    const long long row_end = (long long)(I + 1) * n;
    const long long jb = (se < row_end ? se : row_end) - (long long)I * n;
    const long long r0 = (long long)I * NB;
#pragma unroll
    for (int v = 0; v < VR; ++v)
#pragma unroll
      for (int k = 0; k < VPL; ++k) t.racc[v][k] = Ops<T>::zero();
    if (r0 + NB > n)
      t.masked_rows(A, lda, x, incx, r0, ja, jb, lane, (int)(n - r0));
    else
      t.template dense_rows<ALIGNED>(A, lda, x, incx, r0, ja, jb, lane);
    const int q = w - gemv_first_owner(p, I);
    T* wr = Wr + ((long long)I * p.qmax + q) * NB;
#pragma unroll
    for (int v = 0; v < VR; ++v)
#pragma unroll
      for (int k = 0; k < VPL; ++k) wr[Tile::lane_row(v, lane, k)] = t.racc[v][k];
    s = row_end;
  }
}

// Block (kFinParts x kFinCols threads) handles 32 consecutive outputs of one
// block row K; thread (part, c) adds the slots q = part, part + kFinParts,
// ... in increasing order, and the kFinParts sums are added in part order.
template <class T>
__global__ void __launch_bounds__(kFinParts * kFinCols)
gemv_finalize(GemvPlan p, const T* __restrict__ Wr, T alpha, T beta, int mode,
              T* __restrict__ y, long long incy) {
  __shared__ T part[kFinParts][kFinCols];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int c = threadIdx.x % kFinCols;
  const int pp = threadIdx.x / kFinCols;
  const long long j = (long long)blockIdx.x * kFinCols + c;
  const bool live = j < p.n;
  T* yj = y + j * incy;
  const T y_old = (live && pp == 0 && mode == kFull) ? *yj : Ops<T>::zero();
  T s = Ops<T>::zero();
  if (live) {
    const int K = (int)(j / p.NB);
    const int nq = gemv_nq(p, K);
    const T* wr = Wr + (long long)K * p.qmax * p.NB + (j - (long long)K * p.NB);
    for (int q = pp; q < nq; q += 8 * kFinParts) {   // loads 8 at a time, same order
      T v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = (q + k * kFinParts < nq) ? wr[(long long)(q + k * kFinParts) * p.NB] : Ops<T>::zero();
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (q + k * kFinParts < nq) s = Ops<T>::add(s, v[k]);
    }
  }
  part[pp][c] = s;
  __syncthreads();
  if (pp != 0 || !live) return;
  s = part[0][c];
#pragma unroll
  for (int k = 1; k < kFinParts; ++k) s = Ops<T>::add(s, part[k][c]);
  *yj = mode == kFull ? Ops<T>::add(Ops<T>::mul(alpha, s), Ops<T>::mul(beta, y_old))
                      : Ops<T>::mul(alpha, s);
}

}  // namespace xsymv
