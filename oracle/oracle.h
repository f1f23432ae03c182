/*
 * CPU oracle for xSYMV / xHEMV — TEST INFRASTRUCTURE, not part of the library.
 *
 * Computes y := alpha*A*x + beta*y for a symmetric (SYMV) or Hermitian (HEMV)
 * n-by-n matrix A of which only the upper ('U') or lower ('L') triangle is
 * stored, column-major with leading dimension lda, as in equation (1) of
 * "CUDA-xSYMV の実装と評価" (Implementation and evaluation of CUDA-xSYMV,
 * Imamura, Mukunoki, Yamada, Machida, IPSJ SIG Technical Report
 * 2014-HPC-146), §1.
 *
 * Only the test suite, the package's smoke check and the benchmark's CPU
 * baseline may load this code.  It shares nothing with the CUDA library:
 * no header, helper, table or constant.
 *
 * Two independent codings live here:
 *   oracle_<t>symv / oracle_<t>hemv  — the report's sequential three-part
 *       algorithm (§2.1, figure "Sequential SYMV kernel algorithm"), with a
 *       higher-precision accumulator: binary64 for the float types (s, c),
 *       IEEE binary128 for the double types (d, z) and double-double (w).
 *   oracle_rows — the definition y_i = beta*y_i + alpha*sum_j A(i,j)*x_j on
 *       the explicitly mirrored matrix, for selected rows, in binary128,
 *       together with the error normaliser |alpha|*(|A||x|)_i + |beta|*|y_i|.
 * and, for the general product the report compares SYMV with (§1),
 *   oracle_gemv_rows — y_i = beta*y_i + alpha*sum_j A(i,j)*x_j over all n*n
 *       elements of an unsymmetric A, for selected rows, in binary128.
 *
 * Storage conventions (all host memory, owned by the caller):
 *   s: float      d: double
 *   c: float pairs (re, im)      z: double pairs (re, im)
 *   w: double pairs (hi, lo) read as the unevaluated sum hi + lo
 *   Element A(i,j) (0-based) is at A[i + j*lda] (times 2 for pair types).
 *   Vector element i is at x[kx + i*incx] with kx = 0 for incx > 0 and
 *   kx = (1-n)*incx for incx < 0 (reference-BLAS convention).
 *
 * Return value: 0 on success, else the BLAS argument position of the first
 * bad argument (1 uplo, 2 n, 5 lda, 7 incx, 10 incy); nothing is written on
 * error.
 *
 * ref_hi / ref_lo (may be NULL): the unrounded result as a pair of doubles
 * whose sum is the accumulator value (for complex types re, im interleaved).
 * y itself is overwritten with the result rounded once to its own type
 * (w: hi = round(q), lo = round(q - hi)).
 */
#ifndef XSYMV_ORACLE_H
#define XSYMV_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

int oracle_ssymv(char uplo, int n, float alpha, const float *A, int lda,
                 const float *x, int incx, float beta, float *y, int incy,
                 double *ref_hi, double *ref_lo);
int oracle_dsymv(char uplo, int n, double alpha, const double *A, int lda,
                 const double *x, int incx, double beta, double *y, int incy,
                 double *ref_hi, double *ref_lo);
int oracle_chemv(char uplo, int n, const float *alpha, const float *A, int lda,
                 const float *x, int incx, const float *beta, float *y, int incy,
                 double *ref_hi, double *ref_lo);
int oracle_zhemv(char uplo, int n, const double *alpha, const double *A, int lda,
                 const double *x, int incx, const double *beta, double *y, int incy,
                 double *ref_hi, double *ref_lo);
int oracle_wsymv(char uplo, int n, const double *alpha, const double *A, int lda,
                 const double *x, int incx, const double *beta, double *y, int incy,
                 double *ref_hi, double *ref_lo);

/* kind: 's', 'd', 'c', 'z' or 'w'.  alpha/beta point at 1 (s, d) or 2
 * (c, z: re, im; w: hi, lo) doubles; for 's' and 'c' they must already be
 * the float values widened.  y0 is the input y.  For each of the nrows row
 * indices in rows[] writes the reference value of y_i (ref_hi + ref_lo,
 * complex interleaved) and, if denom is not NULL, the normaliser
 * |alpha| * sum_j |A(i,j)| |x_j| + |beta| |y_i| (one double per row). */
int oracle_rows(char kind, char uplo, int n, const double *alpha, const void *A,
                int lda, const void *x, int incx, const double *beta,
                const void *y0, int incy, int nrows, const long long *rows,
                double *ref_hi, double *ref_lo, double *denom);

/* The general (unsymmetric) product y := alpha*A*x + beta*y that the report
 * compares SYMV with (§1), by its definition, for the nrows row indices in
 * rows[]: all n*n elements of A are read.  kind 's' or 'd' only; alpha and
 * beta point at one double each (for 's' the float values widened).  Writes
 * ref_hi + ref_lo (binary128 result as a double pair) and, if denom is not
 * NULL, |alpha| * sum_j |A(i,j)| |x_j| + |beta| |y_i|.  Returns 0, or the
 * argument position of the first bad argument of the library's xgemv_<t>
 * (1 n, 4 lda, 6 incx, 9 incy); -2 for another kind, -3 for a row out of
 * range. */
int oracle_gemv_rows(char kind, int n, const double *alpha, const void *A, int lda,
                     const void *x, int incx, const double *beta, const void *y0,
                     int incy, int nrows, const long long *rows, double *ref_hi,
                     double *ref_lo, double *denom);

/* Mantissa digits of the binary128 type the oracle accumulates in (113). */
int oracle_quad_mant_dig(void);

#ifdef __cplusplus
}
#endif
#endif
