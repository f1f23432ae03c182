/*
 * CPU oracle for xSYMV / xHEMV — TEST INFRASTRUCTURE, not part of the library.
 * See oracle.h for the interface.  Plain, slow, single-threaded C.
 *
 * Source of the method: "CUDA-xSYMV の実装と評価" (Implementation and
 * evaluation of CUDA-xSYMV), IPSJ 2014-HPC-146:
 *   §1, equation (1)      y := alpha*A*x + beta*y, A = A^T, U or L stored;
 *   §2.1, figure "Sequential SYMV kernel algorithm"
 *                         v = 0 and y *= beta; part one walks the strict
 *                         triangle column by column, adding A(i,j)*x(j) into
 *                         v(i) and A(i,j)*x(i) into a column sum t that is
 *                         added as alpha*t to y(j); part two adds the
 *                         diagonal alpha*A(i,i)*x(i); part three adds
 *                         alpha*v.
 *   §2.2                  the same algorithm for complex Hermitian
 *                         (CHEMV, ZHEMV) and double-double (WSYMV) data.
 * The figure prints the upper-triangle loop only; the lower triangle is its
 * mirror (column j walks rows j+1..n-1).  For Hermitian A the element below
 * the diagonal is conj(A(i,j)), so the column sum takes conj(a)*x(i), and
 * the imaginary part of the diagonal is never read.  beta = 0 overwrites y
 * without reading it; alpha = 0 reads neither A nor x (reference-BLAS
 * conventions; the report's interface is the BLAS one, figure "x-symv API").
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>

#if defined(__x86_64__)
typedef __float128 quad_t;
#define ORACLE_QUAD_MANT __FLT128_MANT_DIG__
#elif defined(__aarch64__)
typedef long double quad_t;
#define ORACLE_QUAD_MANT __LDBL_MANT_DIG__
#else
#error "the oracle needs an IEEE binary128 type"
#endif
_Static_assert(ORACLE_QUAD_MANT == 113, "quad_t must be IEEE binary128");

int oracle_quad_mant_dig(void) { return ORACLE_QUAD_MANT; }

/* ---- argument checking and vector indexing (reference-BLAS rules) ---- */

static int is_upper(char uplo) { return uplo == 'U' || uplo == 'u'; }
static int is_lower(char uplo) { return uplo == 'L' || uplo == 'l'; }

static int check_args(char uplo, int n, int lda, int incx, int incy)
{
    if (!is_upper(uplo) && !is_lower(uplo)) return 1;
    if (n < 0) return 2;
    if (lda < (n > 1 ? n : 1)) return 5;
    if (incx == 0) return 7;
    if (incy == 0) return 10;
    return 0;
}

/* offset of logical element 0 of a vector with stride inc */
static long first_index(int n, int inc) { return inc > 0 ? 0 : (long)(1 - n) * inc; }

/* is (i, j) inside the stored triangle (diagonal included)? */
static int stored(int upper, long i, long j) { return upper ? i <= j : i >= j; }

/* first and one-past-last row of the strict stored part of column j */
static void strict_rows(int upper, int n, int j, int *i0, int *i1)
{
    if (upper) { *i0 = 0;     *i1 = j; }
    else       { *i0 = j + 1; *i1 = n; }
}

static void split_quad(quad_t q, double *hi, double *lo)
{
    double h = (double)q;
    *hi = h;
    *lo = (double)(q - (quad_t)h);
}

/* ------------------------------ SSYMV ---------------------------------- */
/* float data, binary64 accumulator (float products are exact in binary64) */

int oracle_ssymv(char uplo, int n, float alpha, const float *A, int lda,
                 const float *x, int incx, float beta, float *y, int incy,
                 double *ref_hi, double *ref_lo)
{
    int info = check_args(uplo, n, lda, incx, incy);
    if (info) return info;
    if (n == 0) return 0;
    const int up = is_upper(uplo);
    const long kx = first_index(n, incx), ky = first_index(n, incy);
#define X(i) ((double)x[kx + (long)(i) * incx])
#define Y(i) y[ky + (long)(i) * incy]
    if (alpha == 0.0f && beta == 1.0f) {          /* quick return: y unchanged */
        for (int i = 0; i < n; i++) {
            if (ref_hi) ref_hi[i] = Y(i);
            if (ref_lo) ref_lo[i] = 0.0;
        }
        return 0;
    }
    double *v = calloc((size_t)n, sizeof(double));
    double *acc = malloc((size_t)n * sizeof(double));
    if (!v || !acc) { free(v); free(acc); return -1; }
    const double al = alpha, be = beta;

    /* v(1:n) = 0; y(1:n) *= beta */
    for (int i = 0; i < n; i++) acc[i] = (beta == 0.0f) ? 0.0 : be * (double)Y(i);

    if (alpha != 0.0f) {
        /* part one: the strict triangle, column by column */
        for (int j = 0; j < n; j++) {
            int i0, i1;
            strict_rows(up, n, j, &i0, &i1);
            double t = 0.0;
            for (int i = i0; i < i1; i++) {
                double a = A[i + (long)j * lda];
                v[i] += a * X(j);
                t += a * X(i);
            }
            acc[j] += al * t;
        }
        /* part two: the diagonal */
        for (int i = 0; i < n; i++) acc[i] += al * ((double)A[i + (long)i * lda] * X(i));
        /* part three */
        for (int i = 0; i < n; i++) acc[i] += al * v[i];
    }

    for (int i = 0; i < n; i++) {
        Y(i) = (float)acc[i];
        if (ref_hi) ref_hi[i] = acc[i];
        if (ref_lo) ref_lo[i] = 0.0;
    }
#undef X
#undef Y
    free(v);
    free(acc);
    return 0;
}

/* ------------------------------ DSYMV ---------------------------------- */
/* double data, binary128 accumulator (double products are exact in it)   */

int oracle_dsymv(char uplo, int n, double alpha, const double *A, int lda,
                 const double *x, int incx, double beta, double *y, int incy,
                 double *ref_hi, double *ref_lo)
{
    int info = check_args(uplo, n, lda, incx, incy);
    if (info) return info;
    if (n == 0) return 0;
    const int up = is_upper(uplo);
    const long kx = first_index(n, incx), ky = first_index(n, incy);
#define X(i) ((quad_t)x[kx + (long)(i) * incx])
#define Y(i) y[ky + (long)(i) * incy]
    if (alpha == 0.0 && beta == 1.0) {            /* quick return: y unchanged */
        for (int i = 0; i < n; i++) {
            if (ref_hi) ref_hi[i] = Y(i);
            if (ref_lo) ref_lo[i] = 0.0;
        }
        return 0;
    }
    quad_t *v = calloc((size_t)n, sizeof(quad_t));
    quad_t *acc = malloc((size_t)n * sizeof(quad_t));
    if (!v || !acc) { free(v); free(acc); return -1; }
    const quad_t al = alpha, be = beta;

    for (int i = 0; i < n; i++) acc[i] = (beta == 0.0) ? 0 : be * (quad_t)Y(i);

    if (alpha != 0.0) {
        for (int j = 0; j < n; j++) {
            int i0, i1;
            strict_rows(up, n, j, &i0, &i1);
            quad_t t = 0;
            for (int i = i0; i < i1; i++) {
                quad_t a = A[i + (long)j * lda];
                v[i] += a * X(j);
                t += a * X(i);
            }
            acc[j] += al * t;
        }
        for (int i = 0; i < n; i++) acc[i] += al * ((quad_t)A[i + (long)i * lda] * X(i));
        for (int i = 0; i < n; i++) acc[i] += al * v[i];
    }

    for (int i = 0; i < n; i++) {
        double hi, lo;
        split_quad(acc[i], &hi, &lo);
        Y(i) = hi;
        if (ref_hi) ref_hi[i] = hi;
        if (ref_lo) ref_lo[i] = lo;
    }
#undef X
#undef Y
    free(v);
    free(acc);
    return 0;
}

/* ------------------------------ CHEMV ---------------------------------- */
/* complex float data, complex binary64 accumulator                         */

typedef struct { double re, im; } cdbl;

static cdbl cd_add(cdbl a, cdbl b) { return (cdbl){a.re + b.re, a.im + b.im}; }
static cdbl cd_mul(cdbl a, cdbl b)
{
    return (cdbl){a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
}
static cdbl cd_conj(cdbl a) { return (cdbl){a.re, -a.im}; }

int oracle_chemv(char uplo, int n, const float *alpha, const float *A, int lda,
                 const float *x, int incx, const float *beta, float *y, int incy,
                 double *ref_hi, double *ref_lo)
{
    int info = check_args(uplo, n, lda, incx, incy);
    if (info) return info;
    if (n == 0) return 0;
    const int up = is_upper(uplo);
    const long kx = first_index(n, incx), ky = first_index(n, incy);
#define XE(i) ((cdbl){x[2 * (kx + (long)(i) * incx)], x[2 * (kx + (long)(i) * incx) + 1]})
#define AE(i, j) ((cdbl){A[2 * ((long)(i) + (long)(j) * lda)], A[2 * ((long)(i) + (long)(j) * lda) + 1]})
#define YRE(i) y[2 * (ky + (long)(i) * incy)]
#define YIM(i) y[2 * (ky + (long)(i) * incy) + 1]
    if (alpha[0] == 0 && alpha[1] == 0 && beta[0] == 1 && beta[1] == 0) {
        for (int i = 0; i < n; i++) {            /* quick return: y unchanged */
            if (ref_hi) { ref_hi[2 * i] = YRE(i); ref_hi[2 * i + 1] = YIM(i); }
            if (ref_lo) { ref_lo[2 * i] = 0.0; ref_lo[2 * i + 1] = 0.0; }
        }
        return 0;
    }
    cdbl *v = calloc((size_t)n, sizeof(cdbl));
    cdbl *acc = malloc((size_t)n * sizeof(cdbl));
    if (!v || !acc) { free(v); free(acc); return -1; }
    const cdbl al = {alpha[0], alpha[1]}, be = {beta[0], beta[1]};
    const int alpha_zero = alpha[0] == 0.0f && alpha[1] == 0.0f;
    const int beta_zero = beta[0] == 0.0f && beta[1] == 0.0f;

    for (int i = 0; i < n; i++)
        acc[i] = beta_zero ? (cdbl){0.0, 0.0} : cd_mul(be, (cdbl){YRE(i), YIM(i)});

    if (!alpha_zero) {
        for (int j = 0; j < n; j++) {
            int i0, i1;
            strict_rows(up, n, j, &i0, &i1);
            cdbl t = {0.0, 0.0};
            for (int i = i0; i < i1; i++) {
                cdbl a = AE(i, j);
                v[i] = cd_add(v[i], cd_mul(a, XE(j)));
                t = cd_add(t, cd_mul(cd_conj(a), XE(i)));
            }
            acc[j] = cd_add(acc[j], cd_mul(al, t));
        }
        for (int i = 0; i < n; i++) {
            cdbl d = {AE(i, i).re, 0.0};          /* imaginary part not read */
            acc[i] = cd_add(acc[i], cd_mul(al, cd_mul(d, XE(i))));
        }
        for (int i = 0; i < n; i++) acc[i] = cd_add(acc[i], cd_mul(al, v[i]));
    }

    for (int i = 0; i < n; i++) {
        YRE(i) = (float)acc[i].re;
        YIM(i) = (float)acc[i].im;
        if (ref_hi) { ref_hi[2 * i] = acc[i].re; ref_hi[2 * i + 1] = acc[i].im; }
        if (ref_lo) { ref_lo[2 * i] = 0.0; ref_lo[2 * i + 1] = 0.0; }
    }
#undef XE
#undef AE
#undef YRE
#undef YIM
    free(v);
    free(acc);
    return 0;
}

/* ------------------------------ ZHEMV ---------------------------------- */
/* complex double data, complex binary128 accumulator                       */

typedef struct { quad_t re, im; } cquad;

static cquad cq_add(cquad a, cquad b) { return (cquad){a.re + b.re, a.im + b.im}; }
static cquad cq_mul(cquad a, cquad b)
{
    return (cquad){a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
}
static cquad cq_conj(cquad a) { return (cquad){a.re, -a.im}; }

int oracle_zhemv(char uplo, int n, const double *alpha, const double *A, int lda,
                 const double *x, int incx, const double *beta, double *y, int incy,
                 double *ref_hi, double *ref_lo)
{
    int info = check_args(uplo, n, lda, incx, incy);
    if (info) return info;
    if (n == 0) return 0;
    const int up = is_upper(uplo);
    const long kx = first_index(n, incx), ky = first_index(n, incy);
#define XE(i) ((cquad){x[2 * (kx + (long)(i) * incx)], x[2 * (kx + (long)(i) * incx) + 1]})
#define AE(i, j) ((cquad){A[2 * ((long)(i) + (long)(j) * lda)], A[2 * ((long)(i) + (long)(j) * lda) + 1]})
#define YRE(i) y[2 * (ky + (long)(i) * incy)]
#define YIM(i) y[2 * (ky + (long)(i) * incy) + 1]
    if (alpha[0] == 0 && alpha[1] == 0 && beta[0] == 1 && beta[1] == 0) {
        for (int i = 0; i < n; i++) {            /* quick return: y unchanged */
            if (ref_hi) { ref_hi[2 * i] = YRE(i); ref_hi[2 * i + 1] = YIM(i); }
            if (ref_lo) { ref_lo[2 * i] = 0.0; ref_lo[2 * i + 1] = 0.0; }
        }
        return 0;
    }
    cquad *v = calloc((size_t)n, sizeof(cquad));
    cquad *acc = malloc((size_t)n * sizeof(cquad));
    if (!v || !acc) { free(v); free(acc); return -1; }
    const cquad al = {alpha[0], alpha[1]}, be = {beta[0], beta[1]};
    const int alpha_zero = alpha[0] == 0.0 && alpha[1] == 0.0;
    const int beta_zero = beta[0] == 0.0 && beta[1] == 0.0;

    for (int i = 0; i < n; i++)
        acc[i] = beta_zero ? (cquad){0, 0} : cq_mul(be, (cquad){YRE(i), YIM(i)});

    if (!alpha_zero) {
        for (int j = 0; j < n; j++) {
            int i0, i1;
            strict_rows(up, n, j, &i0, &i1);
            cquad t = {0, 0};
            for (int i = i0; i < i1; i++) {
                cquad a = AE(i, j);
                v[i] = cq_add(v[i], cq_mul(a, XE(j)));
                t = cq_add(t, cq_mul(cq_conj(a), XE(i)));
            }
            acc[j] = cq_add(acc[j], cq_mul(al, t));
        }
        for (int i = 0; i < n; i++) {
            cquad d = {AE(i, i).re, 0};           /* imaginary part not read */
            acc[i] = cq_add(acc[i], cq_mul(al, cq_mul(d, XE(i))));
        }
        for (int i = 0; i < n; i++) acc[i] = cq_add(acc[i], cq_mul(al, v[i]));
    }

    for (int i = 0; i < n; i++) {
        double rh, rl, ih, il;
        split_quad(acc[i].re, &rh, &rl);
        split_quad(acc[i].im, &ih, &il);
        YRE(i) = rh;
        YIM(i) = ih;
        if (ref_hi) { ref_hi[2 * i] = rh; ref_hi[2 * i + 1] = ih; }
        if (ref_lo) { ref_lo[2 * i] = rl; ref_lo[2 * i + 1] = il; }
    }
#undef XE
#undef AE
#undef YRE
#undef YIM
    free(v);
    free(acc);
    return 0;
}

/* ------------------------------ WSYMV ---------------------------------- */
/* double-double data (hi + lo), binary128 accumulator                      */

int oracle_wsymv(char uplo, int n, const double *alpha, const double *A, int lda,
                 const double *x, int incx, const double *beta, double *y, int incy,
                 double *ref_hi, double *ref_lo)
{
    int info = check_args(uplo, n, lda, incx, incy);
    if (info) return info;
    if (n == 0) return 0;
    const int up = is_upper(uplo);
    const long kx = first_index(n, incx), ky = first_index(n, incy);
#define DD(p, k) ((quad_t)(p)[2 * (k)] + (quad_t)(p)[2 * (k) + 1])
#define X(i) DD(x, kx + (long)(i) * incx)
#define AE(i, j) DD(A, (long)(i) + (long)(j) * lda)
#define YIDX(i) (ky + (long)(i) * incy)
    if (DD(alpha, 0) == 0 && DD(beta, 0) == 1) {  /* quick return: y unchanged */
        for (int i = 0; i < n; i++) {
            if (ref_hi) ref_hi[i] = y[2 * YIDX(i)];
            if (ref_lo) ref_lo[i] = y[2 * YIDX(i) + 1];
        }
        return 0;
    }
    quad_t *v = calloc((size_t)n, sizeof(quad_t));
    quad_t *acc = malloc((size_t)n * sizeof(quad_t));
    if (!v || !acc) { free(v); free(acc); return -1; }
    const quad_t al = DD(alpha, 0), be = DD(beta, 0);

    for (int i = 0; i < n; i++) acc[i] = (be == 0) ? 0 : be * DD(y, YIDX(i));

    if (al != 0) {
        for (int j = 0; j < n; j++) {
            int i0, i1;
            strict_rows(up, n, j, &i0, &i1);
            quad_t t = 0;
            for (int i = i0; i < i1; i++) {
                quad_t a = AE(i, j);
                v[i] += a * X(j);
                t += a * X(i);
            }
            acc[j] += al * t;
        }
        for (int i = 0; i < n; i++) acc[i] += al * (AE(i, i) * X(i));
        for (int i = 0; i < n; i++) acc[i] += al * v[i];
    }

    for (int i = 0; i < n; i++) {
        double hi, lo;
        split_quad(acc[i], &hi, &lo);
        y[2 * YIDX(i)] = hi;
        y[2 * YIDX(i) + 1] = lo;
        if (ref_hi) ref_hi[i] = hi;
        if (ref_lo) ref_lo[i] = lo;
    }
#undef DD
#undef X
#undef AE
#undef YIDX
    free(v);
    free(acc);
    return 0;
}

/* ---------------- rows of the mirrored matrix, by definition ------------ */

typedef struct { quad_t re, im; } qval;

/* element k of an array of the given kind, widened to a binary128 pair */
static qval load_val(char kind, const void *p, long k)
{
    qval r = {0, 0};
    switch (kind) {
    case 's': r.re = ((const float *)p)[k]; break;
    case 'd': r.re = ((const double *)p)[k]; break;
    case 'c': r.re = ((const float *)p)[2 * k]; r.im = ((const float *)p)[2 * k + 1]; break;
    case 'z': r.re = ((const double *)p)[2 * k]; r.im = ((const double *)p)[2 * k + 1]; break;
    case 'w': r.re = (quad_t)((const double *)p)[2 * k] + (quad_t)((const double *)p)[2 * k + 1]; break;
    }
    return r;
}

static double modulus(qval a) { return hypot((double)a.re, (double)a.im); }

/* A(i,j) of the full matrix: the stored element, or its mirror image
 * (conjugated for a Hermitian matrix, whose diagonal is real) */
static qval full_elem(char kind, int up, const void *A, int lda, long i, long j)
{
    const int herm = (kind == 'c' || kind == 'z');
    qval a;
    if (stored(up, i, j)) {
        a = load_val(kind, A, i + j * (long)lda);
    } else {
        a = load_val(kind, A, j + i * (long)lda);
        if (herm) a.im = -a.im;
    }
    if (herm && i == j) a.im = 0;
    return a;
}

int oracle_rows(char kind, char uplo, int n, const double *alpha, const void *A,
                int lda, const void *x, int incx, const double *beta,
                const void *y0, int incy, int nrows, const long long *rows,
                double *ref_hi, double *ref_lo, double *denom)
{
    int info = check_args(uplo, n, lda, incx, incy);
    if (info) return info;
    if (kind != 's' && kind != 'd' && kind != 'c' && kind != 'z' && kind != 'w') return -2;
    const int up = is_upper(uplo);
    const int cplx = (kind == 'c' || kind == 'z');
    const long kx = first_index(n, incx), ky = first_index(n, incy);
    qval al = {alpha[0], 0}, be = {beta[0], 0};
    if (cplx) { al.im = alpha[1]; be.im = beta[1]; }
    if (kind == 'w') { al.re += (quad_t)alpha[1]; be.re += (quad_t)beta[1]; }
    const int alpha_zero = (al.re == 0 && al.im == 0);
    const int beta_zero = (be.re == 0 && be.im == 0);

    for (int r = 0; r < nrows; r++) {
        const long i = rows[r];
        if (i < 0 || i >= n) return -3;
        /* s = sum_j A(i,j) x_j and d = sum_j |A(i,j)| |x_j| */
        qval s = {0, 0};
        double d = 0.0;
        if (!alpha_zero) {
            for (long j = 0; j < n; j++) {
                qval a = full_elem(kind, up, A, lda, i, j);
                qval xj = load_val(kind, x, kx + j * incx);
                s.re += a.re * xj.re - a.im * xj.im;
                s.im += a.re * xj.im + a.im * xj.re;
                d += modulus(a) * modulus(xj);
            }
        }
        /* alpha*s + beta*y_i */
        qval out = {al.re * s.re - al.im * s.im, al.re * s.im + al.im * s.re};
        double dy = 0.0;
        if (!beta_zero) {
            qval yi = load_val(kind, y0, ky + i * incy);
            out.re += be.re * yi.re - be.im * yi.im;
            out.im += be.re * yi.im + be.im * yi.re;
            dy = modulus(be) * modulus(yi);
        }
        const int w = cplx ? 2 : 1;
        double h, l;
        split_quad(out.re, &h, &l);
        if (ref_hi) ref_hi[w * r] = h;
        if (ref_lo) ref_lo[w * r] = l;
        if (cplx) {
            split_quad(out.im, &h, &l);
            if (ref_hi) ref_hi[w * r + 1] = h;
            if (ref_lo) ref_lo[w * r + 1] = l;
        }
        if (denom) denom[r] = modulus(al) * d + dy;
    }
    return 0;
}

/* ------------------ general matrix-vector product (GEMV) ---------------- */
/* The report measures SYMV against the general product y := alpha*A*x +
 * beta*y, which reads all n*n elements of A (§1: GEMV needs twice the
 * memory traffic of SYMV).  This is that product by its definition, for
 * selected rows, in binary128: y_i = beta*y_i + alpha*sum_j A(i,j)*x_j. */

int oracle_gemv_rows(char kind, int n, const double *alpha, const void *A, int lda,
                     const void *x, int incx, const double *beta, const void *y0,
                     int incy, int nrows, const long long *rows, double *ref_hi,
                     double *ref_lo, double *denom)
{
    if (n < 0) return 1;
    if (lda < (n > 1 ? n : 1)) return 4;
    if (incx == 0) return 6;
    if (incy == 0) return 9;
    if (kind != 's' && kind != 'd') return -2;
    const long kx = first_index(n, incx), ky = first_index(n, incy);
    const quad_t al = alpha[0], be = beta[0];

    for (int r = 0; r < nrows; r++) {
        const long i = rows[r];
        if (i < 0 || i >= n) return -3;
        quad_t s = 0;
        double d = 0.0;
        if (al != 0) {
            for (long j = 0; j < n; j++) {
                const quad_t a = load_val(kind, A, i + j * (long)lda).re;
                const quad_t xj = load_val(kind, x, kx + j * incx).re;
                s += a * xj;
                d += fabs((double)a) * fabs((double)xj);
            }
        }
        quad_t out = al * s;
        double dy = 0.0;
        if (be != 0) {
            const quad_t yi = load_val(kind, y0, ky + i * incy).re;
            out += be * yi;
            dy = fabs((double)be) * fabs((double)yi);
        }
        double h, l;
        split_quad(out, &h, &l);
        if (ref_hi) ref_hi[r] = h;
        if (ref_lo) ref_lo[r] = l;
        if (denom) denom[r] = fabs((double)al) * d + dy;
    }
    return 0;
}
