/*
 * xsymv — symmetric / Hermitian matrix-vector product on NVIDIA GB300 (sm_103a)
 *
 *     y := alpha * A * x + beta * y
 *
 * with A an n-by-n symmetric (xSYMV) or Hermitian (xHEMV) matrix of which only
 * the upper (uplo = 'U') or lower (uplo = 'L') triangle is stored and read.
 * This is equation (1) of "CUDA-xSYMV の実装と評価" (Implementation and
 * evaluation of CUDA-xSYMV; Imamura, Mukunoki, Yamada, Machida, IPSJ SIG
 * Technical Report 2014-HPC-146), §1.  Its figure "x-symv API" (§2.2) gives
 * the five entry points and their BLAS-style argument list, reproduced here
 * with an int status instead of void.  Every stored element leaves HBM once
 * and serves both A(i,j)*x(j) and A(j,i)*x(i) (§2.1), half the traffic of
 * GEMV; cross-block partial sums are combined in a fixed order, so results
 * are bit-identical from run to run (the report's abstract and §2.1,
 * figure "Atomic").
 *
 * Arguments (all entry points; Fortran-BLAS semantics, 0-based in memory):
 *   uplo   'U'/'u': upper triangle stored; 'L'/'l': lower triangle stored.
 *   n      order of A, n >= 0.
 *   alpha  scalar, passed by value.
 *   A      DEVICE pointer to the matrix, column-major: A(i,j) at A[i + j*lda].
 *          Only the uplo triangle (diagonal included) is used; for Hermitian
 *          A the imaginary parts of the diagonal are not used either.  On a
 *          16-byte aligned matrix the diagonal tiles are loaded as 16-byte
 *          vectors, which may also fetch up to 3 (float) or 1 (double,
 *          complex float) elements of the other triangle next to the
 *          diagonal; those values are never used (NaN there is harmless).
 *          Nothing outside rows and columns 0 .. n-1 is read.
 *   lda    leading dimension, lda >= max(1, n).
 *   x      DEVICE pointer; element i at x[kx + i*incx], kx = 0 if incx > 0,
 *          else (1-n)*incx (negative strides run backwards, as in BLAS).
 *   incx   stride of x, non-zero.
 *   beta   scalar.  beta == 0: y is written without being read.
 *   y      DEVICE pointer, same addressing as x with incy.  Only the n
 *          elements y(0..n-1) are written.
 *   incy   stride of y, non-zero.
 *   alpha == 0 means A and x are not read; alpha == 0 and beta == 1 returns
 *   at once without touching anything.
 *
 * Layout of the element types: xsymv_c32 / xsymv_c64 are (re, im) pairs,
 * layout-compatible with cuFloatComplex / cuDoubleComplex (float2 / double2);
 * xsymv_dd is a double-double (hi, lo), the value hi + lo (the report's
 * cuddreal, a double2).
 *
 * Ownership: the caller owns A, x and y (device memory, not freed or kept).
 * The library owns a workspace per (device, stream), allocated with
 * cudaMalloc on first use and grown on demand; it lives until the process
 * exits.  It holds two sets of partial sums (consecutive calls use
 * different ones), so that a call whose A and x do not overlap the previous
 * call's y can start streaming while that call's last kernel still runs.  The ordered-ticket variants ("_tk", below) also keep a small
 * ticket buffer per (device, stream), zeroed when it is allocated.  Work is
 * enqueued on the stream set by xsymv_set_stream (default: the legacy
 * default stream) and runs asynchronously: when a call returns XSYMV_OK the
 * result is ready once that stream has reached it.  Two calls on the same
 * stream are ordered; calls on different streams use different workspaces.
 * Issue the calls that share a stream from one host thread at a time: a call
 * enqueues two or three kernels that share the stream's workspace, and two
 * threads interleaving their launches on one stream would mix them.
 * The first call of a new problem shape (kind, uplo, n, variant) on a stream
 * also enqueues a small kernel that tabulates the work partition; later
 * calls of that shape on that stream reuse the table.
 *
 * Status (return value):
 *   0                 success.
 *   1, 2, 5, 7, 10    the argument at that position is invalid (BLAS xerbla
 *                     convention: 1 uplo, 2 n, 5 lda, 7 incx, 10 incy).
 *                     Arguments are checked before anything is enqueued;
 *                     nothing is read or written.
 *   negative          XSYMV_ERR_* below; a CUDA error is recorded and can be
 *                     read with xsymv_last_cuda_error().
 */
#ifndef XSYMV_H
#define XSYMV_H

#ifdef __cplusplus
extern "C" {
#endif

#define XSYMV_API __attribute__((visibility("default")))

typedef struct { float re, im; } xsymv_c32;
typedef struct { double re, im; } xsymv_c64;
typedef struct { double hi, lo; } xsymv_dd;

#define XSYMV_OK 0
#define XSYMV_ERR_CUDA (-1)       /* a CUDA call or kernel launch failed        */
#define XSYMV_ERR_ALLOC (-2)      /* the workspace could not be allocated       */
#define XSYMV_ERR_DEVICE (-3)     /* no usable device, or not compute cap. 10.3 */
#define XSYMV_ERR_VALUE (-4)      /* invalid argument to a non-BLAS entry point */
#define XSYMV_ERR_TOO_LARGE (-5)  /* problem exceeds xsymv_s_noalloc's scratch  */
#define XSYMV_ERR_TIMEOUT (-6)    /* a kernel gave up waiting; y was set to NaN */

/* SSYMV: float data, float arithmetic. */
XSYMV_API int xsymv_s(char uplo, int n, float alpha, const float *A, int lda,
                      const float *x, int incx, float beta, float *y, int incy);

/* DSYMV: double data, double arithmetic. */
XSYMV_API int xsymv_d(char uplo, int n, double alpha, const double *A, int lda,
                      const double *x, int incx, double beta, double *y, int incy);

/* CHEMV: single-complex Hermitian, A(j,i) = conj(A(i,j)). */
XSYMV_API int xhemv_c(char uplo, int n, xsymv_c32 alpha, const xsymv_c32 *A, int lda,
                      const xsymv_c32 *x, int incx, xsymv_c32 beta, xsymv_c32 *y, int incy);

/* ZHEMV: double-complex Hermitian. */
XSYMV_API int xhemv_z(char uplo, int n, xsymv_c64 alpha, const xsymv_c64 *A, int lda,
                      const xsymv_c64 *x, int incx, xsymv_c64 beta, xsymv_c64 *y, int incy);

/* WSYMV: double-double data and arithmetic (TwoSum / TwoProd-FMA, after
 * Hida, Li and Bailey, the report's reference [14] in §2.2).  Input pairs
 * are renormalised as they are read; results are renormalised pairs. */
XSYMV_API int xsymv_w(char uplo, int n, xsymv_dd alpha, const xsymv_dd *A, int lda,
                      const xsymv_dd *x, int incx, xsymv_dd beta, xsymv_dd *y, int incy);

/* ---- allocation-free SSYMV ----------------------------------------------
 * The report has no counterpart to this entry point.  It is xsymv_s for
 * callers that cannot let a library allocate device memory during a call:
 * a plug-in whose host application owns all device memory and forbids
 * allocating inside the plug-in, or latency-critical code where cudaMalloc /
 * cudaFree would block or synchronise the device.  Same arguments, results
 * and status codes as xsymv_s (xsymv_sync_status reports its timeouts too); it
 * never allocates.  Its workspace is one fixed 16 MiB device array in the
 * library, held on every GPU that loads the library until the process exits;
 * a problem whose workspace does not fit (roughly n > 31000 with the tuned
 * kernels) returns XSYMV_ERR_TOO_LARGE with nothing enqueued and y untouched.
 * The first call with alpha != 0 on a device looks up the array's address
 * on that device; make that call before any stream capture.  It also clears
 * the array's 256-byte status header, the only part that must start at zero.
 * All calls share the array and it keeps the last call's contents (the
 * plan's tables among them): calls that overlap on the GPU, on different
 * streams or from different threads, race on it and corrupt each other's
 * results.  Each call must start on the GPU only after everything the
 * previous call enqueued has finished (calls on one stream are; across
 * streams, wait on an event recorded after the previous call). */
XSYMV_API int xsymv_s_noalloc(char uplo, int n, float alpha, const float *A, int lda,
                              const float *x, int incx, float beta, float *y, int incy);

/* ---- the product split across GPUs by block columns -------------------
 * The report cites Level-2 BLAS on multi-GPU systems (its reference [7],
 * KBLAS, in §1) but describes no split of its own; the plainest reading,
 * taken here: the stored triangle is split by block columns, each GPU holds
 * a panel of consecutive columns, streams it once and produces a
 * full-length partial vector (the row terms of its elements and the column
 * terms of its columns); the partial vectors are then added and merged with
 * beta*y.  These calls are the two steps.  A caller with N GPUs runs one
 * shard per GPU, gathers the N partial vectors (plain copies, e.g. an NCCL
 * all-gather) and runs the reduction; the sum is taken in rank order, so
 * the result is bit-identical from run to run for a fixed N and split.
 *
 * xsymv_shard_bounds: column boundaries of an even split of the stored
 *   triangle of order n into nparts panels: panel r is columns
 *   bounds[r] .. bounds[r+1]-1 (bounds has nparts + 1 entries; bounds[0] = 0,
 *   bounds[nparts] = n, nondecreasing; a panel may be empty).  Each panel
 *   holds about 1/nparts of the stored elements; inner boundaries are
 *   multiples of 16 columns (or n).  Host only (no CUDA call).  Returns 0, or the
 *   position of the first bad argument (1 uplo, 2 n < 0, 3 nparts < 1,
 *   4 bounds NULL).
 *
 * x<sy|he>mv_<k>_shard(uplo, n, col_begin, col_end, A, lda, x, incx, partial):
 *   the panel of stored columns col_begin <= j < col_end (0 <= col_begin <=
 *   col_end <= n) of the symmetric / Hermitian matrix of order n.
 *   A      DEVICE pointer to the panel alone, column-major with leading
 *          dimension lda: element (i, j) (matrix indices) at
 *          A[(i - r0) + (j - col_begin)*lda], with r0 = 0 for uplo 'U' (the
 *          panel has rows 0 .. col_end-1) and r0 = col_begin for 'L' (rows
 *          col_begin .. n-1).  Only the stored triangle's elements are used
 *          (as for xsymv_s: on a 16-byte aligned panel whose boundaries are
 *          multiples of 16 bytes, vectors in diagonal tiles may also fetch a
 *          few unused elements beside the diagonal, inside the panel).
 *   lda    >= max(1, panel rows): col_end for 'U', n - col_begin for 'L'.
 *   x      DEVICE pointer to all of x (n elements, stride incx != 0).
 *   partial DEVICE pointer to n contiguous elements, all written: the
 *          panel's contribution to A*x (no alpha, no beta; zero for an empty
 *          panel and for rows the panel does not reach).
 *   Returns 0, the position of the first bad argument (1 uplo, 2 n,
 *   3 col_begin, 4 col_end, 6 lda, 8 incx; nothing enqueued), or XSYMV_ERR_*
 *   (XSYMV_ERR_VALUE for a forced "_tk" variant).  Uses the stream's
 *   workspace like the other calls; asynchronous on the library's stream.
 *
 * x<sy|he>mv_<k>_reduce(n, nparts, alpha, partials, ldp, beta, y, incy):
 *   y := alpha * (P_0 + P_1 + ... + P_{nparts-1}) + beta * y, where P_r is
 *   the n contiguous elements at partials + r*ldp (DEVICE), added left to
 *   right in r order.  y: DEVICE, stride incy (negative: BLAS order), only
 *   y(0..n-1) written; beta = 0: y not read; alpha = 0: partials not read;
 *   alpha = 0 and beta = 1: nothing touched.  Returns 0, the position of the
 *   first bad argument (1 n < 0, 2 nparts < 1, 5 ldp < max(1, n), 8 incy = 0;
 *   nothing enqueued) or XSYMV_ERR_CUDA. */
XSYMV_API int xsymv_shard_bounds(char uplo, int n, int nparts, int *bounds);

XSYMV_API int xsymv_s_shard(char uplo, int n, int col_begin, int col_end, const float *A,
                            int lda, const float *x, int incx, float *partial);
XSYMV_API int xsymv_d_shard(char uplo, int n, int col_begin, int col_end, const double *A,
                            int lda, const double *x, int incx, double *partial);
XSYMV_API int xhemv_c_shard(char uplo, int n, int col_begin, int col_end, const xsymv_c32 *A,
                            int lda, const xsymv_c32 *x, int incx, xsymv_c32 *partial);
XSYMV_API int xhemv_z_shard(char uplo, int n, int col_begin, int col_end, const xsymv_c64 *A,
                            int lda, const xsymv_c64 *x, int incx, xsymv_c64 *partial);
XSYMV_API int xsymv_w_shard(char uplo, int n, int col_begin, int col_end, const xsymv_dd *A,
                            int lda, const xsymv_dd *x, int incx, xsymv_dd *partial);

XSYMV_API int xsymv_s_reduce(int n, int nparts, float alpha, const float *partials,
                             long long ldp, float beta, float *y, int incy);
XSYMV_API int xsymv_d_reduce(int n, int nparts, double alpha, const double *partials,
                             long long ldp, double beta, double *y, int incy);
XSYMV_API int xhemv_c_reduce(int n, int nparts, xsymv_c32 alpha, const xsymv_c32 *partials,
                             long long ldp, xsymv_c32 beta, xsymv_c32 *y, int incy);
XSYMV_API int xhemv_z_reduce(int n, int nparts, xsymv_c64 alpha, const xsymv_c64 *partials,
                             long long ldp, xsymv_c64 beta, xsymv_c64 *y, int incy);
XSYMV_API int xsymv_w_reduce(int n, int nparts, xsymv_dd alpha, const xsymv_dd *partials,
                             long long ldp, xsymv_dd beta, xsymv_dd *y, int incy);

/* ---- host-buffer variants ----------------------------------------------
 * Same arguments, semantics and status codes as the five calls above, but A,
 * x and y are HOST pointers (device pointers also work).  When all three are
 * page-locked (pinned or cudaHostRegister'ed) host memory, the kernels read
 * A and x and write y in place over the host link (zero-copy; only the
 * stored triangle crosses the link).  Otherwise each call copies the stored
 * triangle (in column panels, so at most a few percent of the other
 * triangle travels too), x and, when beta != 0, y into library-owned device
 * buffers, runs the same kernels and copies the n elements of y back.  The
 * call waits for the current stream: y holds the result when it returns.
 * Staging buffers are kept per (device, stream) for reuse, like the
 * workspace.  On a CUDA error y may be partly written. */
XSYMV_API int xsymv_s_host(char uplo, int n, float alpha, const float *A, int lda,
                           const float *x, int incx, float beta, float *y, int incy);
XSYMV_API int xsymv_d_host(char uplo, int n, double alpha, const double *A, int lda,
                           const double *x, int incx, double beta, double *y, int incy);
XSYMV_API int xhemv_c_host(char uplo, int n, xsymv_c32 alpha, const xsymv_c32 *A, int lda,
                           const xsymv_c32 *x, int incx, xsymv_c32 beta, xsymv_c32 *y, int incy);
XSYMV_API int xhemv_z_host(char uplo, int n, xsymv_c64 alpha, const xsymv_c64 *A, int lda,
                           const xsymv_c64 *x, int incx, xsymv_c64 beta, xsymv_c64 *y, int incy);
XSYMV_API int xsymv_w_host(char uplo, int n, xsymv_dd alpha, const xsymv_dd *A, int lda,
                           const xsymv_dd *x, int incx, xsymv_dd beta, xsymv_dd *y, int incy);

/* Bytes the last host-buffer call moved host-to-device and back (copied,
 * or read / written in place over the link). */
XSYMV_API int xsymv_host_traffic(long long *h2d_bytes, long long *d2h_bytes);

/* Stream for subsequent calls from any thread (a cudaStream_t; NULL = the
 * legacy default stream).  Returns 0. */
XSYMV_API int xsymv_set_stream(void *stream);
XSYMV_API void *xsymv_get_stream(void);

/* ---- failure detection -------------------------------------------------
 * Every wait inside the kernels has a time limit, 2 s by default: waits for
 * bulk copies landing in shared memory (the "_t" variants) and waits for a
 * ticket (the "_tk" variants).  If a copy wait runs out, the kernel records
 * the failure in the workspace, waits (again with the limit) for its copies
 * in flight and returns; the call's y is then filled with NaN.  If a ticket
 * wait runs out, the kernel records the failure and every element of y
 * whose sum could not be completed is set to NaN (elements whose sums
 * completed keep their results).
 * xsymv_sync_status waits for the current stream and returns
 * XSYMV_ERR_TIMEOUT if the latest call on it (device, stream) failed that
 * way, else 0 (or XSYMV_ERR_CUDA).  That covers every SYMV entry point,
 * xsymv_s_noalloc included; a call with nothing that waits (alpha = 0, the
 * general product) reports 0. */
XSYMV_API int xsymv_sync_status(void);
/* Time limit of those waits in ns (0: back to 2 s). */
XSYMV_API int xsymv_set_wait_limit(unsigned long long ns);
/* Test hook: on != 0 makes every bulk-copy barrier expect 16 bytes that
 * never arrive, and makes the first contributor of every ticket chain keep
 * its ticket, so the next calls' waits run out (nothing faults; the kernels
 * return after the time limit).  0 restores normal operation. */
XSYMV_API int xsymv_test_stall(int on);
/* Test hook: sets the last call number handed out on the current device and
 * stream (calls number themselves 1, 2, ... to tag failures in the status
 * word; after 0x7ffffffe they start again at 1 and the status word is
 * cleared), and that of xsymv_s_noalloc on the current device.
 * 0 <= number <= 0x7ffffffe, and the stream must have a workspace or the
 * device an xsymv_s_noalloc call (one earlier call); else XSYMV_ERR_VALUE,
 * nothing changed. */
XSYMV_API int xsymv_test_set_call_number(int number);

/* Human-readable text for a status code (static storage). */
XSYMV_API const char *xsymv_status_string(int status);

/* The cudaError_t of the last failed CUDA call (0 if none). */
XSYMV_API int xsymv_last_cuda_error(void);

/* ---- measurement hooks (used by the benchmark; off by default) ---------- */

/* Record CUDA events around each call's main kernel and whole call on the
 * call's stream.  on = 0 disables and discards what was recorded. */
XSYMV_API int xsymv_timing_enable(int on);

/* Wait for the recorded events, then report the number of timed calls and
 * the summed device time of their main kernels and of the whole calls (ms).
 * Clears the record.  Returns 0, or XSYMV_ERR_CUDA. */
XSYMV_API int xsymv_timing_read(int *calls, double *main_ms, double *call_ms);

/* Roofline denominators measured now on the current device and stream:
 * HBM copy bandwidth (bytes read + written per second, 1 GiB buffers), HBM
 * read bandwidth, and FP64 / FP32 FMA throughput (2 flops per FMA) of a loop
 * of nothing but FMAs with register operands, each the best of a few timed
 * runs.  Allocates and frees two 1 GiB buffers; synchronises the stream.
 * Any output pointer may be NULL. */
XSYMV_API int xsymv_probe_peaks(double *copy_gbs, double *read_gbs, double *fp64_tflops,
                                double *fp32_tflops);

/* The double-double kernels issue every rounded sum, difference and
 * product of two doubles as a fused multiply-add with a unit operand
 * (a + b = fma(a, 1, b), a - b = fma(b, -1, a), a * b = fma(a, b, -0)),
 * which IEEE 754 makes bit-identical to the plain operations and which
 * GB300 issues faster.  This entry checks that on the current device: for
 * i < n it writes out[6i .. 6i+5] = a[i]+b[i], a[i]-b[i], a[i]*b[i] by the
 * plain instructions, then the same three in the kernels' form.  a, b: n
 * doubles; out: 6n doubles; all device memory, not overlapping.  Enqueued
 * on the current stream (no synchronisation).  Returns 0, XSYMV_ERR_VALUE
 * (n < 0, or a NULL pointer with n > 0), XSYMV_ERR_DEVICE or
 * XSYMV_ERR_CUDA.
 * No counterpart in the report: it backs the GB300 form of the DD steps. */
XSYMV_API int xsymv_probe_unit_forms(const double *a, const double *b, double *out,
                                     long long n);

/* Number of kernels this library has launched since it was loaded. */
XSYMV_API long long xsymv_launch_count(void);

/* ---- kernel variants: the tuner's parameter space ----------------------- */

/* kind: 's', 'd', 'c', 'z' or 'w'.  Number of compiled variants (0 for an
 * unknown kind) and the name of variant index: "vr<VR>_u<U>_<p><S>_w<W>"
 * with optional suffixes "_b<B>", "_x<X>", "_g<G>", "_c<R>", "_tk", "_f" =
 * 16-byte vectors per lane (the tile edge is 32 lanes x VR vectors),
 * columns per load step, how off-diagonal columns reach the arithmetic
 * (p = r: 16-byte loads into registers; t: a per-warp shared-memory ring of
 * S chunks filled by bulk (TMA) copies), warps per block, a register cap
 * that fits B blocks per SM, X waves of blocks, the partition cost G of a
 * diagonal-tile column (a dense one costs 4), column reductions batched
 * over R columns, and "_tk": the partial sums are combined by ordered
 * tickets in the same launch (the report's mechanism, §2.1, figures
 * "kernel" and "Atomic": dynamic block IDs, one ticket per chunk of NB
 * outputs passed from contributor to contributor in a fixed order) instead
 * of by a second, fixed-order reduction kernel, and "_f": the fixed-order
 * sums in the same launch, after a grid-wide barrier (one launch per call,
 * the same sums as the two-kernel path of the same plan).  A tuned "_f"
 * variant gives way to its two-kernel twin (the same name without "_f")
 * while calls on a stream run back to back, since two-kernel calls fill
 * each other's tails; the twin runs the same plan, so the results are the
 * same bytes.  A forced variant (xsymv_set_variant) is always used as is.
 * All are bit-identical from run to run; "_tk" results differ from the
 * others only in rounding. */
XSYMV_API int xsymv_variant_count(char kind);
XSYMV_API const char *xsymv_variant_name(char kind, int index);

/* Force variant index for kind (-1: the built-in tuned choice).
 * Returns 0 or XSYMV_ERR_VALUE.  xsymv_s_noalloc refuses a forced "_tk"
 * variant (XSYMV_ERR_VALUE, nothing enqueued): it has no ticket buffer. */
XSYMV_API int xsymv_set_variant(char kind, int index);

/* The variant index a call of this kind, uplo and n would use. */
XSYMV_API int xsymv_selected_variant(char kind, char uplo, int n);

/* Workspace bytes a call of this kind, uplo and n needs on the current
 * device: the 256-byte header and one set of partial sums (what
 * xsymv_s_noalloc needs; the stream workspaces of the other entry points
 * hold two sets and 256 bytes more).  < 0: XSYMV_ERR_*.  A "_tk"
 * variant's ticket buffer (256 bytes + 32 bytes per chunk of NB outputs) is
 * not included. */
XSYMV_API long long xsymv_workspace_bytes(char kind, char uplo, int n);

/* ---- the general product, for comparison ------------------------------
 * "CUDA-xSYMV の実装と評価" (IPSJ 2014-HPC-146), §1 and the abstract:
 * SYMV reads half the matrix that the general matrix-vector product (GEMV)
 * reads, so a memory-bound SYMV is expected to run at about twice GEMV's
 * speed.  These calls are that GEMV, streamed by the same warp loader as the
 * SYMV kernels, so that the claim can be measured on one GPU:
 *
 *   y := alpha*A*x + beta*y,  A an n-by-n general matrix (no symmetry; all
 *   n*n elements are read), column-major with leading dimension lda, no
 *   transpose.  A, x and y are DEVICE pointers owned by the caller; A and x
 *   are read only; y(0..n-1, incy) is the only memory written.  Negative
 *   incx / incy start from the end (BLAS).  beta = 0 overwrites y without
 *   reading it; alpha = 0 reads neither A nor x; n = 0 or (alpha = 0,
 *   beta = 1) returns at once.  Results are bit-identical from run to run
 *   for a fixed variant, stream and device.  Asynchronous on the library's
 *   stream, like the SYMV calls.
 *
 * Returns 0, or the position of the first bad argument in this signature
 * (1: n < 0; 4: lda < max(1, n); 6: incx = 0; 9: incy = 0) with nothing
 * enqueued, or a negative XSYMV_ERR_* code. */
XSYMV_API int xgemv_s(int n, float alpha, const float *A, int lda, const float *x, int incx,
                      float beta, float *y, int incy);
XSYMV_API int xgemv_d(int n, double alpha, const double *A, int lda, const double *x, int incx,
                      double beta, double *y, int incy);

/* type 's' or 'd': the compiled GEMV variants (names as for the SYMV
 * register path, "vr<VR>_u<U>_r0_w<W>[_b<B>]"), forcing one (-1: variant 0),
 * and the index the next call uses.  XSYMV_ERR_VALUE for another type or an
 * index out of range (count: XSYMV_ERR_VALUE; name: NULL). */
XSYMV_API int xgemv_variant_count(char type);
XSYMV_API const char *xgemv_variant_name(char type, int index);
XSYMV_API int xgemv_set_variant(char type, int index);
XSYMV_API int xgemv_selected_variant(char type);

#ifdef __cplusplus
}
#endif
#endif /* XSYMV_H */
