// Host dispatch shared by the five entry points: BLAS argument checks, quick
// returns, variant choice, work partition, workspace and the launches (main
// kernel and finaliser, or the one ordered-ticket kernel).
#pragma once

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "../../include/xsymv.h"
#include "xsymv_fused.cuh"
#include "xsymv_kernels.cuh"
#include "xsymv_ticket.cuh"
#include "xsymv_runtime.h"
#include "xsymv_tuned.h"

namespace xsymv {

// Workspace layout: a 256-byte header (word 0: the status word the main
// kernel sets to the call's epoch when a bounded wait runs out; bytes 8-15:
// the one-launch kernels' grid barrier; bytes 16-47: the finalisers' end
// times and the early main kernels' start times, one per call parity), then
// the column partials Wc, then the row partials Wr (two such sets in the
// stream workspaces).
constexpr long long kHeaderBytes = 256;
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;   // 2 s

// Partition costs (see xsymv_plan.h): a dense column costs kDenseCost; a
// diagonal-tile column (masked, and stepped one column at a time for the
// single-precision kinds) costs more for the bandwidth-bound types and less
// for the FP64-bound ones (it holds half a column's elements on average).
// These are the defaults of the untuned variants; the tuned ones carry their
// own cost (_g<G>).
constexpr int kDenseCost = 4;
template <class T> struct DiagCost { static constexpr int v = 4; };
template <> struct DiagCost<float> { static constexpr int v = 6; };
template <> struct DiagCost<c32> { static constexpr int v = 6; };
template <> struct DiagCost<double> { static constexpr int v = 3; };
template <> struct DiagCost<c64> { static constexpr int v = 3; };
template <> struct DiagCost<dd> { static constexpr int v = 3; };

// Everything one launch of the main kernel needs.
template <class T>
struct MainArgs {
  Plan plan;
  const T* A;
  long long lda;
  const T* x;      // logical element 0
  int incx;
  T* Wc;
  T* Wr;
  int* status;
  int epoch;
  bool aligned;    // A and lda*sizeof(T) on the 16-byte grid
  cudaStream_t stream;
  // ordered-ticket and one-launch (fused) variants: the final merge happens
  // in the same launch
  T* v = nullptr;                  // n running sums (in the workspace, after Wr; tickets)
  void* tk = nullptr;              // ticket buffer (counters, then the tickets)
  unsigned long long call = 0;     // the call's number in the tickets
  T alpha{}, beta{};
  int mode = 0;                    // kFull, kBetaZero (or, fused, kPartial)
  T* y0 = nullptr;                 // logical element 0 of y
  long long incy = 0;
  // the plan's warp and row tables (built before the launch)
  const int4* wt = nullptr;
  const int2* rt = nullptr;
  // the main kernel may stream before the stream's previous kernel (the
  // previous call's finaliser) completes; it waits for it at its end, and
  // notes its start time in the workspace header
  int early = 0;
  // one-launch variants: the header words of the back-to-back bookkeeping
  // (all null: none)
  OverlapWords ow{nullptr, nullptr, nullptr, nullptr};
};

// One compiled configuration of the main kernel.
template <class T>
struct Variant {
  const char* name;
  int NB;      // tile edge = 32 lanes * elements per 16 bytes * VR
  int warps;   // warps per block
  int stages;  // shared-memory ring depth
  int pipe;    // enum Pipe
  int waves;   // warps launched = waves x the warps that fit on the GPU at once
  int diag_cost;  // partition cost of a diagonal-tile column (a dense one costs kDenseCost)
  cudaError_t (*launch)(const MainArgs<T>&);
  int (*ctas_per_sm)();
  int accum;   // enum Accum: workspace + finaliser, or ordered tickets (launch does it all)
};

template <class T, int VR, int U, int S, int P, int WARPS>
constexpr int ring_smem_bytes() {
  return WARPS * RingLayout<T, VR, U, S, P>::WARP_BYTES;
}

template <class T, int VR, int U, int S, int P, int WARPS, int MB, int R = U>
cudaError_t launch_main(const MainArgs<T>& a) {
  constexpr int smem = ring_smem_bytes<T, VR, U, S, P, WARPS>();
  if (smem > 48 * 1024) {
    // the attribute is per device: set once on each device this kernel runs on
    static std::atomic<int> configured[kMaxDevices];
    const int dev = current_device_index();
    if (dev < 0 || !configured[dev].load(std::memory_order_relaxed)) {
      cudaError_t e = cudaFuncSetAttribute(symv_main<T, VR, U, S, P, WARPS, true, MB, R>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      if (dev >= 0) configured[dev].store(1, std::memory_order_relaxed);
    }
  }
  const unsigned long long limit = wait_limit_ns();
  const uint32_t extra = test_extra_tx();
  // programmatic dependent launch: the blocks may be scheduled while the
  // stream's previous kernel finishes; the kernel waits for its completion
  // (griddepcontrol.wait) before touching global memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.plan.W + WARPS - 1) / WARPS));
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = a.aligned ? smem : 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.aligned)
    return cudaLaunchKernelEx(&cfg, symv_main<T, VR, U, S, P, WARPS, true, MB, R>, a.plan, a.A,
                              a.lda, a.x, a.incx, a.Wc, a.Wr, a.wt, a.rt, a.status, a.epoch,
                              limit, extra, a.early);
  return cudaLaunchKernelEx(&cfg, symv_main<T, VR, U, S, P, WARPS, false, MB, R>, a.plan, a.A,
                            a.lda, a.x, a.incx, a.Wc, a.Wr, a.wt, a.rt, a.status, a.epoch, limit,
                            extra, a.early);
}

// resident blocks per SM of one kernel on the current device, computed once
// per device by `count` (a result < 1 counts as 1)
template <class F>
int per_device_count(std::atomic<int> (&cache)[kMaxDevices], F count) {
  const int dev = current_device_index();
  int b = dev >= 0 ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (b == 0) {
    b = count();
    if (b < 1) {
      cudaGetLastError();
      b = 1;
    }
    if (dev >= 0) cache[dev].store(b, std::memory_order_relaxed);
  }
  return b;
}

template <class T, int VR, int U, int S, int P, int WARPS, int MB, int R = U>
int ctas_per_sm() {
  static std::atomic<int> cache[kMaxDevices];
  return per_device_count(cache, [] {
    constexpr int smem = ring_smem_bytes<T, VR, U, S, P, WARPS>();
    int b = 0;
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(symv_main<T, VR, U, S, P, WARPS, true, MB, R>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, symv_main<T, VR, U, S, P, WARPS, true, MB, R>,
                                                      WARPS * 32, smem) != cudaSuccess)
      b = 0;
    return b;
  });
}

// The ordered-ticket kernel (register path): one launch streams the triangle,
// chains the partial sums through the tickets and writes y.
template <class T, int VR, int U, int WARPS, int MB, int R>
cudaError_t launch_ticket(const MainArgs<T>& a) {
  const unsigned grid = (unsigned)((a.plan.W + WARPS - 1) / WARPS);
  TicketCtx<T> c;
  c.Wc = a.Wc;
  c.Wr = a.Wr;
  c.v = a.v;
  c.tk = reinterpret_cast<unsigned long long*>(static_cast<char*>(a.tk) + kTkHeaderBytes);
  c.status = a.status;
  c.epoch = a.epoch;
  c.call = a.call;
  c.limit_ns = wait_limit_ns();
  c.withhold = test_extra_tx() != 0;
  c.alpha = a.alpha;
  c.beta = a.beta;
  c.mode = a.mode;
  c.y = a.y0;
  c.incy = a.incy;
  c.rt = a.rt;
  int* ctr = static_cast<int*>(a.tk);
  if (a.aligned)
    symv_ticket<T, VR, U, WARPS, true, MB, R><<<grid, WARPS * 32, 0, a.stream>>>(
        a.plan, a.A, a.lda, a.x, a.incx, a.Wc, a.Wr, a.wt, a.rt, ctr, c);
  else
    symv_ticket<T, VR, U, WARPS, false, MB, R><<<grid, WARPS * 32, 0, a.stream>>>(
        a.plan, a.A, a.lda, a.x, a.incx, a.Wc, a.Wr, a.wt, a.rt, ctr, c);
  return cudaGetLastError();
}

template <class T, int VR, int U, int WARPS, int MB, int R>
int ctas_per_sm_ticket() {
  static std::atomic<int> cache[kMaxDevices];
  return per_device_count(cache, [] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, symv_ticket<T, VR, U, WARPS, true, MB, R>,
                                                      WARPS * 32, 0) != cudaSuccess)
      b = 0;
    return b;
  });
}

// The one-launch kernel (register path): streams, meets at a grid barrier,
// then every block takes a share of the final merge.  A cooperative launch
// (every block resident at once) and, like the main kernel, a programmatic
// dependent of the stream's previous kernel.
template <class T, int VR, int U, int WARPS, int MB, int R>
cudaError_t launch_fused(const MainArgs<T>& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.plan.W + WARPS - 1) / WARPS));
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const FinalArgs<T> f{a.alpha, a.beta, a.mode, a.y0, a.incy};
  unsigned long long* bar =
      reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(a.status) + kBarrierOffset);
  const unsigned long long limit = wait_limit_ns();
  const int stall = test_extra_tx() != 0;
  if (a.aligned)
    return cudaLaunchKernelEx(&cfg, symv_fused<T, VR, U, WARPS, true, MB, R>, a.plan, a.A, a.lda,
                              a.x, a.incx, a.Wc, a.Wr, a.wt, a.rt, a.status, a.epoch, limit, stall,
                              bar, f, a.ow);
  return cudaLaunchKernelEx(&cfg, symv_fused<T, VR, U, WARPS, false, MB, R>, a.plan, a.A, a.lda,
                            a.x, a.incx, a.Wc, a.Wr, a.wt, a.rt, a.status, a.epoch, limit, stall,
                            bar, f, a.ow);
}

template <class T, int VR, int U, int WARPS, int MB, int R>
int ctas_per_sm_fused() {
  static std::atomic<int> cache[kMaxDevices];
  return per_device_count(cache, [] {
    int b = 0;
    // the smaller of the two instantiations' residencies: the grid must fit
    // whole whichever one runs
    int b2 = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, symv_fused<T, VR, U, WARPS, true, MB, R>,
                                                      WARPS * 32, 0) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, symv_fused<T, VR, U, WARPS, false, MB, R>,
                                                      WARPS * 32, 0) != cudaSuccess)
      return 0;
    return b < b2 ? b : b2;
  });
}

// Variant names: vr<VR>_u<U>_<pipe><STAGES>_w<WARPS>[_b<MINB>][_x<WAVES>][_g<G>][_c<R>][_tk|_f],
// pipe r = loads into registers, t = bulk-copy (TMA) ring of STAGES chunks
// per warp; _b<MINB>: registers capped so that MINB blocks fit on an SM;
// _x<WAVES>: that many waves of blocks instead of one resident wave;
// _g<G>: partition cost G of a diagonal-tile column (default DiagCost);
// _c<R>: column reductions batched over R columns (default U);
// _tk: ordered tickets instead of the workspace finaliser (symv_ticket);
// _f: the workspace sums in the same launch, after a grid barrier (symv_fused).
#define XSYMV_VARIANT_G(T, VR, U, S, P, L, W, MB, X, G, SUF)                              \
  Variant<T> {                                                                            \
    "vr" #VR "_u" #U "_" L #S "_w" #W SUF, 32 * Ops<T>::VPL * (VR), (W), (S), (P), (X),  \
        (G), &launch_main<T, VR, U, S, P, W, MB>, &ctas_per_sm<T, VR, U, S, P, W, MB>,    \
        kAccumWorkspace                                                                   \
  }
#define XSYMV_VARIANT_P(T, VR, U, S, P, L, W, MB, X, SUF) \
  XSYMV_VARIANT_G(T, VR, U, S, P, L, W, MB, X, DiagCost<T>::v, SUF)
#define XSYMV_REG(T, VR, U, W) XSYMV_VARIANT_P(T, VR, U, 0, kPipeRegisters, "r", W, 0, 1, "")
#define XSYMV_REG_MB(T, VR, U, W, MB) \
  XSYMV_VARIANT_P(T, VR, U, 0, kPipeRegisters, "r", W, MB, 1, "_b" #MB)
// X waves of warps: each warp gets 1/X of a resident warp's share and the
// hardware starts new blocks as earlier ones finish
#define XSYMV_REG_MBX(T, VR, U, W, MB, X) \
  XSYMV_VARIANT_P(T, VR, U, 0, kPipeRegisters, "r", W, MB, X, "_b" #MB "_x" #X)
// diagonal-tile columns costed G (dense = kDenseCost) in the partition
#define XSYMV_REG_G(T, VR, U, W, MB, G) \
  XSYMV_VARIANT_G(T, VR, U, 0, kPipeRegisters, "r", W, MB, 1, G, "_b" #MB "_g" #G)
#define XSYMV_TMA(T, VR, U, S, W) XSYMV_VARIANT_P(T, VR, U, S, kPipeBulk, "t", W, 0, 1, "")
// column reductions batched over R columns (_c<R>), diagonal cost G
#define XSYMV_REG_GC(T, VR, U, W, MB, G, R)                                                  \
  Variant<T> {                                                                              \
    "vr" #VR "_u" #U "_r0_w" #W "_b" #MB "_g" #G "_c" #R, 32 * Ops<T>::VPL * (VR), (W), 0,    \
        kPipeRegisters, 1, (G), &launch_main<T, VR, U, 0, kPipeRegisters, W, MB, R>,           \
        &ctas_per_sm<T, VR, U, 0, kPipeRegisters, W, MB, R>, kAccumWorkspace                  \
  }

// ordered tickets (register path): diagonal cost G, batched reductions R
#define XSYMV_TICKET(T, VR, U, W, MB, G, R)                                                     \
  Variant<T> {                                                                                \
    "vr" #VR "_u" #U "_r0_w" #W "_b" #MB "_g" #G "_c" #R "_tk", 32 * Ops<T>::VPL * (VR), (W), 0, \
        kPipeRegisters, 1, (G), &launch_ticket<T, VR, U, W, MB, R>,                            \
        &ctas_per_sm_ticket<T, VR, U, W, MB, R>, kAccumTickets                                 \
  }

// one launch: the main kernel and the final merge after a grid barrier
// (8 warps per block: one finaliser block's threads)
#define XSYMV_FUSED(T, VR, U, W, MB, G, R)                                                      \
  Variant<T> {                                                                                \
    "vr" #VR "_u" #U "_r0_w" #W "_b" #MB "_g" #G "_c" #R "_f", 32 * Ops<T>::VPL * (VR), (W), 0,  \
        kPipeRegisters, 1, (G), &launch_fused<T, VR, U, W, MB, R>,                             \
        &ctas_per_sm_fused<T, VR, U, W, MB, R>, kAccumFused                                    \
  }

// The finaliser's grid: one block per group of kFinCols outputs, or, when
// `compact`, at most one block per SM, each taking the groups g, g + grid,
// ... in turn.  The compact grid is slower on its own (its blocks add their
// groups one after another), but it becomes resident, and so lets the next
// call's main kernel launch, while this call's main kernel still has blocks
// running: back-to-back calls then fill each other's tails.  It is used
// while calls on the stream really overlap (each main kernel that started
// early reports whether it began before the previous finaliser ended);
// isolated calls, calls with other work between them and calls that read
// the previous result keep the full grid.  The sums, hence the results, are
// the same either way.  ow: see OverlapWords (all null: not used).
template <class T>
cudaError_t launch_finalize(const Plan& p, const T* Wc, const T* Wr, const int2* rt, T alpha,
                            T beta, int mode, T* y0, long long incy, const int* status, int epoch,
                            cudaStream_t st, bool compact = false,
                            OverlapWords ow = OverlapWords{nullptr, nullptr, nullptr, nullptr}) {
  // programmatic dependent launch: the launch overlaps the tail of the main
  // kernel, whose completion the finaliser awaits with griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  long long groups = (p.n + kFinCols - 1) / kFinCols;
  int dev = 0, sms = 0;
  if (compact && current_device(&dev, &sms) && groups > (long long)sms) groups = sms;
  cfg.gridDim = dim3((unsigned)groups);
  cfg.blockDim = dim3(kFinParts * kFinCols);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, symv_finalize<T>, p, Wc, Wr, rt, alpha, beta, mode, y0, incy,
                            status, epoch, ow);
}

// ----------------------------------------------------------- plan tables --
// The bytes that identify a plan's tables (all ints: no padding).
struct TablesKey {
  int n, NB, upper, cd, cg, W, G, c0, c1;
};

inline TablesKey tables_key(const Plan& p) {
  return TablesKey{p.n, p.NB, p.upper, p.cd, p.cg, p.W, p.G, p.c0, p.c1};
}

// bytes of the warp table (int4 per warp) followed by the row table (int2
// per block row)
inline long long tables_bytes(const Plan& p) {
  return ((long long)p.W * 16 + 255) / 256 * 256 + (long long)p.nb * 8;
}

inline cudaError_t launch_plan_tables(const Plan& p, void* buf, cudaStream_t st) {
  const long long m = p.W > p.nb ? p.W : p.nb;
  symv_plan_tables<<<(unsigned)((m + 255) / 256), 256, 0, st>>>(
      p, static_cast<int4*>(buf),
      reinterpret_cast<int2*>(static_cast<char*>(buf) + ((long long)p.W * 16 + 255) / 256 * 256));
  return cudaGetLastError();
}

// Point *wt, *rt at the tables of plan p for this stream, building them
// first (one small launch) if the stream's table buffer holds another plan's.
inline int ensure_tables(const Plan& p, cudaStream_t st, const int4** wt, const int2** rt) {
  const TablesKey key = tables_key(p);
  bool ready = false;
  int status = XSYMV_OK;
  void* buf = plan_tables((size_t)tables_bytes(p), st, &key, sizeof(key), &ready, &status);
  if (!buf) return status;
  if (!ready) {
    cudaError_t e = launch_plan_tables(p, buf, st);
    if (e != cudaSuccess) {
      plan_tables_forget(st);
      record_cuda_error(e);
      return XSYMV_ERR_CUDA;
    }
    note_launches(1);
  }
  *wt = static_cast<const int4*>(buf);
  *rt = reinterpret_cast<const int2*>(static_cast<char*>(buf) +
                                      ((long long)p.W * 16 + 255) / 256 * 256);
  return XSYMV_OK;
}

// ---------------------------------------------------------------- checks --
inline int check_args(char uplo, int n, int lda, int incx, int incy) {
  if (uplo != 'U' && uplo != 'u' && uplo != 'L' && uplo != 'l') return 1;
  if (n < 0) return 2;
  if (lda < (n > 1 ? n : 1)) return 5;
  if (incx == 0) return 7;
  if (incy == 0) return 10;
  return 0;
}

inline bool is_zero(float a) { return a == 0.f; }
inline bool is_zero(double a) { return a == 0.0; }
inline bool is_zero(c32 a) { return a.re == 0.f && a.im == 0.f; }
inline bool is_zero(c64 a) { return a.re == 0.0 && a.im == 0.0; }
inline bool is_zero(dd a) { return a.hi == 0.0 && a.lo == 0.0; }
inline bool is_one(float a) { return a == 1.f; }
inline bool is_one(double a) { return a == 1.0; }
inline bool is_one(c32 a) { return a.re == 1.f && a.im == 0.f; }
inline bool is_one(c64 a) { return a.re == 1.0 && a.im == 0.0; }
inline bool is_one(dd a) { return a.hi == 1.0 && a.lo == 0.0; }

inline long long align_up(long long v, long long a) { return (v + a - 1) / a * a; }

template <class T>
struct Workload {
  Plan plan;
  const Variant<T>* variant;
  long long wc_off;     // byte offset of Wc in the workspace
  long long wr_off;     // byte offset of Wr
  long long v_off;      // byte offset of v (ordered-ticket variants)
  long long bytes;      // total workspace bytes
  int twin;             // one-launch variant: its two-kernel twin (the same kernel code
                        // without the final merge), which runs this plan in one wave,
                        // else -1
};

// The two-kernel variant of a one-launch variant: the same name without
// "_f" (and without "_c<R>" when R is U, the default), -1 if there is none.
template <class T>
int twin_index(const Variant<T>* table, int count, int vi) {
  const char* nm = table[vi].name;
  const size_t len = strlen(nm);
  char buf[96];
  if (table[vi].accum != kAccumFused || len < 3 || len - 2 >= sizeof(buf) ||
      strcmp(nm + len - 2, "_f") != 0)
    return -1;
  memcpy(buf, nm, len - 2);
  buf[len - 2] = '\0';
  for (int pass = 0; pass < 2; ++pass) {
    for (int i = 0; i < count; ++i)
      if (table[i].accum == kAccumWorkspace && strcmp(table[i].name, buf) == 0) return i;
    // "_c<R>" with R = U names the default reduction: the twin omits it
    const char* u = strstr(buf, "_u");
    char* c = strrchr(buf, '_');
    if (pass == 0 && u != nullptr && c != nullptr && c[1] == 'c' && atoi(c + 2) == atoi(u + 2))
      *c = '\0';
    else
      break;
  }
  return -1;
}

// The variant a call uses: the forced one, else the tuned entry's variant,
// looked up by name in this kind's table (once per entry, then cached); 0 if
// the tuned table names no compiled variant.
template <class T>
int pick_variant(const Variant<T>* table, int count, char kind, int upper, int n) {
  int f = forced_variant(kind);
  if (f >= 0 && f < count) return f;
  const int e = tuned_entry(kind, upper, n);
  if (e < 0) return 0;
  // resolved[e] = variant index + 1 (0: not looked up yet)
  static std::atomic<int> resolved[kTunedCount];
  int r = resolved[e].load(std::memory_order_relaxed);
  if (r == 0) {
    r = 1;   // variant 0 unless the name is found
    for (int i = 0; i < count; ++i)
      if (strcmp(table[i].name, kTuned[e].variant) == 0) {
        r = i + 1;
        break;
      }
    resolved[e].store(r, std::memory_order_relaxed);
  }
  return r - 1;
}

// The plan of a call: the whole triangle, or only its stored columns
// c0 <= j < c1 (a shard; c1 < 0: n).  The variant is the one tuned for a
// whole triangle of order n_pick (default n).
template <class T>
int plan_call_uncached(const Variant<T>* table, int count, int upper, int n,
                       Workload<T>* out, int c0, int c1, int vi);

// The last few plans of this thread, by (table, device, triangle, n, window,
// variant): a call of a shape seen just before skips the partition
// arithmetic (its row loop is O(n / NB)) and the device queries.
template <class T>
int plan_call(const Variant<T>* table, int count, char kind, int upper, int n, Workload<T>* out,
              int c0 = 0, int c1 = -1, int n_pick = -1) {
  struct Entry {
    const Variant<T>* table;
    int dev, upper, n, c0, c1, vi;
    Workload<T> wl;
  };
  constexpr int kSlots = 4;
  thread_local Entry cache[kSlots] = {};
  thread_local int next = 0;
  const int vi = pick_variant(table, count, kind, upper, n_pick < 0 ? n : n_pick);
  const int dev = current_device_index();
  const int cc1 = c1 < 0 ? n : c1;
  if (dev >= 0)
    for (Entry& e : cache)
      if (e.table == table && e.dev == dev && e.upper == upper && e.n == n && e.c0 == c0 &&
          e.c1 == cc1 && e.vi == vi) {
        *out = e.wl;
        return XSYMV_OK;
      }
  const int status = plan_call_uncached(table, count, upper, n, out, c0, c1, vi);
  if (status == XSYMV_OK && dev >= 0) {
    cache[next] = Entry{table, dev, upper, n, c0, cc1, vi, *out};
    next = (next + 1) % kSlots;
  }
  return status;
}

template <class T>
int plan_call_uncached(const Variant<T>* table, int count, int upper, int n,
                       Workload<T>* out, int c0, int c1, int vi) {
  int dev = 0, sms = 0;
  if (!current_device(&dev, &sms)) return XSYMV_ERR_DEVICE;
  const Variant<T>* v = &table[vi];
  const long long wmax = (long long)sms * v->ctas_per_sm() * v->warps * v->waves;
  out->plan = plan_make(n, v->NB, upper, wmax, kDenseCost, v->diag_cost, v->warps, c0, c1);
  out->variant = v;
  out->wc_off = kHeaderBytes;
  out->wr_off = out->wc_off + align_up(plan_wc_elems(out->plan) * (long long)sizeof(T), 256);
  out->v_off = out->wr_off + align_up(plan_wr_elems(out->plan) * (long long)sizeof(T), 256);
  out->bytes = out->v_off;
  out->twin = -1;
  if (v->accum == kAccumTickets) {
    if (out->plan.W >= (1 << kTkIdBits)) return XSYMV_ERR_VALUE;
    out->bytes += align_up((long long)n * (long long)sizeof(T), 256);
  }
  if (v->accum == kAccumFused) {
    const int t = twin_index(table, count, vi);
    if (t >= 0 && table[t].ctas_per_sm() >= v->ctas_per_sm()) out->twin = t;
  }
  return XSYMV_OK;
}

// -------------------------------------------------------------- the call --
template <class T>
int symv_entry(const Variant<T>* table, int count, char kind, char uplo, int n, T alpha,
               const T* A, int lda, const T* x, int incx, T beta, T* y, int incy) {
  int info = check_args(uplo, n, lda, incx, incy);
  if (info) return info;
  if (n == 0) return XSYMV_OK;
  const bool az = is_zero(alpha), bz = is_zero(beta);
  if (az && is_one(beta)) return XSYMV_OK;

  const int upper = (uplo == 'U' || uplo == 'u');
  cudaStream_t st = current_stream();
  // pointers to logical element 0 (BLAS: negative strides start at the end)
  T* y0 = y + (incy < 0 ? (long long)(1 - n) * incy : 0);
  const T* x0 = x + (incx < 0 ? (long long)(1 - n) * incx : 0);

  if (az) {  // y := beta*y: neither A nor x is read
    int dev = 0, sms = 0;
    if (!current_device(&dev, &sms)) return XSYMV_ERR_DEVICE;
    Plan p = plan_make(n, 32, upper, 1);
    timing_begin(st);
    timing_mid(st);
    cudaError_t e = launch_finalize<T>(p, nullptr, nullptr, nullptr, alpha, beta,
                                       bz ? kZero : kAlphaZero, y0, incy, nullptr, 0, st);
    timing_end(st);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return XSYMV_ERR_CUDA;
    }
    note_launches(1);
    note_call_status(st, nullptr, 0);
    return XSYMV_OK;
  }

  Workload<T> wl;
  int status = plan_call(table, count, kind, upper, n, &wl);
  if (status) return status;
  // back-to-back calls (the stream's flag, see OverlapWords): a tuned
  // one-launch variant gives way to its two-kernel twin, whose calls fill
  // each other's tails.  The twin runs this very plan (its main kernel takes
  // any grid), so the partial sums, their order and the results are the same.
  int* report = nullptr;
  const volatile int* seen = overlap_flag(st, &report);   // null if unavailable
  if (wl.twin >= 0 && forced_variant(kind) < 0 && seen != nullptr && *seen == 1)
    wl.variant = &table[wl.twin];
  int epoch = 0;
  size_t cap = 0;
  // two sets of partial sums: calls of even number use the one after the
  // header, odd ones the one ending (256-byte aligned) at the end of the
  // buffer, so a call's main kernel never writes what the previous call's
  // finaliser may still read, whatever the two calls' sizes (the buffer
  // holds both calls' two sets and 256 bytes more)
  const long long set = wl.bytes - kHeaderBytes;
  char* ws = static_cast<char*>(workspace((size_t)(kHeaderBytes + 2 * set + 256), st, &status, 0,
                                          &epoch, &cap));
  if (!ws) return status;
  const long long odd_start = ((long long)cap - set) / 256 * 256;
  char* sb = ws + ((epoch & 1) ? odd_start - kHeaderBytes : 0);   // this call's set (offsets
                                                                  // wc_off.. count the header)
  MainArgs<T> m{wl.plan, A, lda, x0, incx, reinterpret_cast<T*>(sb + wl.wc_off),
                reinterpret_cast<T*>(sb + wl.wr_off), reinterpret_cast<int*>(ws), epoch,
                (reinterpret_cast<uintptr_t>(A) % 16 == 0) &&
                    (((long long)lda * (long long)sizeof(T)) % 16 == 0),
                st};
  status = ensure_tables(wl.plan, st, &m.wt, &m.rt);
  if (status) return status;
  // overlap bookkeeping in the header: end times of the calls' last kernels
  // and main-kernel start times, one word each per call parity
  unsigned long long* hw = reinterpret_cast<unsigned long long*>(ws + kOverlapOffset);
  const int q = epoch & 1;
  if (wl.variant->accum == kAccumFused) {
    // one launch: the kernel also applies y = alpha*s + beta*y
    m.ow = OverlapWords{hw + q, nullptr, hw + (1 - q), report};
    m.alpha = alpha;
    m.beta = beta;
    m.mode = bz ? kBetaZero : kFull;
    m.y0 = y0;
    m.incy = incy;
    timing_begin(st);
    cudaError_t e = wl.variant->launch(m);
    timing_mid(st);
    timing_end(st);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return XSYMV_ERR_CUDA;
    }
    note_launches(1);
    note_call_status(st, m.status, epoch);
    return XSYMV_OK;
  }
  if (wl.variant->accum == kAccumTickets) {
    // one launch: the kernel also applies y = alpha*s + beta*y
    const long long tk_bytes = kTkHeaderBytes + (long long)wl.plan.nb * kTkStride * 8;
    m.tk = ticket_buffer((size_t)tk_bytes, st, &status, &m.call);
    if (!m.tk) return status;
    m.v = reinterpret_cast<T*>(sb + wl.v_off);
    m.alpha = alpha;
    m.beta = beta;
    m.mode = bz ? kBetaZero : kFull;
    m.y0 = y0;
    m.incy = incy;
    timing_begin(st);
    cudaError_t e = wl.variant->launch(m);
    timing_mid(st);
    timing_end(st);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return XSYMV_ERR_CUDA;
    }
    note_launches(1);
    note_call_status(st, m.status, epoch);
    return XSYMV_OK;
  }
  // the bytes this call reads (A, x) and its finaliser writes (y)
  const uintptr_t es = sizeof(T);
  const uintptr_t a_lo = reinterpret_cast<uintptr_t>(A);
  const uintptr_t a_hi = a_lo + ((uintptr_t)(n - 1) * (uintptr_t)lda + (uintptr_t)n) * es;
  const uintptr_t x_lo = reinterpret_cast<uintptr_t>(x);
  const uintptr_t x_hi = x_lo + ((uintptr_t)(n - 1) * (uintptr_t)(incx < 0 ? -incx : incx) + 1) * es;
  const uintptr_t y_lo = reinterpret_cast<uintptr_t>(y);
  const uintptr_t y_hi = y_lo + ((uintptr_t)(n - 1) * (uintptr_t)(incy < 0 ? -incy : incy) + 1) * es;
  m.early = may_start_early(st, a_lo, a_hi, x_lo, x_hi) ? 1 : 0;
  OverlapWords ow{hw + q, hw + 2 + q, hw + (1 - q), m.early ? report : nullptr};
  const bool compact = m.early && seen != nullptr && *seen == 1;
  timing_begin(st);
  cudaError_t e = wl.variant->launch(m);
  if (e == cudaSuccess) {
    timing_mid(st);
    e = launch_finalize<T>(wl.plan, m.Wc, m.Wr, m.rt, alpha, beta, bz ? kBetaZero : kFull, y0,
                           incy, m.status, epoch, st, compact, ow);
  }
  timing_end(st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  note_launches(2);
  note_call_status(st, m.status, epoch, y_lo, y_hi);
  return XSYMV_OK;
}

// -------------------------------------------------- host-buffer variant --
// device-side address of p when the GPU can read it in place: page-locked
// (pinned or registered) host memory, managed or device memory; nullptr for
// ordinary pageable memory
inline const void* device_view(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged ||
      at.type == cudaMemoryTypeDevice)
    return at.devicePointer;
  return nullptr;
}

// With page-locked host buffers the kernels read A and x and write y in
// place over the host link (zero-copy).  Otherwise the stored triangle (in
// column panels), x and, when beta != 0, y are copied to library-owned device
// memory on the call's stream, the kernels run there and y is copied back.
// Either way the call waits for the stream.
template <class T>
int symv_host_entry(const Variant<T>* table, int count, char kind, char uplo, int n, T alpha,
                    const T* hA, int lda, const T* hx, int incx, T beta, T* hy, int incy) {
  int info = check_args(uplo, n, lda, incx, incy);
  if (info) return info;
  note_host_traffic(0, 0);
  if (n == 0) return XSYMV_OK;
  const bool az = is_zero(alpha), bz = is_zero(beta);
  if (az && is_one(beta)) return XSYMV_OK;
  int dev = 0, sms = 0;
  if (!current_device(&dev, &sms)) return XSYMV_ERR_DEVICE;

  const int upper = (uplo == 'U' || uplo == 'u');
  const long long es = (long long)sizeof(T);

  const void* vA = device_view(hA);
  const void* vx = device_view(hx);
  const void* vy = device_view(hy);
  if (vA && vx && vy) {
    int status = symv_entry<T>(table, count, kind, uplo, n, alpha, static_cast<const T*>(vA), lda,
                               static_cast<const T*>(vx), incx, beta,
                               const_cast<T*>(static_cast<const T*>(vy)), incy);
    if (status) return status;
    cudaError_t e = cudaStreamSynchronize(current_stream());
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return XSYMV_ERR_CUDA;
    }
    const long long tri = az ? 0 : ((long long)n * (n + 1) / 2 + n) * es;
    note_host_traffic(tri + (bz ? 0 : (long long)n * es), (long long)n * es);
    return XSYMV_OK;
  }

  const long long per16 = 16 / es > 0 ? 16 / es : 1;
  const long long ldd = align_up(n, per16);          // 16-byte aligned columns
  const long long a_bytes = align_up(ldd * n * es, 256);
  const long long v_bytes = align_up((long long)n * es, 256);
  cudaStream_t st = current_stream();
  int status = XSYMV_OK;
  char* buf = static_cast<char*>(workspace((size_t)(a_bytes + 2 * v_bytes), st, &status, 1, nullptr));
  if (!buf) return status;
  T* dA = reinterpret_cast<T*>(buf);
  T* dx = reinterpret_cast<T*>(buf + a_bytes);
  T* dy = reinterpret_cast<T*>(buf + a_bytes + v_bytes);

  long long h2d = 0, d2h = 0;
  cudaError_t e = cudaSuccess;
  // strided vector -> contiguous device copy in memory order; a negative
  // stride keeps its sign (stride -1 on the device)
  auto vec_in = [&](const T* h, int inc, T* d) {
    const long long ai = inc < 0 ? -(long long)inc : inc;
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(d, es, h, ai * es, es, n, cudaMemcpyDefault, st);
    h2d += (long long)n * es;
  };
  if (!az) {
    // the triangle in panels of P columns: upper rows [0, j1), lower [j0, n)
    const long long P = align_up((n + 63) / 64, 64);   // at most 64 panels
    for (long long j0 = 0; j0 < n && e == cudaSuccess; j0 += P) {
      const long long j1 = j0 + P < n ? j0 + P : n;
      const long long r0 = upper ? 0 : j0;
      const long long r1 = upper ? j1 : n;
      e = cudaMemcpy2DAsync(dA + j0 * ldd + r0, ldd * es, hA + j0 * (long long)lda + r0,
                            (long long)lda * es, (r1 - r0) * es, j1 - j0, cudaMemcpyDefault, st);
      h2d += (r1 - r0) * es * (j1 - j0);
    }
    vec_in(hx, incx, dx);
  }
  if (!bz) vec_in(hy, incy, dy);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  status = symv_entry<T>(table, count, kind, uplo, n, alpha, dA, (int)ldd, dx, incx < 0 ? -1 : 1,
                         beta, dy, incy < 0 ? -1 : 1);
  if (status) return status;
  const long long ai = incy < 0 ? -(long long)incy : incy;
  e = cudaMemcpy2DAsync(hy, ai * es, dy, es, es, n, cudaMemcpyDefault, st);
  d2h += (long long)n * es;
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  note_host_traffic(h2d, d2h);
  return XSYMV_OK;
}

// ------------------------------------------------------ sharded product --
// One shard of y := alpha*A*x + beta*y split by block columns: the stored
// columns c0 <= j < c1 of A (the shard's panel, in its own array), streamed
// by the same main kernel restricted to that column window; the finaliser
// writes the panel's partial vector s (n elements, contiguous: row terms of
// the panel's elements and column terms of its columns) without alpha or
// beta.  symv_reduce_entry then adds the shards' vectors in rank order.
//
// Panel layout: element (i, j) (matrix indices, i in the stored part of
// column j) at A[(i - r0) + (j - c0) * lda], r0 = 0 for upper storage (the
// panel holds rows 0 .. c1-1) and r0 = c0 for lower (rows c0 .. n-1).
inline int check_shard_args(char uplo, int n, int c0, int c1, int lda, int incx) {
  if (uplo != 'U' && uplo != 'u' && uplo != 'L' && uplo != 'l') return 1;
  if (n < 0) return 2;
  if (c0 < 0 || c0 > n) return 3;
  if (c1 < c0 || c1 > n) return 4;
  const int rows = (uplo == 'U' || uplo == 'u') ? c1 : n - c0;
  if (lda < (rows > 1 ? rows : 1)) return 6;
  if (incx == 0) return 8;
  return 0;
}

template <class T>
int symv_shard_entry(const Variant<T>* table, int count, char kind, char uplo, int n, int c0,
                     int c1, const T* A, int lda, const T* x, int incx, T* partial) {
  int info = check_shard_args(uplo, n, c0, c1, lda, incx);
  if (info) return info;
  if (n == 0) return XSYMV_OK;
  const int upper = (uplo == 'U' || uplo == 'u');
  cudaStream_t st = current_stream();
  const T unused = T{};   // alpha and beta: the partial and zero modes read neither
  if (c0 == c1) {  // an empty panel: its partial vector is zero
    int dev = 0, sms = 0;
    if (!current_device(&dev, &sms)) return XSYMV_ERR_DEVICE;
    Plan p = plan_make(n, 32, upper, 1);
    cudaError_t e = launch_finalize<T>(p, nullptr, nullptr, nullptr, unused, unused, kZero,
                                       partial, 1, nullptr, 0, st);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return XSYMV_ERR_CUDA;
    }
    note_launches(1);
    note_call_status(st, nullptr, 0);
    return XSYMV_OK;
  }
  const T* x0 = x + (incx < 0 ? (long long)(1 - n) * incx : 0);
  // the variant tuned for a whole triangle with as many stored elements
  const long long elems =
      upper ? ((long long)c1 * (c1 + 1) - (long long)c0 * (c0 + 1)) / 2
            : (long long)(c1 - c0) * n - ((long long)c1 * (c1 - 1) - (long long)c0 * (c0 - 1)) / 2;
  long long n_pick = (long long)((sqrt(8.0 * (double)elems + 1.0) - 1.0) / 2.0);
  while (n_pick * (n_pick + 1) / 2 < elems) ++n_pick;
  while (n_pick > 1 && (n_pick - 1) * n_pick / 2 >= elems) --n_pick;
  Workload<T> wl;
  int status = plan_call(table, count, kind, upper, n, &wl, c0, c1, (int)n_pick);
  if (status) return status;
  if (wl.variant->accum == kAccumTickets) return XSYMV_ERR_VALUE;   // no ticket shards
  int epoch = 0;
  char* ws = static_cast<char*>(workspace((size_t)wl.bytes, st, &status, 0, &epoch));
  if (!ws) return status;
  // the kernels address A(i, j) at A_k + i + j*lda (matrix indices)
  const long long r0 = upper ? 0 : c0;
  const uintptr_t a_addr = reinterpret_cast<uintptr_t>(A) -
                           (uintptr_t)((r0 + (long long)c0 * lda) * (long long)sizeof(T));
  const T* Ak = reinterpret_cast<const T*>(a_addr);
  // 16-byte vectors only when every vector a column's stored rows need lies
  // inside the panel: the window's edges on the 16-byte grid too
  const bool aligned = a_addr % 16 == 0 && ((long long)lda * (long long)sizeof(T)) % 16 == 0 &&
                       ((long long)c0 * (long long)sizeof(T)) % 16 == 0 &&
                       (c1 == n || ((long long)c1 * (long long)sizeof(T)) % 16 == 0);
  MainArgs<T> m{wl.plan, Ak, lda, x0, incx, reinterpret_cast<T*>(ws + wl.wc_off),
                reinterpret_cast<T*>(ws + wl.wr_off), reinterpret_cast<int*>(ws), epoch, aligned,
                st};
  status = ensure_tables(wl.plan, st, &m.wt, &m.rt);
  if (status) return status;
  const bool fused = wl.variant->accum == kAccumFused;
  if (fused) {   // the partial vector in the same launch
    m.alpha = unused;
    m.beta = unused;
    m.mode = kPartial;
    m.y0 = partial;
    m.incy = 1;
  }
  timing_begin(st);
  cudaError_t e = wl.variant->launch(m);
  if (e == cudaSuccess) {
    timing_mid(st);
    if (!fused)
      e = launch_finalize<T>(wl.plan, m.Wc, m.Wr, m.rt, unused, unused, kPartial, partial, 1,
                             m.status, epoch, st);
  }
  timing_end(st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  note_launches(fused ? 1 : 2);
  note_call_status(st, m.status, epoch);
  return XSYMV_OK;
}

// y := alpha * (P_0 + ... + P_{N-1}) + beta * y, the parts added in rank
// order (P_r at P + r*ldp, n contiguous elements each).
template <class T>
int symv_reduce_entry(int n, int nparts, T alpha, const T* P, long long ldp, T beta, T* y,
                      int incy) {
  if (n < 0) return 1;
  if (nparts < 1) return 2;
  if (ldp < (n > 1 ? n : 1)) return 5;
  if (incy == 0) return 8;
  if (n == 0) return XSYMV_OK;
  const bool az = is_zero(alpha), bz = is_zero(beta);
  if (az && is_one(beta)) return XSYMV_OK;
  cudaStream_t st = current_stream();
  T* y0 = y + (incy < 0 ? (long long)(1 - n) * incy : 0);
  const int mode = az ? (bz ? kZero : kAlphaZero) : (bz ? kBetaZero : kFull);
  symv_reduce<T><<<(unsigned)((n + kReduceThreads - 1) / kReduceThreads), kReduceThreads, 0, st>>>(
      n, nparts, P, ldp, alpha, beta, mode, y0, incy);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  note_launches(1);
  note_call_status(st, nullptr, 0);
  return XSYMV_OK;
}

template <class T>
long long workspace_bytes(const Variant<T>* table, int count, char kind, char uplo, int n) {
  if (check_args(uplo, n, n > 1 ? n : 1, 1, 1)) return XSYMV_ERR_VALUE;
  if (n == 0) return 0;
  Workload<T> wl;
  int status = plan_call(table, count, kind, uplo == 'U' || uplo == 'u', n, &wl);
  return status ? status : wl.bytes;
}

}  // namespace xsymv

// The sharded product's two C entry points of one kind (see include/xsymv.h):
// SHARD(uplo, n, col_begin, col_end, A, lda, x, incx, partial) and
// REDUCE(n, nparts, alpha, partials, ldp, beta, y, incy).
#define XSYMV_DEFINE_SHARDS(SHARD, REDUCE, KIND, CT, T, TABLE)                                \
  extern "C" XSYMV_API int SHARD(char uplo, int n, int col_begin, int col_end, const CT* A,   \
                                 int lda, const CT* x, int incx, CT* partial) {               \
    static_assert(sizeof(CT) == sizeof(T), "C-ABI type layout");                              \
    return xsymv::symv_shard_entry<T>(TABLE, (int)(sizeof(TABLE) / sizeof(TABLE[0])), KIND,   \
                                      uplo, n, col_begin, col_end,                            \
                                      reinterpret_cast<const T*>(A), lda,                     \
                                      reinterpret_cast<const T*>(x), incx,                    \
                                      reinterpret_cast<T*>(partial));                         \
  }                                                                                           \
  extern "C" XSYMV_API int REDUCE(int n, int nparts, CT alpha, const CT* partials,            \
                                  long long ldp, CT beta, CT* y, int incy) {                  \
    T a, b;                                                                                   \
    memcpy(&a, &alpha, sizeof(T));                                                            \
    memcpy(&b, &beta, sizeof(T));                                                             \
    return xsymv::symv_reduce_entry<T>(n, nparts, a, reinterpret_cast<const T*>(partials),    \
                                       ldp, b, reinterpret_cast<T*>(y), incy);                \
  }

// Per-kind tables and introspection functions (defined in each xsymv_<k>.cu).
#define XSYMV_DEFINE_INTROSPECTION(KIND, T, TABLE)                                          \
  namespace xsymv {                                                                         \
  int variant_count_##KIND() { return (int)(sizeof(TABLE) / sizeof(TABLE[0])); }            \
  const char* variant_name_##KIND(int i) {                                                  \
    return (i >= 0 && i < variant_count_##KIND()) ? TABLE[i].name : nullptr;                \
  }                                                                                         \
  int selected_variant_##KIND(char uplo, int n) {                                           \
    return pick_variant<T>(TABLE, variant_count_##KIND(), #KIND[0], uplo == 'U' || uplo == 'u', n); \
  }                                                                                         \
  long long workspace_bytes_##KIND(char uplo, int n) {                                      \
    return workspace_bytes<T>(TABLE, variant_count_##KIND(), #KIND[0], uplo, n);            \
  }                                                                                         \
  }
