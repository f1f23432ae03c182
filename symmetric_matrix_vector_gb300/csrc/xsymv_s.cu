// Entry point xsymv_s of the xsymv C ABI and its compiled kernel variants.
#include <mutex>
#include <vector>

#include "xsymv_entry.cuh"

namespace xsymv {
static const Variant<float> kVariants_s[] = {
    XSYMV_REG(float, 1, 4, 8),
    XSYMV_REG(float, 1, 2, 8),
    XSYMV_REG(float, 1, 8, 8),
    XSYMV_REG(float, 1, 4, 4),
    XSYMV_REG(float, 2, 2, 8),
    XSYMV_REG_MB(float, 1, 4, 8, 5),
    XSYMV_REG_MB(float, 1, 2, 8, 5),
    XSYMV_REG_MB(float, 1, 2, 8, 6),
    XSYMV_TMA(float, 1, 8, 3, 8),
    XSYMV_REG_MBX(float, 1, 2, 8, 6, 4),
    XSYMV_REG_G(float, 1, 2, 8, 6, 5),
    XSYMV_REG_G(float, 1, 2, 8, 6, 7),
    XSYMV_REG_G(float, 1, 2, 8, 6, 9),
    XSYMV_REG_G(float, 1, 2, 8, 6, 11),
    XSYMV_REG_G(float, 1, 2, 8, 0, 9),
    XSYMV_REG_G(float, 1, 2, 8, 6, 14),
    XSYMV_TICKET(float, 1, 2, 8, 6, 9, 2),
    XSYMV_TICKET(float, 1, 2, 8, 0, 9, 2),
    XSYMV_TICKET(float, 2, 2, 8, 0, 6, 2),
    XSYMV_TICKET(float, 2, 2, 8, 4, 6, 2),
    XSYMV_REG_G(float, 2, 2, 8, 4, 9),
    XSYMV_REG_G(float, 2, 2, 8, 4, 11),
    XSYMV_REG_G(float, 2, 2, 8, 4, 13),
    XSYMV_REG_G(float, 2, 1, 8, 5, 6),
    XSYMV_REG_G(float, 2, 2, 8, 4, 7),
    XSYMV_REG_G(float, 2, 2, 8, 4, 8),
    XSYMV_REG_G(float, 2, 2, 8, 4, 12),
    XSYMV_FUSED(float, 1, 2, 8, 6, 11, 2),
    XSYMV_FUSED(float, 2, 2, 8, 4, 12, 2),
    XSYMV_FUSED(float, 2, 2, 8, 4, 11, 2),
    XSYMV_FUSED(float, 1, 2, 8, 6, 7, 2),
    XSYMV_FUSED(float, 2, 2, 8, 4, 13, 2),
    XSYMV_FUSED(float, 2, 2, 8, 4, 9, 2),
    XSYMV_FUSED(float, 1, 2, 8, 6, 9, 2),
    XSYMV_FUSED(float, 1, 2, 8, 6, 14, 2),
};
static_assert(sizeof(float) == sizeof(float), "C-ABI type layout");
}  // namespace xsymv

XSYMV_DEFINE_INTROSPECTION(s, float, kVariants_s)
XSYMV_DEFINE_SHARDS(xsymv_s_shard, xsymv_s_reduce, 's', float, float, xsymv::kVariants_s)

extern "C" XSYMV_API int xsymv_s(char uplo, int n, float alpha, const float* A, int lda, const float* x,
                                int incx, float beta, float* y, int incy) {
  using T = float;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_entry<T>(xsymv::kVariants_s,
                              (int)(sizeof(xsymv::kVariants_s) / sizeof(xsymv::kVariants_s[0])),
                              's', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                              reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                              incy);
}

extern "C" XSYMV_API int xsymv_s_host(char uplo, int n, float alpha, const float* A, int lda, const float* x,
                                   int incx, float beta, float* y, int incy) {
  using T = float;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_host_entry<T>(xsymv::kVariants_s,
                                   (int)(sizeof(xsymv::kVariants_s) / sizeof(xsymv::kVariants_s[0])),
                                   's', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                                   reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                                   incy);
}

// ---------------------------------------------------------------------------
// xsymv_s_noalloc: SSYMV that never allocates device memory.
//
// Some callers cannot let a library allocate device memory during a call:
// a plug-in whose host application owns all device memory and forbids
// allocations inside the plug-in, or latency-critical code where cudaMalloc /
// cudaFree would block or synchronise the device.  For them this entry point
// runs the same two kernels as xsymv_s, with the partial-sum workspace taken
// from the fixed device array below instead of a cudaMalloc'd buffer.
//
// * The array holds kNoallocScratchBytes (16 MiB) on every GPU that loads
//   this library, until the process exits.  Problems whose workspace does
//   not fit (roughly n > 31000 with the tuned kernels on GB300) are
//   rejected with XSYMV_ERR_TOO_LARGE before anything is enqueued.
// * The first call on a device that needs the array (alpha != 0) looks up
//   its device address (cudaGetSymbolAddress, with that device current) and
//   caches it; make that first call before any stream capture.
// * Only the array's first 256 bytes (a status word the kernels set if a
//   bounded wait runs out) must start at zero; that first call clears them
//   with cudaMemsetAsync on its stream.  Every other workspace slot the
//   finaliser reads is written by the main kernel of the same call.  The
//   array keeps the last call's contents, among them the plan's warp and
//   row tables: a call rebuilds them (one extra small launch) only when its
//   plan differs from the previous call's on the device.
// * All calls share the one array: calls that overlap on the GPU (on
//   different streams, or from different host threads) race and corrupt
//   each other's results.  Order them: each call must start on the GPU only
//   after everything the previous call enqueued has finished (one stream
//   does that; with several, an event recorded after the previous call).
static constexpr long long kNoallocScratchBytes = 16ll << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {
struct NoallocDevice {
  int device;
  void* scratch;
  int epoch;   // last call number on this device
  xsymv::TablesKey tables;   // the plan whose tables the array holds (n = -1: none)
};
std::mutex g_noalloc_mu;
std::vector<NoallocDevice> g_noalloc_devices;

// device address of g_noalloc_scratch on the current device and a fresh call
// number; the first call on a device clears the status header on `stream`.
// *dev_index: the device's entry (for the tables record).
int noalloc_scratch(void** out, int* epoch, cudaStream_t stream, size_t* dev_index) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) {
    xsymv::record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  for (size_t i = 0; i < g_noalloc_devices.size(); ++i) {
    NoallocDevice& s = g_noalloc_devices[i];
    if (s.device == d) {
      if (s.epoch >= 0x7ffffffe) {
        // call numbers start again at 1: clear the status word first (see
        // the workspace's call numbers)
        e = cudaMemsetAsync(s.scratch, 0, 256, stream);
        if (e != cudaSuccess) {
          xsymv::record_cuda_error(e);
          return XSYMV_ERR_CUDA;
        }
        s.epoch = 0;
      }
      ++s.epoch;
      *out = s.scratch;
      *epoch = s.epoch;
      *dev_index = i;
      return XSYMV_OK;
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e == cudaSuccess && p != nullptr) e = cudaMemsetAsync(p, 0, 256, stream);
  if (e != cudaSuccess || p == nullptr) {
    xsymv::record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  g_noalloc_devices.push_back(NoallocDevice{d, p, 1, xsymv::TablesKey{-1, 0, 0, 0, 0, 0, 0, 0, 0}});
  *out = p;
  *epoch = 1;
  *dev_index = g_noalloc_devices.size() - 1;
  return XSYMV_OK;
}
}  // namespace

namespace xsymv {
// test hook (xsymv_test_set_call_number): the last call number handed out on
// the current device
bool noalloc_set_call_number(int number) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  for (NoallocDevice& s : g_noalloc_devices)
    if (s.device == d) {
      s.epoch = number;
      return true;
    }
  return false;
}
}  // namespace xsymv

extern "C" XSYMV_API int xsymv_s_noalloc(char uplo, int n, float alpha, const float* A, int lda,
                                         const float* x, int incx, float beta, float* y,
                                         int incy) {
  using namespace xsymv;
  int info = check_args(uplo, n, lda, incx, incy);
  if (info) return info;
  if (n == 0) return XSYMV_OK;
  const bool az = alpha == 0.f, bz = beta == 0.f;
  if (az && beta == 1.f) return XSYMV_OK;

  const int upper = (uplo == 'U' || uplo == 'u');
  cudaStream_t st = current_stream();
  float* y0 = y + (incy < 0 ? (long long)(1 - n) * incy : 0);
  const float* x0 = x + (incx < 0 ? (long long)(1 - n) * incx : 0);

  if (az) {  // y := beta*y, no workspace needed
    Plan p = plan_make(n, 32, upper, 1);
    cudaError_t e = launch_finalize<float>(p, nullptr, nullptr, nullptr, alpha, beta,
                                           bz ? kZero : kAlphaZero, y0, incy, nullptr, 0, st);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return XSYMV_ERR_CUDA;
    }
    note_launches(1);
    note_call_status(st, nullptr, 0);
    return XSYMV_OK;
  }

  // plan and size check first: a refused call enqueues nothing
  const int count = (int)(sizeof(kVariants_s) / sizeof(kVariants_s[0]));
  Workload<float> wl;
  int status = plan_call<float>(kVariants_s, count, 's', upper, n, &wl);
  if (status) return status;
  // the ordered-ticket kernels keep state in a second, allocated buffer
  if (wl.variant->accum == kAccumTickets) return XSYMV_ERR_VALUE;
  // the plan's tables follow the workspace in the same array
  const long long tab_off = align_up(wl.bytes, 256);
  if (tab_off + tables_bytes(wl.plan) > kNoallocScratchBytes) return XSYMV_ERR_TOO_LARGE;

  void* scratch = nullptr;
  int epoch = 0;
  size_t dev_index = 0;
  status = noalloc_scratch(&scratch, &epoch, st, &dev_index);
  if (status) return status;
  char* ws = static_cast<char*>(scratch);
  MainArgs<float> m{wl.plan, A, lda, x0, incx, reinterpret_cast<float*>(ws + wl.wc_off),
                    reinterpret_cast<float*>(ws + wl.wr_off), reinterpret_cast<int*>(ws), epoch,
                    (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (((long long)lda * 4) % 16 == 0),
                    st};
  m.wt = reinterpret_cast<const int4*>(ws + tab_off);
  m.rt = reinterpret_cast<const int2*>(ws + tab_off + ((long long)wl.plan.W * 16 + 255) / 256 * 256);
  const bool fused = wl.variant->accum == kAccumFused;
  if (fused) {   // one launch: the kernel also applies y = alpha*s + beta*y
    m.alpha = alpha;
    m.beta = beta;
    m.mode = bz ? kBetaZero : kFull;
    m.y0 = y0;
    m.incy = incy;
  }
  int launches = fused ? 1 : 2;
  cudaError_t e = cudaSuccess;
  {
    const TablesKey key = tables_key(wl.plan);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    TablesKey& have = g_noalloc_devices[dev_index].tables;
    if (memcmp(&have, &key, sizeof(key)) != 0) {
      e = launch_plan_tables(wl.plan, ws + tab_off, st);
      have = e == cudaSuccess ? key : TablesKey{-1, 0, 0, 0, 0, 0, 0, 0, 0};
      ++launches;
    }
  }
  if (e == cudaSuccess) e = wl.variant->launch(m);
  if (e == cudaSuccess && !fused)
    e = launch_finalize<float>(wl.plan, m.Wc, m.Wr, m.rt, alpha, beta, bz ? kBetaZero : kFull, y0,
                               incy, m.status, epoch, st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  note_launches(launches);
  note_call_status(st, m.status, epoch);
  return XSYMV_OK;
}
