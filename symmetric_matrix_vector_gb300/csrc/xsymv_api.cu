// Host runtime of the xsymv library: stream selection, workspace cache,
// launch counter, event timing, status strings and variant overrides.
// The five compute entry points live in xsymv_{s,d,c,z,w}.cu.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/xsymv.h"
#include "xsymv_runtime.h"

namespace xsymv {

// Shard boundaries are multiples of this many columns (except n), so that
// every kind's panels keep the 16-byte grid of the whole matrix.
constexpr long long kShardAlign = 16;

namespace {

std::atomic<cudaStream_t> g_stream{nullptr};
std::atomic<long long> g_launches{0};
std::atomic<int> g_last_error{0};

std::mutex g_mu;

struct WsEntry {
  int device;
  cudaStream_t stream;
  int slot;
  void* ptr;
  size_t bytes;
  int epoch;     // last call number handed out (slot 0)
};
std::vector<WsEntry> g_ws;

struct DevInfo {
  int device;
  int sms;
};
std::vector<DevInfo> g_dev;

struct TimedCall {
  cudaEvent_t ev[3];
};
bool g_timing = false;
std::atomic<bool> g_timing_on{false};   // g_timing, readable without the lock
std::vector<TimedCall> g_timed;      // calls recorded since the last read
TimedCall g_cur{};                   // call being recorded
std::vector<cudaEvent_t> g_free_ev;  // event pool

int g_forced[5] = {-1, -1, -1, -1, -1};

int kind_index(char k) {
  switch (k) {
    case 's': case 'S': return 0;
    case 'd': case 'D': return 1;
    case 'c': case 'C': return 2;
    case 'z': case 'Z': return 3;
    case 'w': case 'W': return 4;
  }
  return -1;
}

cudaEvent_t take_event() {
  if (!g_free_ev.empty()) {
    cudaEvent_t e = g_free_ev.back();
    g_free_ev.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

cudaStream_t current_stream() { return g_stream.load(); }

int current_device_index() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return (d >= 0 && d < kMaxDevices) ? d : -1;
}

void record_cuda_error(cudaError_t e) {
  if (e != cudaSuccess) g_last_error.store((int)e);
}

bool current_device(int* dev, int* sm_count) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return false;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  for (const DevInfo& di : g_dev)
    if (di.device == d) {
      *dev = d;
      *sm_count = di.sms;
      return true;
    }
  int major = 0, minor = 0, sms = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d)) != cudaSuccess) {
    record_cuda_error(e);
    return false;
  }
  if (major != 10 || minor != 3) return false;  // built for sm_103a only
  g_dev.push_back(DevInfo{d, sms});
  *dev = d;
  *sm_count = sms;
  return true;
}

std::atomic<long long> g_h2d{0}, g_d2h{0};
std::atomic<unsigned long long> g_wait_limit{2000000000ull};
std::atomic<uint32_t> g_extra_tx{0};

void* workspace(size_t bytes, cudaStream_t stream, int* status, int slot, int* epoch,
                size_t* capacity) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    *status = XSYMV_ERR_CUDA;
    return nullptr;
  }
  if (bytes < 256) bytes = 256;
  std::lock_guard<std::mutex> lk(g_mu);
  WsEntry* w = nullptr;
  for (WsEntry& c : g_ws)
    if (c.device == d && c.stream == stream && c.slot == slot) w = &c;
  if (w == nullptr) {
    g_ws.push_back(WsEntry{d, stream, slot, nullptr, 0, 0});
    w = &g_ws.back();
  }
  if (w->bytes < bytes) {
    if (w->ptr != nullptr) {
      // the old buffer may still be in use by work queued on `stream`
      e = cudaStreamSynchronize(stream);
      if (e == cudaSuccess) e = cudaFree(w->ptr);
      w->ptr = nullptr;
      w->bytes = 0;
      if (e != cudaSuccess) {
        record_cuda_error(e);
        *status = XSYMV_ERR_CUDA;
        return nullptr;
      }
      bytes += bytes / 8;
    }
    e = cudaMalloc(&w->ptr, bytes);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      cudaGetLastError();
      w->ptr = nullptr;
      *status = XSYMV_ERR_ALLOC;
      return nullptr;
    }
    w->bytes = bytes;
    if (slot == 0) {
      e = cudaMemsetAsync(w->ptr, 0, 256, stream);   // status header
      if (e != cudaSuccess) {
        record_cuda_error(e);
        *status = XSYMV_ERR_CUDA;
        return nullptr;
      }
      w->epoch = 0;
    }
  }
  if (epoch != nullptr) {
    if (w->epoch >= 0x7ffffffe) {
      // call numbers start again at 1: clear the status word first (on the
      // stream, before this call's kernels), or a failure recorded under a
      // larger old number would hide the failures of the next calls
      e = cudaMemsetAsync(w->ptr, 0, 256, stream);
      if (e != cudaSuccess) {
        record_cuda_error(e);
        *status = XSYMV_ERR_CUDA;
        return nullptr;
      }
      w->epoch = 0;
    }
    *epoch = ++w->epoch;
  }
  if (capacity != nullptr) *capacity = w->bytes;
  return w->ptr;
}

namespace {
struct CallStatus {
  int device;
  cudaStream_t stream;
  const int* status;   // nullptr: the latest call has no status word
  int epoch;
  uintptr_t y_lo, y_hi;   // bytes its finaliser writes (empty: it did not end with one)
};
std::vector<CallStatus> g_call_status;
}  // namespace

void note_call_status(cudaStream_t stream, const int* status, int epoch, uintptr_t y_lo,
                      uintptr_t y_hi) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  for (CallStatus& c : g_call_status)
    if (c.device == d && c.stream == stream) {
      c.status = status;
      c.epoch = epoch;
      c.y_lo = y_lo;
      c.y_hi = y_hi;
      return;
    }
  g_call_status.push_back(CallStatus{d, stream, status, epoch, y_lo, y_hi});
}

namespace {
struct OverlapFlag {
  int device;
  cudaStream_t stream;
  int* host;   // page-locked, mapped
  int* dev;
};
std::vector<OverlapFlag> g_overlap;
}  // namespace

const volatile int* overlap_flag(cudaStream_t stream, int** dev) {
  *dev = nullptr;
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  for (const OverlapFlag& f : g_overlap)
    if (f.device == d && f.stream == stream) {
      *dev = f.dev;
      return f.host;
    }
  void* h = nullptr;
  void* dp = nullptr;
  if (cudaHostAlloc(&h, sizeof(int), cudaHostAllocMapped) != cudaSuccess ||
      cudaHostGetDevicePointer(&dp, h, 0) != cudaSuccess) {
    cudaGetLastError();
    if (h != nullptr) cudaFreeHost(h);
    g_overlap.push_back(OverlapFlag{d, stream, nullptr, nullptr});   // do not try again
    return nullptr;
  }
  *static_cast<int*>(h) = 0;
  g_overlap.push_back(OverlapFlag{d, stream, static_cast<int*>(h), static_cast<int*>(dp)});
  *dev = static_cast<int*>(dp);
  return static_cast<int*>(h);
}

bool may_start_early(cudaStream_t stream, uintptr_t a_lo, uintptr_t a_hi, uintptr_t x_lo,
                     uintptr_t x_hi) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  for (const CallStatus& c : g_call_status)
    if (c.device == d && c.stream == stream) {
      if (c.y_lo >= c.y_hi) return false;
      const bool hits_a = a_lo < c.y_hi && c.y_lo < a_hi;
      const bool hits_x = x_lo < c.y_hi && c.y_lo < x_hi;
      return !hits_a && !hits_x;
    }
  return false;
}

namespace {
struct TkEntry {
  int device;
  cudaStream_t stream;
  void* ptr;
  size_t bytes;
  unsigned long long call;   // last call number handed out
};
std::vector<TkEntry> g_tk;
}  // namespace

void* ticket_buffer(size_t bytes, cudaStream_t stream, int* status, unsigned long long* call) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    *status = XSYMV_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  TkEntry* t = nullptr;
  for (TkEntry& c : g_tk)
    if (c.device == d && c.stream == stream) t = &c;
  if (t == nullptr) {
    g_tk.push_back(TkEntry{d, stream, nullptr, 0, 0});
    t = &g_tk.back();
  }
  if (t->bytes < bytes) {
    if (t->ptr != nullptr) {
      // the old buffer may still be in use by work queued on `stream`
      e = cudaStreamSynchronize(stream);
      if (e == cudaSuccess) e = cudaFree(t->ptr);
      t->ptr = nullptr;
      t->bytes = 0;
      if (e != cudaSuccess) {
        record_cuda_error(e);
        *status = XSYMV_ERR_CUDA;
        return nullptr;
      }
    }
    e = cudaMalloc(&t->ptr, bytes);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      cudaGetLastError();
      t->ptr = nullptr;
      *status = XSYMV_ERR_ALLOC;
      return nullptr;
    }
    // zero counters, and tickets that name no call (call numbers start at 1)
    e = cudaMemsetAsync(t->ptr, 0, bytes, stream);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      *status = XSYMV_ERR_CUDA;
      return nullptr;
    }
    t->bytes = bytes;
  }
  *call = ++t->call;
  return t->ptr;
}

namespace {
struct TabEntry {
  int device;
  cudaStream_t stream;
  void* ptr;
  size_t bytes;
  std::vector<unsigned char> key;   // the plan whose tables the buffer holds (empty: none)
};
std::vector<TabEntry> g_tab;

TabEntry* tab_entry(int d, cudaStream_t stream) {
  for (TabEntry& t : g_tab)
    if (t.device == d && t.stream == stream) return &t;
  return nullptr;
}
}  // namespace

void* plan_tables(size_t bytes, cudaStream_t stream, const void* key, size_t key_bytes,
                  bool* ready, int* status) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    *status = XSYMV_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  TabEntry* t = tab_entry(d, stream);
  if (t == nullptr) {
    g_tab.push_back(TabEntry{d, stream, nullptr, 0, {}});
    t = &g_tab.back();
  }
  if (t->bytes < bytes) {
    t->key.clear();
    if (t->ptr != nullptr) {
      // the old buffer may still be in use by work queued on `stream`
      e = cudaStreamSynchronize(stream);
      if (e == cudaSuccess) e = cudaFree(t->ptr);
      t->ptr = nullptr;
      t->bytes = 0;
      if (e != cudaSuccess) {
        record_cuda_error(e);
        *status = XSYMV_ERR_CUDA;
        return nullptr;
      }
      bytes += bytes / 8;
    }
    e = cudaMalloc(&t->ptr, bytes);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      cudaGetLastError();
      t->ptr = nullptr;
      *status = XSYMV_ERR_ALLOC;
      return nullptr;
    }
    t->bytes = bytes;
  }
  const unsigned char* k = static_cast<const unsigned char*>(key);
  *ready = t->key.size() == key_bytes && std::equal(t->key.begin(), t->key.end(), k);
  if (!*ready) t->key.assign(k, k + key_bytes);
  return t->ptr;
}

void plan_tables_forget(cudaStream_t stream) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (TabEntry* t = tab_entry(d, stream)) t->key.clear();
}

unsigned long long wait_limit_ns() { return g_wait_limit.load(); }
uint32_t test_extra_tx() { return g_extra_tx.load(); }

void note_launches(int k) { g_launches.fetch_add(k); }

void note_host_traffic(long long h2d, long long d2h) {
  g_h2d.store(h2d);
  g_d2h.store(d2h);
}

void timing_begin(cudaStream_t s) {
  if (!g_timing_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_timing) return;
  for (int i = 0; i < 3; ++i) g_cur.ev[i] = take_event();
  if (g_cur.ev[0]) cudaEventRecord(g_cur.ev[0], s);
}
void timing_mid(cudaStream_t s) {
  if (!g_timing_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_timing && g_cur.ev[1]) cudaEventRecord(g_cur.ev[1], s);
}
void timing_end(cudaStream_t s) {
  if (!g_timing_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_timing) return;
  if (g_cur.ev[2]) cudaEventRecord(g_cur.ev[2], s);
  if (g_cur.ev[0] && g_cur.ev[1] && g_cur.ev[2]) {
    g_timed.push_back(g_cur);
  } else {
    for (int i = 0; i < 3; ++i)
      if (g_cur.ev[i]) g_free_ev.push_back(g_cur.ev[i]);
  }
  g_cur = TimedCall{};
}

int forced_variant(char kind) {
  int k = kind_index(kind);
  return k < 0 ? -1 : g_forced[k];
}

}  // namespace xsymv

using namespace xsymv;

extern "C" {

XSYMV_API int xsymv_set_stream(void* stream) {
  g_stream.store(reinterpret_cast<cudaStream_t>(stream));
  return XSYMV_OK;
}

XSYMV_API void* xsymv_get_stream(void) { return reinterpret_cast<void*>(g_stream.load()); }

XSYMV_API const char* xsymv_status_string(int status) {
  switch (status) {
    case 0: return "success";
    case 1: return "invalid argument 1 (uplo): must be 'U', 'u', 'L' or 'l'";
    case 2: return "invalid argument 2 (n): must be >= 0";
    case 5: return "invalid argument 5 (lda): must be >= max(1, n)";
    case 7: return "invalid argument 7 (incx): must be non-zero";
    case 10: return "invalid argument 10 (incy): must be non-zero";
    case XSYMV_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case XSYMV_ERR_ALLOC: return "workspace allocation failed";
    case XSYMV_ERR_DEVICE: return "no usable device (compute capability 10.3 required)";
    case XSYMV_ERR_VALUE: return "invalid value";
    case XSYMV_ERR_TIMEOUT:
      return "a bounded wait in the main kernel ran out; the call's y was set to NaN";
    case XSYMV_ERR_TOO_LARGE:
      return "problem too large for xsymv_s_noalloc's fixed 16 MiB workspace (use xsymv_s)";
  }
  return "unknown status";
}

XSYMV_API int xsymv_last_cuda_error(void) { return g_last_error.load(); }

XSYMV_API int xsymv_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timing = on != 0;
  g_timing_on.store(g_timing);
  if (!g_timing) {
    for (TimedCall& t : g_timed)
      for (int i = 0; i < 3; ++i) g_free_ev.push_back(t.ev[i]);
    g_timed.clear();
  }
  return XSYMV_OK;
}

XSYMV_API int xsymv_timing_read(int* calls, double* main_ms, double* call_ms) {
  std::lock_guard<std::mutex> lk(g_mu);
  double m = 0.0, c = 0.0;
  int status = XSYMV_OK;
  for (TimedCall& t : g_timed) {
    cudaError_t e = cudaEventSynchronize(t.ev[2]);
    float a = 0.f, b = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&a, t.ev[0], t.ev[1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&b, t.ev[0], t.ev[2]);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      status = XSYMV_ERR_CUDA;
    }
    m += a;
    c += b;
  }
  if (calls) *calls = (int)g_timed.size();
  if (main_ms) *main_ms = m;
  if (call_ms) *call_ms = c;
  for (TimedCall& t : g_timed)
    for (int i = 0; i < 3; ++i) g_free_ev.push_back(t.ev[i]);
  g_timed.clear();
  return status;
}

XSYMV_API long long xsymv_launch_count(void) { return g_launches.load(); }

XSYMV_API int xsymv_sync_status(void) {
  cudaStream_t s = g_stream.load();
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  const int* ptr = nullptr;
  int epoch = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (const CallStatus& c : g_call_status)
      if (c.device == d && c.stream == s) {
        ptr = c.status;
        epoch = c.epoch;
      }
  }
  if (ptr == nullptr || epoch == 0) return XSYMV_OK;
  int word = 0;
  e = cudaMemcpy(&word, ptr, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  return word == epoch ? XSYMV_ERR_TIMEOUT : XSYMV_OK;
}

XSYMV_API int xsymv_set_wait_limit(unsigned long long ns) {
  g_wait_limit.store(ns == 0 ? 2000000000ull : ns);
  return XSYMV_OK;
}

XSYMV_API int xsymv_test_stall(int on) {
  g_extra_tx.store(on ? 16u : 0u);
  return XSYMV_OK;
}

XSYMV_API int xsymv_test_set_call_number(int number) {
  if (number < 0 || number > 0x7ffffffe) return XSYMV_ERR_VALUE;
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  const cudaStream_t s = g_stream.load();
  bool found = noalloc_set_call_number(number);
  std::lock_guard<std::mutex> lk(g_mu);
  for (WsEntry& w : g_ws)
    if (w.device == d && w.stream == s && w.slot == 0 && w.ptr != nullptr) {
      w.epoch = number;
      found = true;
    }
  return found ? XSYMV_OK : XSYMV_ERR_VALUE;
}

XSYMV_API int xsymv_host_traffic(long long* h2d_bytes, long long* d2h_bytes) {
  if (h2d_bytes) *h2d_bytes = g_h2d.load();
  if (d2h_bytes) *d2h_bytes = g_d2h.load();
  return XSYMV_OK;
}

XSYMV_API int xsymv_variant_count(char kind) {
  switch (kind_index(kind)) {
    case 0: return variant_count_s();
    case 1: return variant_count_d();
    case 2: return variant_count_c();
    case 3: return variant_count_z();
    case 4: return variant_count_w();
  }
  return 0;
}

XSYMV_API const char* xsymv_variant_name(char kind, int index) {
  switch (kind_index(kind)) {
    case 0: return variant_name_s(index);
    case 1: return variant_name_d(index);
    case 2: return variant_name_c(index);
    case 3: return variant_name_z(index);
    case 4: return variant_name_w(index);
  }
  return nullptr;
}

XSYMV_API int xsymv_selected_variant(char kind, char uplo, int n) {
  switch (kind_index(kind)) {
    case 0: return selected_variant_s(uplo, n);
    case 1: return selected_variant_d(uplo, n);
    case 2: return selected_variant_c(uplo, n);
    case 3: return selected_variant_z(uplo, n);
    case 4: return selected_variant_w(uplo, n);
  }
  return XSYMV_ERR_VALUE;
}

XSYMV_API long long xsymv_workspace_bytes(char kind, char uplo, int n) {
  switch (kind_index(kind)) {
    case 0: return workspace_bytes_s(uplo, n);
    case 1: return workspace_bytes_d(uplo, n);
    case 2: return workspace_bytes_c(uplo, n);
    case 3: return workspace_bytes_z(uplo, n);
    case 4: return workspace_bytes_w(uplo, n);
  }
  return XSYMV_ERR_VALUE;
}

XSYMV_API int xsymv_shard_bounds(char uplo, int n, int nparts, int* bounds) {
  if (uplo != 'U' && uplo != 'u' && uplo != 'L' && uplo != 'l') return 1;
  if (n < 0) return 2;
  if (nparts < 1) return 3;
  if (bounds == nullptr) return 4;
  const bool upper = (uplo == 'U' || uplo == 'u');
  // stored elements in the columns before c
  auto before = [&](long long c) -> long long {
    return upper ? c * (c + 1) / 2 : c * (long long)n - c * (c - 1) / 2;
  };
  const long long total = before(n);
  bounds[0] = 0;
  for (int r = 1; r < nparts; ++r) {
    // the first column c at which the share of parts 0 .. r-1 is reached
    const long long want = (long long)((__int128)total * r / nparts);
    long long lo = 0, hi = n;
    while (lo < hi) {
      const long long mid = (lo + hi) / 2;
      if (before(mid) >= want) hi = mid; else lo = mid + 1;
    }
    long long c = (lo + kShardAlign / 2) / kShardAlign * kShardAlign;   // nearest multiple
    if (c > n) c = n;
    if (c < bounds[r - 1]) c = bounds[r - 1];
    bounds[r] = (int)c;
  }
  bounds[nparts] = n;
  return XSYMV_OK;
}

XSYMV_API int xsymv_set_variant(char kind, int index) {
  int k = kind_index(kind);
  if (k < 0 || index < -1 || index >= xsymv_variant_count(kind)) return XSYMV_ERR_VALUE;
  g_forced[k] = index;
  return XSYMV_OK;
}

}  // extern "C"
