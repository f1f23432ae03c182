// Host-side services shared by the five entry points: stream, device
// properties, per-(device, stream) workspace, launch counting, event timing
// and variant overrides.  Implemented in xsymv_api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace xsymv {

cudaStream_t current_stream();

// Kernel attributes and occupancy belong to a device, and one process may
// drive several GPUs: the kernels' per-device caches have kMaxDevices slots,
// indexed by current_device_index() (-1 on a CUDA error or a device number
// beyond the slots; such calls compute afresh every time).
constexpr int kMaxDevices = 64;
int current_device_index();

// current device and its multiprocessor count; false if there is no usable
// device (records the CUDA error)
bool current_device(int* dev, int* sm_count);

// buffer of at least `bytes` for (current device, stream, slot); nullptr and
// *status set on failure.  Slot 0: the kernels' workspace; slot 1: device
// copies of host operands for the host-buffer entry points.
// For slot 0 the first 256 bytes (the status header) are zeroed when the
// buffer is allocated, and *epoch receives a fresh call number (> 0) that the
// kernels write to the status word if they give up on a wait.
// *capacity (if given) receives the buffer's allocated size (>= bytes).
void* workspace(size_t bytes, cudaStream_t stream, int* status, int slot, int* epoch,
                size_t* capacity = nullptr);

// Record where the latest call on (current device, stream) keeps its
// status word and the call number its kernels write there if a bounded wait
// runs out; xsymv_sync_status reads it.  status == nullptr: the call has no
// status word (it launched no kernel that waits).  y_lo < y_hi: the call
// ended with the two-kernel path's finaliser, which writes (at most) the
// bytes [y_lo, y_hi) and reads the workspace half of its call number's
// parity; the next call's main kernel may then stream before it finishes
// (may_start_early).
void note_call_status(cudaStream_t stream, const int* status, int epoch, uintptr_t y_lo = 0,
                      uintptr_t y_hi = 0);

// A host-mapped word per (current device, stream) in which the main
// kernels of early-started calls report whether they overlapped the previous
// finaliser: returns its host address (read it to see the latest report)
// and sets *dev to its device address; nullptr (and *dev = nullptr) if it
// could not be allocated.
const volatile int* overlap_flag(cudaStream_t stream, int** dev);

// true if the latest call on (current device, stream) ended with a
// finaliser whose writes miss both byte ranges [a_lo, a_hi) and [x_lo, x_hi)
bool may_start_early(cudaStream_t stream, uintptr_t a_lo, uintptr_t a_hi, uintptr_t x_lo,
                     uintptr_t x_hi);

// Set the last call number of the allocation-free entry point on the current
// device (defined beside it); false if that entry point has not been called
// on this device yet.
bool noalloc_set_call_number(int number);

// buffer of at least `bytes` for the ordered-ticket kernels on (current
// device, stream): zeroed when it is allocated, written by nothing but those
// kernels.  *call receives a fresh call number (>= 1, never reused for the
// buffer) that the kernel's tickets carry.  nullptr and *status set on failure.
void* ticket_buffer(size_t bytes, cudaStream_t stream, int* status, unsigned long long* call);

// buffer of at least `bytes` on (current device, stream) for a plan's warp
// and row tables (see xsymv_plan.h).  *ready is true when the buffer already
// holds the tables of `key` (compared bytewise); either way the buffer is
// recorded as holding them, so the caller must enqueue their construction
// on `stream` when *ready is false, or call plan_tables_forget() if it
// cannot.  A buffer that had to grow holds no tables.  nullptr and *status
// set on failure.
void* plan_tables(size_t bytes, cudaStream_t stream, const void* key, size_t key_bytes,
                  bool* ready, int* status);
void plan_tables_forget(cudaStream_t stream);

// time limit of every bounded wait in the kernels
unsigned long long wait_limit_ns();
// extra bytes announced on every ring barrier: 0, except when a test makes
// the waits run out on purpose
uint32_t test_extra_tx();

// bytes moved by the last host-buffer call
void note_host_traffic(long long h2d, long long d2h);

void note_launches(int k);
void record_cuda_error(cudaError_t e);

// event timing around one call: begin() before the main kernel, mid() after
// it, end() after the last kernel.  Does nothing unless timing is enabled.
void timing_begin(cudaStream_t s);
void timing_mid(cudaStream_t s);
void timing_end(cudaStream_t s);

// -1 unless a variant was forced for this kind
int forced_variant(char kind);

// per-kind introspection, defined next to each kind's variant table
#define XSYMV_DECLARE_INTROSPECTION(KIND)            \
  int variant_count_##KIND();                        \
  const char* variant_name_##KIND(int i);            \
  int selected_variant_##KIND(char uplo, int n);     \
  long long workspace_bytes_##KIND(char uplo, int n);
XSYMV_DECLARE_INTROSPECTION(s)
XSYMV_DECLARE_INTROSPECTION(d)
XSYMV_DECLARE_INTROSPECTION(c)
XSYMV_DECLARE_INTROSPECTION(z)
XSYMV_DECLARE_INTROSPECTION(w)
#undef XSYMV_DECLARE_INTROSPECTION

}  // namespace xsymv
