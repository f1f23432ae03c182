// The whole call in one launch: symv_fused streams the triangle exactly as
// symv_main does, waits at a grid-wide barrier until every block has written
// its partial sums, then every block takes a share of the final merge, the
// same fixed-order sums as symv_finalize (so results are bit-identical to
// the two-kernel path of the same plan).  It saves the finaliser's launch and
// the gap between the two kernels, a few microseconds that weigh at small n.
//
// The barrier needs every block of the grid resident at once: the grid is
// the resident wave the occupancy calculator reports, launched as a
// cooperative grid (the driver then starts all of its blocks together or
// waits until it can).  Its wait is bounded: when the limit runs out the
// call is marked failed in the status word (its outputs become NaN) and the
// kernel returns; nothing is left that the next call could trip over.
#pragma once

#include "xsymv_ticket.cuh"

namespace xsymv {

// The grid barrier's word (64 bits in the workspace header): the call number
// in the high half, the blocks that have arrived in the low half.  A block
// first raises the word to (epoch << 32) with atomicMax, which clears an
// earlier call's count (call numbers increase; when they start again at 1
// the whole header is zeroed), then adds one; every block then waits until
// the word reads (epoch << 32) + blocks.  A call that gave up leaves a count
// the next call's first atomicMax discards.
constexpr long long kBarrierOffset = 8;   // bytes into the workspace header

__device__ __forceinline__ bool grid_barrier(unsigned long long* bar, int epoch, unsigned target,
                                             unsigned long long limit_ns) {
  const unsigned long long tag = (unsigned long long)(unsigned)epoch << 32;
  atomicMax(bar, tag);
  atomicAdd(bar, 1ull);
  const unsigned long long want = tag | target;
  if (ld_acquire_u64(bar) >= want) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_u64(bar) >= want) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// A one-launch kernel that begins less than this after the previous call
// on its stream ended ran back to back with it: the two calls were queued
// together, with no other kernel between them.  (Measured on GB300: a
// cooperative grid queued behind another begins 2.4-4.7 us after the last
// block of the one before it ends; a kernel of the caller in between adds
// its own two launch gaps and its run time.  A wrong answer costs only
// speed, and the next call's report corrects it.)
constexpr unsigned long long kBackToBackNs = 6000;

// the final merge's arguments (as for symv_finalize)
template <class T>
struct FinalArgs {
  T alpha, beta;
  int mode;
  T* y;            // logical element 0
  long long incy;
};

template <class T, int VR, int U, int WARPS, bool ALIGNED, int MINB, int R>
__global__ void __launch_bounds__(WARPS * 32, MINB)
symv_fused(Plan p, const T* __restrict__ A, long long lda, const T* __restrict__ x, int incx,
           T* __restrict__ Wc, T* __restrict__ Wr, const int4* __restrict__ wt,
           const int2* __restrict__ rt, int* status, int epoch, unsigned long long limit_ns,
           int stall, unsigned long long* bar, FinalArgs<T> f, OverlapWords ow) {
  static_assert(WARPS * 32 == kFinParts * kFinCols, "one finaliser block per thread block");
  constexpr int NB = WarpTile<T, VR, U>::NB;
  __shared__ RowBuffers<T, NB, WARPS> rb;
  __shared__ T part[kFinParts][kFinCols];
  const int lane = threadIdx.x & 31;
  const int wl = threadIdx.x >> 5;
  const int w = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  if (lane < 2) rb.row[wl][lane] = -1;
  __syncwarp();
  const bool reporter = ow.report != nullptr && blockIdx.x == 0 && threadIdx.x == 0;
  const unsigned long long began = reporter ? global_ns() : 0;
  // launched as a programmatic dependent of the stream's previous kernel:
  // nothing of global memory is touched before that kernel has completed.
  // (This grid lets its own dependents start only after the barrier below,
  // so that their blocks cannot take the places this grid's blocks need.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // did this call follow the previous one back to back?  (The host reads the
  // answer when it enqueues later calls, and then prefers the two-kernel
  // twin of this variant, whose calls fill each other's tails.)
  if (reporter) {
    const unsigned long long prev = *reinterpret_cast<const volatile unsigned long long*>(ow.prev_end);
    *reinterpret_cast<volatile int*>(ow.report) = began < prev + kBackToBackNs ? 1 : 0;
  }
  if (w < p.W) {
    Ring rg{0u, 0u, 0, 0u, 0u};
    stream_warp<T, VR, U, 1, false, ALIGNED, R, WARPS>(p, w, wl, blockIdx.x, lane, rg, A, lda, x,
                                                       incx, Wc, Wr, wt, rt, rb, limit_ns);
  }
  __syncthreads();
  row_partials_combine<T, NB, WARPS>(p, Wr, rt, blockIdx.x, rb);
  // every thread's workspace writes, then the block's arrival
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    // the test hook waits for one block more than there are
    // a block that gave up marks the call failed: the final sums then write NaN
    if (!grid_barrier(bar, epoch, gridDim.x + (stall ? 1u : 0u), limit_ns)) atomicMax(status, epoch);
  }
  __syncthreads();
  __threadfence();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long nfb = (p.n + kFinCols - 1) / kFinCols;
  for (long long fb = blockIdx.x; fb < nfb; fb += gridDim.x) {
    // (4 loads in flight: the kernels with a tight register cap keep their
    // streaming registers free of spills)
    finalize_outputs<T, true, 4>(p, Wc, Wr, rt, f.alpha, f.beta, f.mode, f.y, f.incy, status,
                                 epoch, fb, part);
    __syncthreads();
  }
  // the time the grid's last block ends (a reduction nobody waits for)
  if (ow.end != nullptr && threadIdx.x == 0) atomicMax(ow.end, global_ns());
}

}  // namespace xsymv
