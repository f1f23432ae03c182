// Ordered-ticket accumulation: the report's own way of combining the
// cross-block partial sums ("CUDA-xSYMV の実装と評価", IPSJ 2014-HPC-146,
// §2.1, figures "kernel" and "Atomic"), as an alternative to the fixed-order
// workspace reduction of symv_finalize.
//
// The report's blocks take dynamic IDs in start order (atomicInc on a
// master counter), and every row chunk of its vector v has a ticket that the
// blocks pass on in a fixed ID order (atomicCAS / atomicExch), so that the
// additions into v happen in the same order on every run.  symv_ticket does
// the same on GB300, in one launch:
//
//   * Each block takes a dynamic ID (atomicAdd on a counter) when it starts;
//     warp w = ID * WARPS + warp-in-block streams the share of the triangle
//     that warp w owns in the partition of xsymv_plan.h (column partials to
//     Wc, row partials to Wr, exactly as symv_main does).
//   * Then the block's warps, which own consecutive column ranges, act as one
//     contributor: for every output chunk K the block contributed to, one of
//     its warps waits for chunk K's ticket to name the block, adds the
//     block's partial sums of the chunk (in a fixed order) into v, and hands
//     the ticket to the next contributing block.  Contributors of a chunk
//     are ordered by block ID; the first one starts the chain by storing,
//     the last one applies y = alpha*(v + its part) + beta*y.  No
//     addition's order depends on timing, so results are bit-identical from
//     run to run.
//   * A block waits only for blocks with smaller IDs, which started earlier
//     (dynamic IDs), so the chain always progresses.  Every wait still has
//     a time limit: when it runs out the warp marks the call failed (status
//     word := the call's epoch), writes NaN to the outputs of every chunk it
//     had not completed, and stops; the chains it would have continued then
//     run out too, so every output whose sum did not complete is NaN.
//     Another warp that sees the failure stops the same way without waiting
//     for its own limit.
//   * The last block to finish resets the two block counters.
//
// Tickets are 64-bit words "(call << 24) | block" in a buffer that only these
// kernels write; the call number grows by one per launch, so a ticket left by
// an earlier call can never name a block of this one.
#pragma once

#include "xsymv_kernels.cuh"

namespace xsymv {

// ticket buffer: int counters at words kTkStart (blocks started) and kTkDone
// (blocks finished), then from byte kTkHeaderBytes one ticket per chunk,
// kTkStride 64-bit words apart (a 32-byte sector each)
constexpr int kTkStart = 0;
constexpr int kTkDone = 8;
constexpr long long kTkHeaderBytes = 256;
constexpr int kTkStride = 4;
constexpr int kTkIdBits = 24;     // block ID bits of a ticket
constexpr int kTkRows = 32;       // block rows of a block kept in shared memory

enum Accum {
  kAccumWorkspace = 0,   // symv_main + symv_finalize (fixed-order sums of the workspace)
  kAccumTickets = 1,     // symv_ticket (ordered tickets, one launch)
  kAccumFused = 2,       // symv_fused (the same fixed-order sums after a grid barrier, one launch)
};

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long r;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(r) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long r;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(r) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ int ld_relaxed_int(const int* p) {
  int r;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
  return r;
}

// loads and stores of T at the L2 (never served from a possibly stale L1)
template <class T>
__device__ __forceinline__ T ld_l2(const T* p) {
  static_assert(sizeof(T) == 4 || sizeof(T) == 8 || sizeof(T) == 16, "element size");
  T r;
  if (sizeof(T) == 4) {
    const unsigned b = __ldcg(reinterpret_cast<const unsigned*>(p));
    memcpy(&r, &b, sizeof(T));
  } else if (sizeof(T) == 8) {
    const unsigned long long b = __ldcg(reinterpret_cast<const unsigned long long*>(p));
    memcpy(&r, &b, sizeof(T));
  } else {
    const ulonglong2 b = __ldcg(reinterpret_cast<const ulonglong2*>(p));
    memcpy(&r, &b, sizeof(T));
  }
  return r;
}
template <class T>
__device__ __forceinline__ void st_l2(T* p, T v) {
  if (sizeof(T) == 4) {
    unsigned b;
    memcpy(&b, &v, 4);
    __stcg(reinterpret_cast<unsigned*>(p), b);
  } else if (sizeof(T) == 8) {
    unsigned long long b;
    memcpy(&b, &v, 8);
    __stcg(reinterpret_cast<unsigned long long*>(p), b);
  } else {
    ulonglong2 b;
    memcpy(&b, &v, 16);
    __stcg(reinterpret_cast<ulonglong2*>(p), b);
  }
}

// Everything the ticket phase needs besides the plan.
template <class T>
struct TicketCtx {
  const T* Wc;
  const T* Wr;
  T* v;                       // n elements: the running sums
  unsigned long long* tk;     // chunk K's ticket at tk[K * kTkStride]
  int* status;
  int epoch;                  // the call's number in the status word
  unsigned long long call;    // the call's number in the tickets
  unsigned long long limit_ns;
  int withhold;               // test hook: first contributors keep their tickets
  T alpha, beta;
  int mode;                   // kFull or kBetaZero
  T* y;                       // logical element 0 of y
  long long incy;
  const int2* rt;             // the plan's row table
};

// A block's share of one block row: the columns [ja, jb) its warps own
// (ja >= jb: none).
struct GroupRow {
  long long ja, jb;
};

// the group's rows Ia..Ib; rows Ia .. Ia+kTkRows-1 are in shared memory,
// later ones (only when a block's share spans more block rows) recomputed
struct GroupRows {
  int w0, w1;          // warps of the group
  int gid;             // the group's (block's) index: its row-partial slots
  int Ia, Ib;
  const GroupRow* sm;  // kTkRows entries
};

__device__ __forceinline__ GroupRow group_row(const Plan& p, const GroupRows& g, int I) {
  if (I - g.Ia < kTkRows) return g.sm[I - g.Ia];
  GroupRow r{0, 0};
  if (!plan_group_cols(p, g.w0, g.w1, I, &r.ja, &r.jb)) r.ja = r.jb = 0;
  return r;
}

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const int u = __shfl_xor_sync(0xffffffffu, v, o);
    v = u < v ? u : v;
  }
  return v;
}

// the smallest chunk > after that the group contributes to (>= nb if none);
// lane l looks at row Ia + l
__device__ __forceinline__ int next_chunk(const Plan& p, const GroupRows& g, int lane, int after) {
  int best = 0x7fffffff;
  if (lane < kTkRows && g.Ia + lane <= g.Ib) {
    const GroupRow r = g.sm[lane];
    if (r.ja < r.jb) best = plan_row_next_chunk(p, g.Ia + lane, r.ja, r.jb, after);
  }
  best = warp_min(best);
#pragma unroll 1
  for (int I = g.Ia + kTkRows; I <= g.Ib; ++I) {
    const GroupRow r = group_row(p, g, I);
    if (r.ja >= r.jb) continue;
    const int c = plan_row_next_chunk(p, I, r.ja, r.jb, after);
    best = c < best ? c : best;
  }
  return best;
}

// The group's partial sums of chunk K, added to s[m] (lane l holds outputs
// K*NB + l + 32m, m < M): column partials of its rows in increasing row
// order, then, in row K, the group's row partial (its slot of the row).
// has[m] is false where there was no term yet.  Offsets are 32-bit.
template <class T, int M>
__device__ __forceinline__ void chunk_part(const Plan& p, const TicketCtx<T>& c,
                                           const GroupRows& g, int K, int lane, T (&s)[M],
                                           bool (&has)[M]) {
  const long long k0 = (long long)K * p.NB;
  const int live = (int)((long long)p.n - k0 < p.NB ? (long long)p.n - k0 : p.NB);
#pragma unroll 1
  for (int I = g.Ia; I <= g.Ib; ++I) {
    const GroupRow r = group_row(p, g, I);
    if (r.ja >= r.jb) continue;
    // this row's columns of the chunk, relative to its first column
    const int lo = (int)((r.ja > k0 ? r.ja : k0) - k0);
    const int hi = (int)((r.jb < k0 + p.NB ? r.jb : k0 + p.NB) - k0);
    if (lo < hi) {
      const T* wc = c.Wc + (long long)I * p.n + k0 + lane;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int o = lane + 32 * m;
        if (o >= lo && o < hi) {
          const T t = ld_l2(wc + 32 * m);
          s[m] = has[m] ? Ops<T>::add(s[m], t) : t;
          has[m] = true;
        }
      }
    }
    if (I == K) {
      const T* wr = c.Wr + ((long long)K * p.qmax + (g.gid - __ldg(&c.rt[K].x))) * p.NB + lane;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        if (lane + 32 * m < live) {
          const T t = ld_l2(wr + 32 * m);
          s[m] = has[m] ? Ops<T>::add(s[m], t) : t;
          has[m] = true;
        }
      }
    }
  }
}

// y := NaN on the outputs of chunk K (a chain that could not complete)
template <class T, int M>
__device__ __forceinline__ void chunk_nan(const Plan& p, const TicketCtx<T>& c, int K, int lane) {
  const long long k0 = (long long)K * p.NB;
  const int live = (int)((long long)p.n - k0 < p.NB ? (long long)p.n - k0 : p.NB);
  T* yk = c.y + (k0 + lane) * c.incy;
  const long long step = 32 * c.incy;
#pragma unroll
  for (int m = 0; m < M; ++m)
    if (lane + 32 * m < live) yk[m * step] = Ops<T>::nan();
}

// The group's link in chunk K's chain, once the ticket names it (or it is
// the first contributor): add its part into v and pass the ticket to group
// `next`, or, as the last contributor (next < 0), write the chunk's outputs.
template <class T, int M>
__device__ __forceinline__ void chunk_link(const Plan& p, const TicketCtx<T>& c,
                                           const GroupRows& g, int K, bool first, int next,
                                           int lane) {
  const long long k0 = (long long)K * p.NB;
  const int live = (int)((long long)p.n - k0 < p.NB ? (long long)p.n - k0 : p.NB);
  T* vk = c.v + k0 + lane;
  T s[M];
  bool has[M];
  // the chain so far (v) first, then this group's part: the loads of both
  // are in flight together
#pragma unroll
  for (int m = 0; m < M; ++m) {
    has[m] = !first && lane + 32 * m < live;
    s[m] = has[m] ? ld_l2(vk + 32 * m) : Ops<T>::zero();
  }
  chunk_part<T, M>(p, c, g, K, lane, s, has);
  if (next < 0) {
    T* yk = c.y + (k0 + lane) * c.incy;
    const long long step = 32 * c.incy;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      if (lane + 32 * m < live) {
        const T sum = has[m] ? s[m] : Ops<T>::zero();
        T* yj = yk + m * step;
        if (c.mode == kFull)
          *yj = Ops<T>::add(Ops<T>::mul(c.alpha, sum), Ops<T>::mul(c.beta, *yj));
        else
          *yj = Ops<T>::mul(c.alpha, sum);
      }
    }
    return;
  }
#pragma unroll
  for (int m = 0; m < M; ++m)
    if (lane + 32 * m < live) st_l2(vk + 32 * m, has[m] ? s[m] : Ops<T>::zero());
  __threadfence();   // this lane's stores to v are visible before the ticket moves
  __syncwarp();
  if (lane == 0 && !(c.withhold && first))
    st_release_u64(c.tk + (long long)K * kTkStride, (c.call << kTkIdBits) | (unsigned)next);
}

// The ticket phase of group (block) gid after all its warps have streamed
// their shares: the group's chunks in increasing order, dealt round-robin to
// its warps (warp `wl` of `nw` takes entries wl, wl + nw, ...); each warp
// polls up to 32 of its chunks at once (lane k the k-th) and links each as
// soon as its ticket names the group.
template <class T, int NB>
__device__ __forceinline__ void ticket_phase(const Plan& p, const TicketCtx<T>& c,
                                             const GroupRows& g, int gid, int G, int wl, int nw,
                                             int lane) {
  constexpr int M = NB / 32;
  const unsigned long long mine = (c.call << kTkIdBits) | (unsigned)gid;
  int cur = -1;   // the group's chunks <= cur have been dealt
#pragma unroll 1
  for (;;) {
    // this warp's next batch: every nw-th chunk of the group's list
    int ck = -1, cnt = 0;
#pragma unroll 1
    while (cnt < 32) {
      int K = cur;
#pragma unroll 1
      for (int i = 0; i < nw; ++i) {
        K = next_chunk(p, g, lane, K);
        if (K >= p.nb) break;
        if (i == wl) {
          if (lane == cnt) ck = K;
          ++cnt;
        }
      }
      if (K >= p.nb) {
        cur = p.nb;
        break;
      }
      cur = K;
    }
    if (cnt == 0) return;
    bool pending = lane < cnt;
    int first = -1, next = -1;
    bool ready = false;
    if (pending) {
      first = plan_group_first(p, ck, G);
      next = plan_group_next(p, ck, gid, G);
      ready = first == gid;
    }
    unsigned long long t0 = global_ns();
    int spins = 0;
    bool failed = false;
    while (__any_sync(0xffffffffu, pending)) {
      if (pending && !ready && ld_relaxed_u64(c.tk + (long long)ck * kTkStride) == mine) {
        fence_acq_rel();   // with the relaxed load that saw it: acquire the link before
        ready = true;
      }
      const unsigned rm = __ballot_sync(0xffffffffu, pending && ready);
      if (rm) {
        const int k = __ffs(rm) - 1;
        const int K = __shfl_sync(0xffffffffu, ck, k);
        const bool f = __shfl_sync(0xffffffffu, first, k) == gid;
        const int nx = __shfl_sync(0xffffffffu, next, k);
        __syncwarp();   // lane k's acquire orders the other lanes' reads of v
        chunk_link<T, M>(p, c, g, K, f, nx, lane);
        if (lane == k) pending = false;
        t0 = global_ns();
        spins = 0;
        continue;
      }
      __nanosleep(32);
      if ((++spins & 63) == 0) {
        const bool out = global_ns() - t0 > c.limit_ns || ld_relaxed_int(c.status) == c.epoch;
        if (__any_sync(0xffffffffu, out)) {
          failed = true;
          break;
        }
      }
    }
    if (failed) {
      if (lane == 0) atomicMax(c.status, c.epoch);
      // this batch's unlinked chunks, then this warp's share of the rest
      unsigned left = __ballot_sync(0xffffffffu, pending);
#pragma unroll 1
      while (left) {
        const int k = __ffs(left) - 1;
        chunk_nan<T, M>(p, c, __shfl_sync(0xffffffffu, ck, k), lane);
        left &= left - 1;
      }
      int K = cur;
#pragma unroll 1
      for (int i = 0; (K = next_chunk(p, g, lane, K)) < p.nb; ++i)
        if (i % nw == wl) chunk_nan<T, M>(p, c, K, lane);
      return;
    }
  }
}

// One launch: dynamic block IDs, the warps' shares of the stream (register
// path, as symv_main), then the block's links.  ctr: the ticket buffer's
// counters.
template <class T, int VR, int U, int WARPS, bool ALIGNED, int MINB, int R = U>
__global__ void __launch_bounds__(WARPS * 32, MINB)
symv_ticket(Plan p, const T* __restrict__ A, long long lda, const T* __restrict__ x, int incx,
            T* Wc, T* Wr, const int4* __restrict__ wt, const int2* __restrict__ rt, int* ctr,
            TicketCtx<T> c) {
  constexpr int NB = WarpTile<T, VR, U>::NB;
  __shared__ int s_blk;
  __shared__ GroupRow s_rows[kTkRows];
  __shared__ RowBuffers<T, NB, WARPS> rb;
  if (threadIdx.x == 0) s_blk = atomicAdd(ctr + kTkStart, 1);
  const int lane = threadIdx.x & 31;
  const int wl = (int)(threadIdx.x >> 5);
  if (lane < 2) rb.row[wl][lane] = -1;
  __syncthreads();
  const int blk = s_blk;
  const int w = blk * WARPS + wl;
  if (w < p.W) {
    Ring rg{0u, 0u, 0, 0u, 0u};
    stream_warp<T, VR, U, 1, false, ALIGNED, R, WARPS>(p, w, wl, blk, lane, rg, A, lda, x, incx,
                                                       Wc, Wr, wt, rt, rb, c.limit_ns);
  }
  __syncthreads();
  row_partials_combine<T, NB, WARPS>(p, Wr, rt, blk, rb);
  // the block's warps act as one contributor: their workspace writes are
  // visible to the whole block after the barrier
  GroupRows g;
  g.gid = blk;
  g.w0 = blk * WARPS;
  g.w1 = g.w0 + WARPS < p.W ? g.w0 + WARPS : p.W;
  g.sm = s_rows;
  if (g.w0 < p.W) {
    g.Ia = plan_row_of(p, plan_wstart(p, g.w0));
    g.Ib = plan_row_of(p, plan_wstart(p, g.w1) - 1);
    if ((int)threadIdx.x < kTkRows) {
      GroupRow r{0, 0};
      const int I = g.Ia + (int)threadIdx.x;
      if (I > g.Ib || !plan_group_cols(p, g.w0, g.w1, I, &r.ja, &r.jb)) r.ja = r.jb = 0;
      s_rows[threadIdx.x] = r;
    }
  }
  __syncthreads();
  if (g.w0 < p.W) ticket_phase<T, NB>(p, c, g, blk, WARPS, wl, WARPS, lane);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ctr + kTkDone, 1) == (int)gridDim.x - 1) {
      // every block has taken its ID: the next launch counts from zero
      ctr[kTkStart] = 0;
      ctr[kTkDone] = 0;
    }
  }
}

}  // namespace xsymv
