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
//   * Then, for every output chunk K it contributed to, the warp waits for
//     chunk K's ticket to name it, adds its own partial sums of the chunk
//     (in a fixed order) into v, and hands the ticket to the next
//     contributor.  The contributors of a chunk are ordered by warp index;
//     the first one starts the chain by storing, the last one applies
//     y = alpha*(v + its part) + beta*y.  No addition's order depends on
//     timing, so results are bit-identical from run to run.
//   * A warp waits only for warps with smaller indices, which started
//     earlier (dynamic IDs), so the chain always progresses.  Every wait
//     still has a time limit: when it runs out the warp marks the call
//     failed (status word := the call's epoch), writes NaN to the outputs of
//     every chunk it had not completed, and stops; the chains it would have
//     continued then run out too, so every output whose sum did not
//     complete is NaN.  Another warp that sees the failure stops the same
//     way without waiting for its own limit.
//   * The last block to finish resets the two block counters.
//
// Tickets are 64-bit words "(call << 24) | warp" in a buffer that only these
// kernels write; the call number grows by one per launch, so a ticket left by
// an earlier call can never name a warp of this one.
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
constexpr int kTkWarpBits = 24;   // warp index bits of a ticket

enum Accum {
  kAccumWorkspace = 0,   // symv_main + symv_finalize (fixed-order sums of the workspace)
  kAccumTickets = 1,     // symv_ticket (ordered tickets, one launch)
};

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long r;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(r) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
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
};

// Warp w's block rows Ia..Ib: lane l < 32 caches row Ia + l (the columns
// [ja, jb) it owns there and its row-partial slot q), so that the ticket
// phase needs no plan arithmetic per link; rows past the first 32 (only
// when a warp's share spans more than 32 block rows) are recomputed.
struct WarpRows {
  int Ia, Ib;
  bool own;          // this lane's row: does the warp own columns there
  long long ja, jb;  // and which
  int q;             // its slot among the row's warps
};

__device__ __forceinline__ WarpRows warp_rows(const Plan& p, int w, int lane) {
  WarpRows r;
  r.Ia = plan_row_of(p, plan_wstart(p, w));
  r.Ib = plan_row_of(p, plan_wstart(p, w + 1) - 1);
  r.own = false;
  r.ja = r.jb = 0;
  r.q = 0;
  const int I = r.Ia + lane;
  if (I <= r.Ib) {
    r.own = plan_warp_cols(p, w, I, &r.ja, &r.jb);
    if (r.own) r.q = w - plan_first_owner(p, I);
  }
  return r;
}

// row I's entry (every lane calls this for the same I)
__device__ __forceinline__ bool row_cols(const Plan& p, const WarpRows& r, int w, int I,
                                         long long* ja, long long* jb, int* q) {
  const int l = I - r.Ia;
  if (l < 32) {
    const bool own = __shfl_sync(0xffffffffu, r.own, l);
    *ja = __shfl_sync(0xffffffffu, r.ja, l);
    *jb = __shfl_sync(0xffffffffu, r.jb, l);
    *q = __shfl_sync(0xffffffffu, r.q, l);
    return own;
  }
  if (!plan_warp_cols(p, w, I, ja, jb)) return false;
  *q = w - plan_first_owner(p, I);
  return true;
}

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const int u = __shfl_xor_sync(0xffffffffu, v, o);
    v = u < v ? u : v;
  }
  return v;
}

// the smallest chunk > after that warp w contributes to (>= nb if none)
__device__ __forceinline__ int next_chunk(const Plan& p, const WarpRows& r, int w, int lane,
                                          int after) {
  int best = (r.Ia + lane <= r.Ib && r.own) ? plan_row_next_chunk(p, r.Ia + lane, r.ja, r.jb, after)
                                            : 0x7fffffff;
  best = warp_min(best);
#pragma unroll 1
  for (int I = r.Ia + 32; I <= r.Ib; ++I) {
    long long ja, jb;
    if (!plan_warp_cols(p, w, I, &ja, &jb)) continue;
    const int c = plan_row_next_chunk(p, I, ja, jb, after);
    best = c < best ? c : best;
  }
  return best;
}

// Warp w's partial sums of chunk K: lane l holds outputs K*NB + l + 32m,
// m < M.  Column partials of its rows in increasing row order, the row
// partial of block row K after row K's column partials; has[m] is false
// where the warp has no term.  Offsets within the chunk are 32-bit.
template <class T, int M>
__device__ __forceinline__ void chunk_part(const Plan& p, const TicketCtx<T>& c,
                                           const WarpRows& rows, int w, int K, int lane,
                                           T (&s)[M], bool (&has)[M]) {
  const long long k0 = (long long)K * p.NB;
  const int live = (int)((long long)p.n - k0 < p.NB ? (long long)p.n - k0 : p.NB);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    s[m] = Ops<T>::zero();
    has[m] = false;
  }
#pragma unroll 1
  for (int I = rows.Ia; I <= rows.Ib; ++I) {
    long long ja, jb;
    int q;
    if (!row_cols(p, rows, w, I, &ja, &jb, &q)) continue;
    // this row's columns of the chunk, relative to its first column
    const int lo = (int)((ja > k0 ? ja : k0) - k0);
    const int hi = (int)((jb < k0 + p.NB ? jb : k0 + p.NB) - k0);
    if (lo < hi) {
      const T* wc = c.Wc + (long long)I * p.n + k0 + lane;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int r = lane + 32 * m;
        if (r >= lo && r < hi) {
          const T t = ld_l2(wc + 32 * m);
          s[m] = has[m] ? Ops<T>::add(s[m], t) : t;
          has[m] = true;
        }
      }
    }
    if (I == K) {
      const T* wr = c.Wr + ((long long)K * p.qmax + q) * p.NB + lane;
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

// Warp w's link in chunk K's chain, once the ticket names it (or it is the
// first contributor): add its part into v and pass the ticket to `next`, or,
// as the last contributor (next < 0), write the chunk's outputs of y.
template <class T, int M>
__device__ __forceinline__ void chunk_link(const Plan& p, const TicketCtx<T>& c,
                                           const WarpRows& rows, int w, int K, bool first,
                                           int next, int lane) {
  const long long k0 = (long long)K * p.NB;
  const int live = (int)((long long)p.n - k0 < p.NB ? (long long)p.n - k0 : p.NB);
  T s[M];
  bool has[M];
  chunk_part<T, M>(p, c, rows, w, K, lane, s, has);
  T* vk = c.v + k0 + lane;
  if (!first) {
    // the chain so far: v, then this warp's part
#pragma unroll
    for (int m = 0; m < M; ++m) {
      if (lane + 32 * m < live && (has[m] || next < 0)) {
        const T t = ld_l2(vk + 32 * m);
        s[m] = has[m] ? Ops<T>::add(t, s[m]) : t;
        has[m] = true;
      }
    }
  }
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
  for (int m = 0; m < M; ++m) {
    // the first contributor defines every element of the chunk
    if (lane + 32 * m < live && (has[m] || first))
      st_l2(vk + 32 * m, has[m] ? s[m] : Ops<T>::zero());
  }
  __threadfence();   // this lane's stores to v are visible before the ticket moves
  __syncwarp();
  if (lane == 0 && !(c.withhold && first))
    st_release_u64(c.tk + (long long)K * kTkStride, (c.call << kTkWarpBits) | (unsigned)next);
}

// The ticket phase of warp w (after it has streamed its share): every chunk
// it contributed to, up to 32 at a time (lane k polls the k-th), each linked
// as soon as its ticket names this warp.
template <class T, int NB>
__device__ __forceinline__ void ticket_phase(const Plan& p, const TicketCtx<T>& c, int w,
                                             int lane) {
  constexpr int M = NB / 32;
  const WarpRows rows = warp_rows(p, w, lane);
  const unsigned long long mine = (c.call << kTkWarpBits) | (unsigned)w;
  const long long limit =
      (long long)(c.limit_ns < (1ull << 61) ? c.limit_ns : (1ull << 61)) * 2;   // <= 2 GHz
  int done_upto = -1;   // chunks <= done_upto are linked
#pragma unroll 1
  for (;;) {
    int ck = -1, cnt = 0, cur = done_upto;
#pragma unroll 1
    for (; cnt < 32; ++cnt) {
      const int K = next_chunk(p, rows, w, lane, cur);
      if (K >= p.nb) break;
      if (lane == cnt) ck = K;
      cur = K;
    }
    if (cnt == 0) return;
    bool pending = lane < cnt;
    int first = -1, next = -1;
    bool ready = false;
    if (pending) {
      first = plan_chain_first(p, ck);
      next = plan_chain_next(p, ck, w);
      ready = first == w;
    }
    long long t0 = clock64();
    int spins = 0;
    bool failed = false;
    while (__any_sync(0xffffffffu, pending)) {
      if (pending && !ready) ready = ld_acquire_u64(c.tk + (long long)ck * kTkStride) == mine;
      const unsigned rm = __ballot_sync(0xffffffffu, pending && ready);
      if (rm) {
        const int k = __ffs(rm) - 1;
        const int K = __shfl_sync(0xffffffffu, ck, k);
        const bool f = __shfl_sync(0xffffffffu, first, k) == w;
        const int nx = __shfl_sync(0xffffffffu, next, k);
        __syncwarp();   // lane k's acquire orders the other lanes' reads of v
        chunk_link<T, M>(p, c, rows, w, K, f, nx, lane);
        if (lane == k) pending = false;
        t0 = clock64();
        spins = 0;
        continue;
      }
      if ((++spins & 63) == 0) {
        const bool out = clock64() - t0 > limit || ld_relaxed_int(c.status) == c.epoch;
        if (__any_sync(0xffffffffu, out)) {
          failed = true;
          break;
        }
      }
    }
    if (failed) {
      if (lane == 0) atomicMax(c.status, c.epoch);
      // this batch's unlinked chunks, then every later chunk of the warp
      unsigned left = __ballot_sync(0xffffffffu, pending);
#pragma unroll 1
      while (left) {
        const int k = __ffs(left) - 1;
        chunk_nan<T, M>(p, c, __shfl_sync(0xffffffffu, ck, k), lane);
        left &= left - 1;
      }
#pragma unroll 1
      for (int K = next_chunk(p, rows, w, lane, cur); K < p.nb; K = next_chunk(p, rows, w, lane, K))
        chunk_nan<T, M>(p, c, K, lane);
      return;
    }
    done_upto = cur;
  }
}

// One launch: dynamic block IDs, the warp's share of the stream (register
// path, as symv_main), then its links.  ctr: the ticket buffer's counters.
template <class T, int VR, int U, int WARPS, bool ALIGNED, int MINB, int R = U>
__global__ void __launch_bounds__(WARPS * 32, MINB)
symv_ticket(Plan p, const T* __restrict__ A, long long lda, const T* __restrict__ x, int incx,
            T* Wc, T* Wr, int* ctr, TicketCtx<T> c) {
  constexpr int NB = WarpTile<T, VR, U>::NB;
  __shared__ int s_blk;
  if (threadIdx.x == 0) s_blk = atomicAdd(ctr + kTkStart, 1);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int w = s_blk * WARPS + (int)(threadIdx.x >> 5);
  if (w < p.W) {
    Ring rg{0u, 0u, 0, 0u, 0u};
    stream_warp<T, VR, U, 1, false, ALIGNED, R>(p, w, lane, rg, A, lda, x, incx, Wc, Wr,
                                                c.limit_ns);
    __syncwarp();   // the warp's workspace writes are visible to all its lanes
    ticket_phase<T, NB>(p, c, w, lane);
  }
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
