// xSYMV / xHEMV kernels for sm_103a: y := alpha*A*x + beta*y with A symmetric
// (Hermitian for complex types), only the upper or lower triangle stored in
// column-major order with leading dimension lda.
//
// Method ("CUDA-xSYMV の実装と評価", IPSJ 2014-HPC-146, §2.1): every stored
// element A(i,j), i != j, is read from memory once and used twice, for the
// row term A(i,j)*x(j) of y(i) and the column term conj(A(i,j))*x(i) of y(j);
// this halves the memory traffic of GEMV.  The report's kernels are the
// preprocess (y *= beta, v = 0), main (parts one and two) and postprocess
// (y += alpha*v) of figure "kernel", with ordered tickets for the updates of
// v.  Here the same arithmetic is organised for GB300:
//
//   symv_main      Each warp streams an equal share of the triangle's column
//                  segments (see xsymv_plan.h).  A column segment is the
//                  NB-row piece of one matrix column inside one block row:
//                  the 32 lanes cover its NB rows (VR 16-byte vectors per
//                  lane), U columns at a time.  Off-diagonal columns are read
//                  either straight into registers (kPipeRegisters) or through
//                  a per-warp shared-memory ring filled by bulk asynchronous
//                  copies (cp.async.bulk, the TMA engine) completed on
//                  mbarriers (kPipeBulk).  Row terms stay in the lane's
//                  registers for the whole block row (each lane owns its
//                  rows); column terms are summed across the 32 lanes with a
//                  butterfly reduce-scatter of the U columns and written to
//                  the workspace.  The diagonal tile goes through the same
//                  arithmetic with a triangle mask: its stored part is read
//                  once and contributes to both sides, which is what the
//                  report's mirrored copy in shared memory (part two)
//                  achieves (on aligned matrices as 16-byte vectors, whose
//                  few elements across the diagonal are ignored).
//   symv_finalize  For every output element, sums the workspace slots of its
//                  row in a fixed order and applies y = alpha*s + beta*y (the
//                  report's part three and beta scaling).  No atomic
//                  operation touches data, so results are bit-identical from
//                  run to run.
//
// On GB300 the register path is the faster one for SSYMV/CHEMV: what sets
// the speed is the 16-byte loads in flight per SM, so the tuned variants cap
// registers (40 per thread and 48 warps per SM with 4 rows per lane; 64 and
// 32 warps with 8 rows per lane, twice the bytes per warp, at large n).
// Both kernels are launched as programmatic dependents (main after the
// stream's previous kernel, finaliser after main) and wait for their
// predecessor before touching global memory.  Every wait of the bulk-copy ring
// on an mbarrier has a time limit.  A wait that runs out marks the call
// failed (status word := the call's epoch), waits (again with a limit) for
// the warp's copies still in flight and leaves the kernel; the finaliser then
// writes NaN to y and the host can read the status.
#pragma once

#include <string.h>

#include <type_traits>

#include "xsymv_plan.h"
#include "xsymv_scalar.cuh"

namespace xsymv {

// Bytes into the workspace header of the overlap bookkeeping of
// back-to-back calls: four 64-bit words, the finalisers' end times and the
// early main kernels' start times, one of each per call parity.
constexpr long long kOverlapOffset = 16;

template <int U> struct Log2;
template <> struct Log2<1> { static constexpr int v = 0; };
template <> struct Log2<2> { static constexpr int v = 1; };
template <> struct Log2<4> { static constexpr int v = 2; };
template <> struct Log2<8> { static constexpr int v = 3; };
template <> struct Log2<16> { static constexpr int v = 4; };
template <> struct Log2<32> { static constexpr int v = 5; };

// -------------------------------------------------- async-copy primitives --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// one arrival that also announces `bytes` of asynchronous transfers
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// HBM -> shared bulk copy; dst, src 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

// The GPU's global nanosecond timer (%globaltimer): the same time base on
// every SM, independent of the SM clock.
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// store the global timer at p (a 64-bit word), one instruction pair
__device__ __forceinline__ void note_time(void* p) {
  asm volatile("{\n\t.reg .u64 t;\n\tmov.u64 t, %%globaltimer;\n\tst.global.u64 [%0], t;\n\t}" ::"l"(p)
               : "memory");
}

// Wait for phase `parity` of the mbarrier, giving up once limit_ns have
// passed on the global timer (read every 256 tries).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Sum v[0..U) over the 32 lanes of the warp.  On return lane l holds the
// total of column u = l >> (5 - log2 U); the additions happen in a fixed
// pattern, independent of timing.
template <class T, int U>
__device__ __forceinline__ T reduce_scatter(T (&v)[U], int lane) {
  constexpr int H = Log2<U>::v;
  int off = 16;
#pragma unroll
  for (int h = 0; h < H; ++h) {
    const int half = U >> (h + 1);
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      T send = up ? v[i] : v[i + half];
      T keep = up ? v[i + half] : v[i];
      v[i] = Ops<T>::add(keep, Ops<T>::shfl_xor(send, off));
    }
    off >>= 1;
  }
#pragma unroll
  for (int o = 16 >> H; o >= 1; o >>= 1) v[0] = Ops<T>::add(v[0], Ops<T>::shfl_xor(v[0], o));
  return v[0];
}

// How off-diagonal columns travel from HBM to the arithmetic.
enum Pipe {
  kPipeRegisters = 0,   // 16-byte loads straight into registers, U columns at a time
  kPipeBulk = 1,        // per-warp shared-memory ring filled by cp.async.bulk (TMA) copies
};

// Per-warp ring of STAGES chunks in shared memory (bulk-copy pipe only);
// chunk = U column segments of NB elements, plus one mbarrier per stage.
template <class T, int VR, int U, int STAGES, int PIPE>
struct RingLayout {
  static constexpr int NB = 32 * Ops<T>::VPL * VR;
  static constexpr int COL_BYTES = NB * (int)sizeof(T);
  static constexpr int STAGE_BYTES = U * COL_BYTES;
  static constexpr int DATA_BYTES = PIPE == kPipeBulk ? STAGES * STAGE_BYTES : 0;
  static constexpr int BAR_BYTES = PIPE == kPipeBulk ? ((STAGES * 8 + 15) / 16) * 16 : 0;
  static constexpr int WARP_BYTES = DATA_BYTES + BAR_BYTES;
};

struct Ring {
  uint32_t data;      // shared address of stage 0
  uint32_t bars;      // shared address of the first mbarrier
  int head;           // stage of the next chunk to consume
  uint32_t phase;     // bit s: parity of stage s's next completion
  uint32_t extra_tx;  // bytes announced beyond the copies (0; > 0 only to test the time limit)
};

template <class T, int VR, int U>
struct WarpTile {
  static constexpr int VPL = Ops<T>::VPL;
  static constexpr int NB = 32 * VPL * VR;
  static constexpr int H = Log2<U>::v;

  // one block row's state for this lane
  T xi[VR][VPL];
  T racc[VR][VPL];

  // row held by (vector v, element k) of this lane, relative to the block row
  __device__ __forceinline__ static int lane_row(int v, int lane, int k) {
    return (v * 32 + lane) * VPL + k;
  }

  // row terms into racc; column terms reduced over the warp and written to
  // wc[0 .. cnt) (a[u] = column u of the chunk, xl on lane u = its x)
  __device__ __forceinline__ void accumulate(T (&a)[U][VR][VPL], T xl, int cnt, T* wc,
                                             int lane) {
    T cp[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const T xj = Ops<T>::shfl(xl, u);
      T c = Ops<T>::zero();
#pragma unroll
      for (int v = 0; v < VR; ++v)
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
          racc[v][k] = Ops<T>::madd(racc[v][k], a[u][v][k], xj);
          c = Ops<T>::maddc(c, a[u][v][k], xi[v][k]);
        }
      cp[u] = c;
    }
    T red = reduce_scatter<T, U>(cp, lane);
    const int uo = lane >> (5 - H);
    if ((lane & ((32 >> H) - 1)) == 0 && uo < cnt) wc[uo] = red;
  }

  // the lane's rows of the U columns col, col + lda, ... (col: this lane's
  // first element), with 16-byte vector loads (ALIGNED) or element loads
  template <bool ALIGNED>
  __device__ __forceinline__ static void load_cols(const T* col, long long lda,
                                                   T (&a)[U][VR][VPL]) {
    if (ALIGNED) {
      uint4 raw[U][VR];
      const T* c = col;
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int v = 0; v < VR; ++v) raw[u][v] = ldg_stream16(c + v * 32 * VPL);
        c += lda;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int v = 0; v < VR; ++v) Unpack<T>::run(raw[u][v], a[u][v]);
    } else {
      const T* c = col;
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int v = 0; v < VR; ++v)
#pragma unroll
          for (int k = 0; k < VPL; ++k) a[u][v][k] = Ops<T>::load(c + v * 32 * VPL + k);
        c += lda;
      }
    }
  }

  // Columns [ja, jb) of the block row at r0, all NB rows stored, read with
  // 16-byte vector loads (ALIGNED) or element loads straight into registers.
  // The loop keeps only running pointers and a 32-bit count live.
  //
  // R > U batches the column reductions: the column terms of R columns,
  // loaded U at a time, are reduced across the warp together, which takes
  // one butterfly of R values (R - 1 + 5 - log2 R additions per lane) in
  // place of R/U butterflies of U values, and keeps the shuffles' latency
  // out of all but one load step in R/U.
  template <bool ALIGNED, int R = U>
  __device__ __forceinline__ void dense_cols(const T* __restrict__ A, long long lda,
                                             const T* __restrict__ x, int incx, long long r0,
                                             long long ja, long long jb, T* wc_row, int lane) {
    static_assert(R % U == 0 && R <= 32, "R: a multiple of U, at most 32");
    const T* col = A + ja * lda + r0 + lane_row(0, lane, 0);   // this lane, column ja
    const T* xp = x + ja * (long long)incx;
    T* wc = wc_row + ja;
    int left = (int)(jb - ja);
    if (R > U) {
      constexpr int HR = Log2<R>::v;
      for (; left >= R; left -= R) {
        const T xl = (lane < R) ? Ops<T>::load(xp + lane * incx) : Ops<T>::zero();
        T cp[R];
        // one load step per iteration (not unrolled, so that no more than U
        // columns of loads are held in registers); the column terms move
        // down the cp window by U per step, so that after R/U steps cp[i]
        // holds column i
#pragma unroll 1
        for (int s = 0; s < R / U; ++s) {
          T a[U][VR][VPL];
          load_cols<ALIGNED>(col, lda, a);
#pragma unroll
          for (int i = 0; i < R - U; ++i) cp[i] = cp[i + U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const T xj = Ops<T>::shfl(xl, s * U + u);
            T c = Ops<T>::zero();
#pragma unroll
            for (int v = 0; v < VR; ++v)
#pragma unroll
              for (int k = 0; k < VPL; ++k) {
                racc[v][k] = Ops<T>::madd(racc[v][k], a[u][v][k], xj);
                c = Ops<T>::maddc(c, a[u][v][k], xi[v][k]);
              }
            cp[R - U + u] = c;
          }
          col += U * lda;
        }
        const T red = reduce_scatter<T, R>(cp, lane);
        if ((lane & ((32 >> HR) - 1)) == 0) wc[lane >> (5 - HR)] = red;
        xp += R * incx;
        wc += R;
      }
    }
    for (; left >= U; left -= U) {
      const T xl = (lane < U) ? Ops<T>::load(xp + lane * incx) : Ops<T>::zero();
      T a[U][VR][VPL];
      load_cols<ALIGNED>(col, lda, a);
      accumulate(a, xl, U, wc, lane);
      col += U * lda;
      xp += U * incx;
      wc += U;
    }
    if (left > 0) masked_cols<false>(A, lda, x, incx, r0, jb - left, jb, wc_row, lane, 0, 0);
  }

  // ---- the general product (no symmetry): row terms only ----

  // Columns [ja, jb) of the block row at r0 with all NB rows inside the
  // matrix: racc += A(rows, j) * x(j), the same loads as dense_cols.
  template <bool ALIGNED>
  __device__ __forceinline__ void dense_rows(const T* __restrict__ A, long long lda,
                                             const T* __restrict__ x, int incx, long long r0,
                                             long long ja, long long jb, int lane) {
    const T* col = A + ja * lda + r0 + lane_row(0, lane, 0);
    const T* xp = x + ja * (long long)incx;
    int left = (int)(jb - ja);
    for (; left >= U; left -= U) {
      const T xl = (lane < U) ? Ops<T>::load(xp + lane * incx) : Ops<T>::zero();
      T a[U][VR][VPL];
      load_cols<ALIGNED>(col, lda, a);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const T xj = Ops<T>::shfl(xl, u);
#pragma unroll
        for (int v = 0; v < VR; ++v)
#pragma unroll
          for (int k = 0; k < VPL; ++k) racc[v][k] = Ops<T>::madd(racc[v][k], a[u][v][k], xj);
      }
      col += U * lda;
      xp += U * incx;
    }
    if (left > 0) masked_rows(A, lda, x, incx, r0, jb - left, jb, lane, NB);
  }

  // Columns [ja, jb) of the block row at r0, rows r0 .. r0 + nl - 1 only
  // (nl <= NB): element loads, U columns per step.
  __device__ __forceinline__ void masked_rows(const T* __restrict__ A, long long lda,
                                              const T* __restrict__ x, int incx, long long r0,
                                              long long ja, long long jb, int lane, int nl) {
    const T* col = A + ja * lda + r0;
#pragma unroll 1
    for (long long j0 = ja; j0 < jb; j0 += U, col += U * lda) {
      const int cnt = (int)((jb - j0) < U ? (jb - j0) : U);
      const T xl = (lane < cnt) ? Ops<T>::load(x + (j0 + lane) * incx) : Ops<T>::zero();
      const T* c = col;
#pragma unroll
      for (int u = 0; u < U; ++u, c += lda) {
        const T xj = Ops<T>::shfl(xl, u);
#pragma unroll
        for (int v = 0; v < VR; ++v)
#pragma unroll
          for (int k = 0; k < VPL; ++k) {
            const int rl = lane_row(v, lane, k);
            if (u < cnt && rl < nl)
              racc[v][k] = Ops<T>::madd(racc[v][k], Ops<T>::load(c + rl), xj);
          }
      }
    }
  }

  // issue the bulk copies of chunk c (columns ja + c*U ..) into its stage
  template <int STAGES>
  __device__ __forceinline__ static void ring_fill(const Ring& rg, long long c,
                                                   const T* __restrict__ A, long long lda,
                                                   long long r0, long long ja, long long jb,
                                                   int lane) {
    constexpr int COL_BYTES = NB * (int)sizeof(T);
    const int st = (int)((rg.head + c) % STAGES);
    const long long j0 = ja + c * U;
    const int cnt = (int)((jb - j0) < U ? (jb - j0) : U);
    const uint32_t bar = rg.bars + 8u * st;
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(cnt * COL_BYTES) + rg.extra_tx);
    __syncwarp();
    if (lane < cnt)
      bulk_g2s(rg.data + (uint32_t)(st * U + lane) * COL_BYTES, A + (j0 + lane) * lda + r0,
               COL_BYTES, bar);
  }

  // Columns [ja, jb) of the block row at r0 (all NB rows stored, 16-byte
  // aligned), streamed through the warp's ring.  Returns false if a wait ran
  // out (after draining the copies still in flight).
  template <int STAGES>
  __device__ __forceinline__ bool dense_cols_ring(Ring& rg, const T* __restrict__ A,
                                                  long long lda, const T* __restrict__ x,
                                                  int incx, long long r0, long long ja,
                                                  long long jb, T* wc_row, int lane,
                                                  unsigned long long limit_ns) {
    constexpr int COL_BYTES = NB * (int)sizeof(T);
    const long long nch = (jb - ja + U - 1) / U;
    for (long long c = 0; c < nch && c < STAGES; ++c)
      ring_fill<STAGES>(rg, c, A, lda, r0, ja, jb, lane);
    // x of the chunk's columns, loaded two chunks ahead so that its L2
    // latency overlaps the waits and arithmetic of the chunks before
    auto load_x = [&](long long c) -> T {
      const long long j0 = ja + c * U;
      return (c < nch && lane < U && j0 + lane < jb) ? Ops<T>::load(x + (j0 + lane) * incx)
                                                     : Ops<T>::zero();
    };
    T x_next = load_x(0);
    T x_after = load_x(1);
    for (long long c = 0; c < nch; ++c) {
      const int st = (int)((rg.head + c) % STAGES);
      const uint32_t par = (rg.phase >> st) & 1u;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(rg.bars + 8u * st, par, limit_ns));
      if (!ok) {
        // drain: every chunk c .. min(c+STAGES, nch)-1 has copies in flight
        for (long long k = c; k < nch && k < c + STAGES; ++k) {
          const int s2 = (int)((rg.head + k) % STAGES);
          mbar_wait_bounded(rg.bars + 8u * s2, (rg.phase >> s2) & 1u, limit_ns);
        }
        return false;
      }
      rg.phase ^= 1u << st;
      const long long j0 = ja + c * U;
      const int cnt = (int)((jb - j0) < U ? (jb - j0) : U);
      const T xl = x_next;
      x_next = x_after;
      x_after = load_x(c + 2);
      T a[U][VR][VPL];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int v = 0; v < VR; ++v) {
          if (u < cnt) {
            const uint4 raw = lds128(rg.data + (uint32_t)(st * U + u) * COL_BYTES +
                                     (uint32_t)(v * 32 + lane) * 16u);
            Unpack<T>::run(raw, a[u][v]);
          } else {
#pragma unroll
            for (int k = 0; k < VPL; ++k) a[u][v][k] = Ops<T>::zero();
          }
        }
      // the stage is refilled only after its values have been used by the
      // arithmetic, so the asynchronous write cannot overtake the reads
      accumulate(a, xl, cnt, wc_row + j0, lane);
      __syncwarp();
      if (c + STAGES < nch) ring_fill<STAGES>(rg, c + STAGES, A, lda, r0, ja, jb, lane);
    }
    rg.head = (int)((rg.head + nch) % STAGES);
    return true;
  }

  // Columns [ja, jb) with per-element masks: rows must be < n and, when
  // DIAG, inside the stored triangle (upper: row <= col; lower: row >= col).
  // On the diagonal only the row term is taken (and for a Hermitian matrix
  // only the real part of the element).  UD columns per step (U, like the
  // dense loop, unless the caller asks for fewer), so that diagonal tiles
  // keep loads in flight and do not hold their warps back; each element
  // address is a running column pointer plus a constant.
  //
  // VEC (16-byte aligned matrices): a lane's VPL consecutive rows that are
  // all below row n and hold at least one element inside the mask are read
  // as one 16-byte vector, the way dense columns are; a vector that crosses
  // the diagonal then also brings the up to VPL - 1 elements beside it on
  // the other side (in the same 32-byte sector, inside the caller's array:
  // rows < n <= lda), which are never used.  Per element loads, the
  // diagonal tiles issued VPL times the requests per byte of the dense
  // columns, and their warps fell behind when the tiles came from DRAM.
  // Without VEC, elements outside the mask are never read.  The arithmetic,
  // and so the rounding, is the same either way.
  template <bool DIAG, bool VEC = false, int UD = U>
  __device__ __forceinline__ void masked_cols(const T* __restrict__ A, long long lda,
                                              const T* __restrict__ x, int incx, long long r0,
                                              long long ja, long long jb, T* wc_row, int lane,
                                              long long n, int upper) {
    const T* col = A + ja * lda + r0;
    // rows and columns relative to r0 fit in 32 bits (|j - r0| < n)
    const int nl = (int)((n - r0) < NB ? (n - r0) : NB);
#pragma unroll 1
    for (long long j0 = ja; j0 < jb; j0 += UD, col += UD * lda) {
      const int cnt = (int)((jb - j0) < UD ? (jb - j0) : UD);
      const int jl0 = (int)(j0 - r0);
      const T xl = (lane < cnt) ? Ops<T>::load(x + (j0 + lane) * incx) : Ops<T>::zero();
      // VEC: the step's vectors, all issued before the arithmetic (as in
      // the dense loop); a vector below row n but wholly outside the mask is
      // not read (zeros stand in)
      uint4 raw[VEC ? UD : 1][VEC ? VR : 1];
      if (VEC) {
        const T* c = col;
#pragma unroll
        for (int u = 0; u < UD; ++u, c += lda)
#pragma unroll
          for (int v = 0; v < VR; ++v) {
            const int rl0 = lane_row(v, lane, 0);
            const int jl = jl0 + u;
            const bool need = u < cnt && rl0 + VPL <= nl &&
                              (!DIAG || (upper ? rl0 <= jl : rl0 + VPL - 1 >= jl));
            raw[VEC ? u : 0][VEC ? v : 0] = need ? ldg_stream16(c + rl0) : make_uint4(0u, 0u, 0u, 0u);
          }
      }
      T cp[UD];
      const T* c = col;
#pragma unroll
      for (int u = 0; u < UD; ++u, c += lda) {
        const int jl = jl0 + u;
        const T xj = Ops<T>::shfl(xl, u);
        T cu = Ops<T>::zero();
#pragma unroll
        for (int v = 0; v < VR; ++v) {
          T av[VPL];
          if (VEC) Unpack<T>::run(raw[VEC ? u : 0][VEC ? v : 0], av);
          const bool whole = VEC && lane_row(v, lane, 0) + VPL <= nl;   // read as a vector
#pragma unroll
          for (int k = 0; k < VPL; ++k) {
            const int rl = lane_row(v, lane, k);
            bool valid = u < cnt;
            if (DIAG) valid = valid && rl < nl && (upper ? rl <= jl : rl >= jl);
            if (valid) {
              T a = whole ? av[k] : Ops<T>::load(c + rl);
              if (DIAG && rl == jl) {
                racc[v][k] = Ops<T>::madd(racc[v][k], Ops<T>::diag(a), xj);
              } else {
                racc[v][k] = Ops<T>::madd(racc[v][k], a, xj);
                cu = Ops<T>::maddc(cu, a, xi[v][k]);
              }
            }
          }
        }
        cp[u] = cu;
      }
      T red = reduce_scatter<T, UD>(cp, lane);
      constexpr int HD = Log2<UD>::v;
      const int uo = lane >> (5 - HD);
      if ((lane & ((32 >> HD) - 1)) == 0 && uo < cnt) wc_row[j0 + uo] = red;
    }
  }
};

// ----------------------------------------------------------------------------
// the plan's warp and row tables (see xsymv_plan.h), once per plan
// ----------------------------------------------------------------------------
static __global__ void symv_plan_tables(Plan p, int4* __restrict__ wt, int2* __restrict__ rt) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < p.W) {
    int Ia, Ib;
    long long ja, jb;
    plan_warp_entry(p, (int)t, &Ia, &Ib, &ja, &jb);
    wt[t] = make_int4(Ia, Ib, (int)ja, (int)jb);
  }
  if (t < p.nb) {
    const int nq = plan_nq(p, (int)t);   // 0: a row outside the column window
    rt[t] = make_int2(nq > 0 ? plan_first_owner(p, (int)t) / p.G : 0, nq);
  }
}

// ----------------------------------------------------------------------------
// row partials: one slot per thread block and block row
// ----------------------------------------------------------------------------
// A warp's row partials of its first and last block rows go to its two
// shared-memory buffers; the row partials of the rows strictly between (rows
// no other warp touches) go straight to the block's slot.  After the block's
// warps are done, the block adds the buffers of each row in warp order and
// writes the sum to its slot (row_partials_combine).
template <class T, int NB, int WARPS>
struct RowBuffers {
  T buf[WARPS][2][NB];   // [warp][first / last row][row within the block row]
  int row[WARPS][2];     // block row held by each buffer, -1: none
};

// block b's slot of block row I (first block of the row: rt[I].x)
template <class T>
__device__ __forceinline__ T* row_slot(const Plan& p, T* Wr, const int2* __restrict__ rt, int b,
                                       int I) {
  return Wr + ((long long)I * p.qmax + (b - __ldg(&rt[I].x))) * p.NB;
}

// All threads of the block, after a barrier that follows every warp's
// stream: the rows of the buffers, in increasing order, each summed over the
// warps in warp order and written to block b's slot.
template <class T, int NB, int WARPS>
__device__ __forceinline__ void row_partials_combine(const Plan& p, T* Wr,
                                                     const int2* __restrict__ rt, int b,
                                                     const RowBuffers<T, NB, WARPS>& rb) {
  int lo = 0x7fffffff, hi = -1;
#pragma unroll
  for (int w = 0; w < WARPS; ++w)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int I = rb.row[w][k];
      if (I >= 0) {
        lo = I < lo ? I : lo;
        hi = I > hi ? I : hi;
      }
    }
  for (int I = lo; I <= hi; ++I) {
    T* slot = nullptr;
    for (int r = threadIdx.x; r < NB; r += blockDim.x) {
      T s = Ops<T>::zero();
      bool has = false;
#pragma unroll
      for (int w = 0; w < WARPS; ++w)
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (rb.row[w][k] == I) {
            const T v = rb.buf[w][k][r];
            s = has ? Ops<T>::add(s, v) : v;
            has = true;
          }
      if (has) {
        if (slot == nullptr) slot = row_slot(p, Wr, rt, b, I);
        slot[r] = s;
      }
    }
  }
}

// ----------------------------------------------------------------------------
// one warp's share of the triangle
// ----------------------------------------------------------------------------
// For every block row I in which warp w (warp wl of block b) owns columns
// (from the plan's warp table wt; row table rt): the columns of the diagonal
// tile (masked), then the off-diagonal ones (through the ring when RING,
// else straight into registers), column partials to Wc[I*n + j], then the
// row partial: to the warp's buffer in rb for its first and last rows, to
// block b's slot in Wr for the rows between.  Returns false if a bounded
// wait of the ring ran out (the warp then stops at once).
template <class T, int VR, int U, int STAGES, bool RING, bool ALIGNED, int R, int WARPS>
__device__ __forceinline__ bool stream_warp(const Plan& p, int w, int wl, int b, int lane,
                                            Ring& rg, const T* __restrict__ A, long long lda,
                                            const T* __restrict__ x, int incx,
                                            T* __restrict__ Wc, T* __restrict__ Wr,
                                            const int4* __restrict__ wt,
                                            const int2* __restrict__ rt,
                                            RowBuffers<T, WarpTile<T, VR, U>::NB, WARPS>& rb,
                                            unsigned long long limit_ns) {
  using Tile = WarpTile<T, VR, U>;
  constexpr int VPL = Tile::VPL;
  constexpr int NB = Tile::NB;
  // columns per step in the diagonal tiles: one for the single-precision
  // kinds read as vectors (with U columns the step's vectors and masks
  // spilled under those kernels' register caps), U otherwise
  constexpr bool kSingle = std::is_same<T, float>::value || std::is_same<T, c32>::value;
  constexpr int UD = (ALIGNED && kSingle) ? 1 : U;
  const int4 d = __ldg(wt + w);   // rows d.x .. d.y, from column d.z to column d.w
  const long long n = p.n;
  Tile t;

  for (int I = d.x; I <= d.y; ++I) {
    const long long cb = plan_colbase(p, I);
    const long long ja = I == d.x ? (long long)d.z : cb;
    const long long jb = I == d.y ? (long long)d.w : cb + plan_rowlen(p, I);
    if (ja >= jb) continue;   // no column of this row starts in the range
    const long long r0 = (long long)I * NB;

#pragma unroll
    for (int v = 0; v < VR; ++v)
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        const long long r = r0 + Tile::lane_row(v, lane, k);
        t.xi[v][k] = (r < n) ? Ops<T>::load(x + r * incx) : Ops<T>::zero();
        t.racc[v][k] = Ops<T>::zero();
      }

    T* wc_row = Wc + (long long)I * n;
    const long long dA = r0;
    const long long dB = (r0 + NB < n) ? r0 + NB : n;   // diagonal tile columns [dA, dB)
    // the diagonal tile's columns of this segment first (masked), then the
    // off-diagonal ones: upper [max(ja,dB), jb), lower [ja, min(jb,dA)), so
    // that nothing but the row terms is live after the long dense loop
    const long long a0 = ja > dA ? ja : dA;
    const long long a1 = p.upper ? (jb < dB ? jb : dB) : jb;
    if (a0 < a1)
      t.template masked_cols<true, ALIGNED, UD>(A, lda, x, incx, r0, a0, a1, wc_row, lane, n, p.upper);
    const long long b0 = p.upper ? (ja > dB ? ja : dB) : ja;
    const long long b1 = p.upper ? jb : (jb < dA ? jb : dA);
    if (b0 < b1) {
      if (r0 + NB > n) {
        // a last, incomplete block row (lower storage only): rows masked
        t.template masked_cols<true, ALIGNED, UD>(A, lda, x, incx, r0, b0, b1, wc_row, lane, n, 0);
      } else if (RING) {
        if (!t.template dense_cols_ring<(STAGES > 0 ? STAGES : 1)>(rg, A, lda, x, incx, r0, b0, b1,
                                                                   wc_row, lane, limit_ns))
          return false;
      } else {
        t.template dense_cols<ALIGNED, R>(A, lda, x, incx, r0, b0, b1, wc_row, lane);
      }
    }

    // the row partial: rows between the first and the last are this warp's
    // alone (straight to the block's slot); the first and last rows are
    // shared with other warps (to this warp's buffers, combined later)
    const int k = I == d.x ? 0 : (I == d.y ? 1 : -1);
    T* wr = k < 0 ? row_slot(p, Wr, rt, b, I) : rb.buf[wl][k];
#pragma unroll
    for (int v = 0; v < VR; ++v)
#pragma unroll
      for (int kk = 0; kk < VPL; ++kk) wr[Tile::lane_row(v, lane, kk)] = t.racc[v][kk];
    if (k >= 0 && lane == 0) rb.row[wl][k] = I;
  }
  return true;
}

// ----------------------------------------------------------------------------
// main kernel
// ----------------------------------------------------------------------------
// PIPE (see enum Pipe) applies to 16-byte aligned matrices; otherwise
// off-diagonal columns are read with element loads.  Dynamic shared memory
// = WARPS * RingLayout::WARP_BYTES.  MINB > 0 asks the compiler to fit MINB
// blocks per SM (a register cap); 0 leaves the choice to the compiler.  R:
// columns per batched column reduction on the register path (R = U: none).
template <class T, int VR, int U, int STAGES, int PIPE, int WARPS, bool ALIGNED, int MINB,
          int R = U>
__global__ void __launch_bounds__(WARPS * 32, MINB)
symv_main(Plan p, const T* __restrict__ A, long long lda, const T* __restrict__ x, int incx,
          T* __restrict__ Wc, T* __restrict__ Wr, const int4* __restrict__ wt,
          const int2* __restrict__ rt, int* status, int epoch, unsigned long long limit_ns,
          uint32_t extra_tx, int early) {
  using Lay = RingLayout<T, VR, U, STAGES, PIPE>;
  constexpr bool RING = (PIPE == kPipeBulk) && ALIGNED;
  __shared__ RowBuffers<T, WarpTile<T, VR, U>::NB, WARPS> rb;
  // let the finaliser (launched as a programmatic dependent) get scheduled as
  // blocks of this grid retire; it waits for this grid's completion itself
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int wl = threadIdx.x >> 5;
  const int w = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  if (lane < 2) rb.row[wl][lane] = -1;
  __syncwarp();

  Ring rg{0u, 0u, 0, 0u, extra_tx};
  if (RING && w < p.W) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* base = smem + (size_t)wl * Lay::WARP_BYTES;
    rg.data = smem_addr(base);
    rg.bars = smem_addr(base + Lay::DATA_BYTES);
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < (STAGES > 0 ? STAGES : 1); ++s) mbar_init(rg.bars + 8u * s, 1);
      mbar_init_fence();
    }
    __syncwarp();
  }
  // launched as a programmatic dependent of the stream's previous kernel
  // (the previous call's finaliser lets it start early): nothing of global
  // memory is touched before that kernel has completed -- unless `early`:
  // the host has checked that the previous kernel is a finaliser whose
  // writes (its y) miss A and x, and this call's partial sums go to the other
  // half of the workspace, so the stream can start at once; the wait then
  // comes at the end, so that this grid completes only after that finaliser
  // (the next kernels' ordering rests on it)
  if (!early) asm volatile("griddepcontrol.wait;" ::: "memory");
  // an early grid notes when it began, in the header word of its call's
  // parity (the finaliser compares it with the previous finaliser's end)
  if (early && blockIdx.x == 0 && threadIdx.x == 0)
    note_time(reinterpret_cast<char*>(status) + kOverlapOffset + 8 * (2 + (epoch & 1)));
  bool ok = true;
  if (w < p.W)
    ok = stream_warp<T, VR, U, STAGES, RING, ALIGNED, R, WARPS>(p, w, wl, blockIdx.x, lane, rg, A,
                                                                lda, x, incx, Wc, Wr, wt, rt, rb,
                                                                limit_ns);
  if (!ok && lane == 0) atomicMax(status, epoch);   // (its row buffers are incomplete: y is NaN)
  __syncthreads();
  row_partials_combine<T, WarpTile<T, VR, U>::NB, WARPS>(p, Wr, rt, blockIdx.x, rb);
  if (early) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ----------------------------------------------------------------------------
// finalize: y := alpha * (fixed-order sum of the workspace slots) + beta * y
// ----------------------------------------------------------------------------
// What the final merge writes: y = alpha*s + beta*y (kFull), alpha*s
// (kBetaZero), beta*y (kAlphaZero), 0 (kZero), or the sum s itself
// (kPartial: one shard's partial vector, merged later by symv_reduce).
enum FinalMode { kFull = 0, kBetaZero = 1, kAlphaZero = 2, kZero = 3, kPartial = 4 };

// the merged output of one element (shared by the finaliser and the
// reduction of shards, so both round alike)
template <class T>
__device__ __forceinline__ T final_value(int mode, T alpha, T s, T beta, T y_old) {
  if (mode == kFull) return Ops<T>::add(Ops<T>::mul(alpha, s), Ops<T>::mul(beta, y_old));
  if (mode == kBetaZero) return Ops<T>::mul(alpha, s);
  if (mode == kAlphaZero) return Ops<T>::mul(beta, y_old);
  if (mode == kPartial) return s;
  return Ops<T>::zero();
}

constexpr int kFinParts = 8;    // partial sums per output element (the combination order
                                // below depends on it: changing it changes the rounding)
constexpr int kFinCols = 32;    // output elements per block

// a workspace element written by this kernel's other blocks (COHERENT: read
// at the L2, never from a possibly stale L1 or the read-only path) or by an
// earlier kernel
template <bool COHERENT, class T>
__device__ __forceinline__ T ld_ws(const T* p) {
  static_assert(sizeof(T) == 4 || sizeof(T) == 8 || sizeof(T) == 16, "element size");
  T r;
  if (sizeof(T) == 4) {
    const unsigned* q = reinterpret_cast<const unsigned*>(p);
    const unsigned b = COHERENT ? __ldcg(q) : __ldg(q);
    memcpy(&r, &b, sizeof(T));
  } else if (sizeof(T) == 8) {
    const unsigned long long* q = reinterpret_cast<const unsigned long long*>(p);
    const unsigned long long b = COHERENT ? __ldcg(q) : __ldg(q);
    memcpy(&r, &b, sizeof(T));
  } else {
    const ulonglong2* q = reinterpret_cast<const ulonglong2*>(p);
    const ulonglong2 b = COHERENT ? __ldcg(q) : __ldg(q);
    memcpy(&r, &b, sizeof(T));
  }
  return r;
}

// Outputs fb*kFinCols .. fb*kFinCols + kFinCols - 1 (they lie in one block
// row K because NB is a multiple of 32), computed by threads 0 ..
// kFinParts*kFinCols - 1 of the block; every one of them must call this.
// Thread (part, c) adds, in increasing order, the column partials of block
// rows I = I0+part, I0+part+kFinParts, ... and the row-partial slots q = part,
// part+kFinParts, ...; the kFinParts sums are then added in part order.  The
// order depends only on (n, NB, W), never on timing.
template <class T, bool COHERENT, int LG = 8>
__device__ __forceinline__ void finalize_outputs(const Plan& p, const T* Wc, const T* Wr,
                                                 const int2* __restrict__ rt, T alpha, T beta,
                                                 int mode, T* y, long long incy,
                                                 const int* status, int epoch, long long fb,
                                                 T (&part)[kFinParts][kFinCols]) {
  const int c = threadIdx.x % kFinCols;
  const int pp = threadIdx.x / kFinCols;
  const long long j = fb * kFinCols + c;
  const bool live = j < p.n;
  T* yj = y + j * incy;
  // y, and the first row-partial slot, are loaded up front so that their
  // latency overlaps the column-partial loads
  const bool need_y = live && pp == 0 && (mode == kFull || mode == kAlphaZero);
  const T y_old = need_y ? *yj : Ops<T>::zero();
  T s = Ops<T>::zero();
  if (live && (mode == kFull || mode == kBetaZero || mode == kPartial)) {
    const int K = (int)(j / p.NB);
    const int jj = (int)(j - (long long)K * p.NB);
    // column partials exist only for the window's columns
    const bool in_window = j >= p.c0 && j < p.c1;
    const int I0 = p.upper ? 0 : K;
    const int I1 = !in_window ? I0 - 1 : (p.upper ? K : p.nb - 1);
    const int nq = __ldg(&rt[K].y);
    const T* wr = Wr + (long long)K * p.qmax * p.NB + jj;
    const T wr_first = pp < nq ? ld_ws<COHERENT>(wr + (long long)pp * p.NB) : Ops<T>::zero();
    const T* wc = Wc + j;
    // column partials I = I0+pp, I0+pp+kFinParts, ... <= I1, then row
    // partials q = pp, pp+kFinParts, ... < nq, added in that order; loads
    // are issued LG at a time (the last group predicated), so a thread waits
    // for about (count / LG) memory round trips (LG does not change the order
    // of the additions)
    for (int I = I0 + pp; I <= I1; I += LG * kFinParts) {
      T v[LG];
#pragma unroll
      for (int k = 0; k < LG; ++k)
        v[k] = (I + k * kFinParts <= I1) ? ld_ws<COHERENT>(wc + (long long)(I + k * kFinParts) * p.n)
                                         : Ops<T>::zero();
#pragma unroll
      for (int k = 0; k < LG; ++k)
        if (I + k * kFinParts <= I1) s = Ops<T>::add(s, v[k]);
    }
    if (pp < nq) s = Ops<T>::add(s, wr_first);
    for (int q = pp + kFinParts; q < nq; q += LG * kFinParts) {
      T v[LG];
#pragma unroll
      for (int k = 0; k < LG; ++k)
        v[k] = (q + k * kFinParts < nq) ? ld_ws<COHERENT>(wr + (long long)(q + k * kFinParts) * p.NB)
                                        : Ops<T>::zero();
#pragma unroll
      for (int k = 0; k < LG; ++k)
        if (q + k * kFinParts < nq) s = Ops<T>::add(s, v[k]);
    }
  }
  part[pp][c] = s;
  __syncthreads();
  if (pp == 0 && live) {
    s = part[0][c];
#pragma unroll
    for (int k = 1; k < kFinParts; ++k) s = Ops<T>::add(s, part[k][c]);
    T out = final_value(mode, alpha, s, beta, y_old);
    if (status != nullptr && (COHERENT ? __ldcg(status) : *status) == epoch)
      out = Ops<T>::nan();   // the main kernel (or this kernel's grid barrier) gave up
    *yj = out;
  }
}

// Words of the stream workspace's header through which back-to-back calls
// learn whether they overlap (all null: not used): `end` receives the end
// time of this call's last kernel (finaliser, or one-launch kernel); when
// `report` is set, `prev_end` holds the previous call's end time and
// *report (host-mapped) gets 1 if this call ran back to back with it: for a
// finaliser, its call's main kernel started early and `start` holds that
// start time, which must precede `prev_end`; a one-launch kernel compares
// its own start with `prev_end` (kBackToBackNs).
struct OverlapWords {
  unsigned long long* end;
  const unsigned long long* start;
  const unsigned long long* prev_end;
  int* report;
};

// Block (kFinParts x kFinCols threads) b handles the groups of outputs
// fb*32 .. fb*32+31 for fb = b, b + grid, ...
template <class T>
__global__ void __launch_bounds__(kFinParts * kFinCols)
symv_finalize(Plan p, const T* __restrict__ Wc, const T* __restrict__ Wr,
              const int2* __restrict__ rt, T alpha, T beta, int mode, T* __restrict__ y,
              long long incy, const int* status, int epoch, OverlapWords ow) {
  __shared__ T part[kFinParts][kFinCols];
  // the next call's main kernel, a programmatic dependent, may be scheduled
  // once every block of this grid runs; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // wait until the preceding grid on the stream (the main kernel) has
  // completed and its writes are visible (no-op without a programmatic launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // after an early main kernel: did it start before the previous finaliser
  // ended (nothing else ran between the two calls)?  The host reads the
  // answer when it enqueues later calls, and gives their finalisers the
  // compact grid while the answer is yes
  if (ow.report != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    const unsigned long long began = *reinterpret_cast<const volatile unsigned long long*>(ow.start);
    const unsigned long long ended = *reinterpret_cast<const volatile unsigned long long*>(ow.prev_end);
    *reinterpret_cast<volatile int*>(ow.report) = began < ended ? 1 : 0;
  }
  const long long nfb = (p.n + kFinCols - 1) / kFinCols;
  for (long long fb = blockIdx.x; fb < nfb; fb += gridDim.x) {
    finalize_outputs<T, false>(p, Wc, Wr, rt, alpha, beta, mode, y, incy, status, epoch, fb, part);
    __syncthreads();   // (part is reused by the next group)
  }
  // the time the grid's last block ends (a reduction nobody waits for): the
  // next call's finaliser compares it with the start of that call's main kernel
  if (ow.end != nullptr && threadIdx.x == 0) atomicMax(ow.end, global_ns());
}

// ----------------------------------------------------------------------------
// reduce: the shards' partial vectors summed in rank order, then merged
// ----------------------------------------------------------------------------
// y(i) := alpha * (P_0(i) + P_1(i) + ... + P_{N-1}(i)) + beta * y(i), the sum
// taken left to right in part (rank) order, P_r(i) at P[r*ldp + i]: the
// block-column split of the stored triangle across GPUs reduced in one fixed
// order, so the result is bit-identical from run to run.  One thread per
// output element; the parts' loads are issued 8 at a time.
constexpr int kReduceThreads = 256;

template <class T>
__global__ void __launch_bounds__(kReduceThreads)
symv_reduce(int n, int nparts, const T* __restrict__ P, long long ldp, T alpha, T beta, int mode,
            T* __restrict__ y, long long incy) {
  const long long i = (long long)blockIdx.x * kReduceThreads + threadIdx.x;
  if (i >= n) return;
  T* yi = y + i * incy;
  const T y_old = (mode == kFull || mode == kAlphaZero) ? *yi : Ops<T>::zero();
  T s = Ops<T>::zero();
  if (mode == kFull || mode == kBetaZero) {
    for (int r0 = 0; r0 < nparts; r0 += 8) {
      T v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = r0 + k < nparts ? P[(long long)(r0 + k) * ldp + i] : Ops<T>::zero();
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (r0 + k < nparts) s = (r0 + k == 0) ? v[k] : Ops<T>::add(s, v[k]);
    }
  }
  *yi = final_value(mode, alpha, s, beta, y_old);
}

}  // namespace xsymv
