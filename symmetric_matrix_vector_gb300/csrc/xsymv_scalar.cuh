// Scalar types of the five xSYMV / xHEMV variants and the few operations the
// kernels need on them: zero, add, the two multiply-adds of a stored element
// (row term A(i,j)*x(j) and column term conj(A(i,j))*x(i)), warp shuffles and
// 16-byte streaming loads.
//
// Types (as listed in §2.2 and figure "x-symv API" of "CUDA-xSYMV の実装と
// 評価", IPSJ 2014-HPC-146): float, double, single and double complex
// (float2 / double2 layout) and double-double (a double2 holding hi + lo).
//
// Double-double follows Hida, Li and Bailey's quad-double paper (the report's
// reference for its DD format): TwoSum, QuickTwoSum, TwoProd through FMA, and
// the accurate ("IEEE") addition.  Every DD step uses the explicitly rounded
// intrinsics so the compiler can neither contract nor reassociate it.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace xsymv {

struct c32 { float re, im; };
struct c64 { double re, im; };
struct dd { double hi, lo; };

// ---------------------------------------------------------------- DD core --
// The rounded sum, difference and product of two doubles, as the DD steps
// use them.  They are issued as fused multiply-adds with a unit operand held
// in a register: fma(a, 1, b), fma(b, -1, a) and fma(a, b, -0) round the
// exact a + b, a - b and a * b once, as the plain instructions do (signed
// zeros included: x + (-0) = x), so every DD result is bit-identical; but
// on GB300 a register-operand DFMA occupies the FP64 pipe for fewer cycles
// than a DADD or DMUL (measured: 2.0 against 1.68 instructions per clock
// per SM), which makes the DD kernels about 14 % faster.  Built with
// XSYMV_DD_FMA=0 they use the plain instructions instead.
#ifndef XSYMV_DD_FMA
#define XSYMV_DD_FMA 1
#endif
#if XSYMV_DD_FMA
// +1, -1, -0 in global memory, read by an opaque load: the compiler must
// not learn their values, or it turns fma(a, b, -0) back into a product and
// fma(x, 1, y) into a sum, which it may then contract into one fused
// operation (a different rounding).  The load has no side effects, so it is
// hoisted out of loops and the units stay in registers.
static __device__ double g_dd_units[3] = {1.0, -1.0, -0.0};
__device__ __forceinline__ double dd_unit(int i) {
  double v;
  asm("ld.global.nc.f64 %0, [%1];" : "=d"(v) : "l"(g_dd_units + i));
  return v;
}
__device__ __forceinline__ double d_add(double a, double b) { return __fma_rn(a, dd_unit(0), b); }
__device__ __forceinline__ double d_sub(double a, double b) { return __fma_rn(b, dd_unit(1), a); }
__device__ __forceinline__ double d_mul(double a, double b) { return __fma_rn(a, b, dd_unit(2)); }
#else
__device__ __forceinline__ double d_add(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ double d_sub(double a, double b) { return __dsub_rn(a, b); }
__device__ __forceinline__ double d_mul(double a, double b) { return __dmul_rn(a, b); }
#endif
__device__ __forceinline__ double d_fma(double a, double b, double c) { return __fma_rn(a, b, c); }

__device__ __forceinline__ void two_sum(double a, double b, double& s, double& e) {
  s = d_add(a, b);
  double bb = d_sub(s, a);
  e = d_add(d_sub(a, d_sub(s, bb)), d_sub(b, bb));
}
__device__ __forceinline__ void quick_two_sum(double a, double b, double& s, double& e) {
  s = d_add(a, b);
  e = d_sub(b, d_sub(s, a));
}
__device__ __forceinline__ dd dd_add(dd a, dd b) {
  double s1, s2, t1, t2;
  two_sum(a.hi, b.hi, s1, s2);
  two_sum(a.lo, b.lo, t1, t2);
  s2 = d_add(s2, t1);
  quick_two_sum(s1, s2, s1, s2);
  s2 = d_add(s2, t2);
  quick_two_sum(s1, s2, s1, s2);
  return dd{s1, s2};
}
__device__ __forceinline__ dd dd_mul(dd a, dd b) {
  double p = d_mul(a.hi, b.hi);
  double e = d_fma(a.hi, b.hi, -p);
  e = d_fma(a.hi, b.lo, e);
  e = d_fma(a.lo, b.hi, e);
  double s, t;
  quick_two_sum(p, e, s, t);
  return dd{s, t};
}
// acc + a*b: TwoProd with FMA gives the high parts' product exactly as
// p + e, the cross terms a.hi*b.lo and a.lo*b.hi are folded into e, and the
// pair (p, e) goes straight into the accurate addition, whose TwoSum steps
// absorb an e slightly above half an ulp of p; renormalising the product
// first (dd_mul's QuickTwoSum) would cost three more operations and change
// nothing the addition does not already do.
__device__ __forceinline__ dd dd_madd(dd acc, dd a, dd b) {
  const double p = d_mul(a.hi, b.hi);
  double e = d_fma(a.hi, b.hi, -p);
  e = d_fma(a.hi, b.lo, e);
  e = d_fma(a.lo, b.hi, e);
  return dd_add(acc, dd{p, e});
}
__device__ __forceinline__ dd dd_renorm(dd a) {
  dd r;
  quick_two_sum(a.hi, a.lo, r.hi, r.lo);
  return r;
}

// --------------------------------------------------------------- traits ----
// VPL: elements per 16-byte vector load.  HERM: complex Hermitian variant.
template <class T> struct Ops;

template <> struct Ops<float> {
  static constexpr int VPL = 4;
  static constexpr bool HERM = false;
  __device__ __forceinline__ static float zero() { return 0.f; }
  __device__ __forceinline__ static float nan() { return __int_as_float(0x7fffffff); }
  __device__ __forceinline__ static float add(float a, float b) { return a + b; }
  __device__ __forceinline__ static float mul(float a, float b) { return a * b; }
  // acc + a*b and acc + conj(a)*b
  __device__ __forceinline__ static float madd(float acc, float a, float b) { return fmaf(a, b, acc); }
  __device__ __forceinline__ static float maddc(float acc, float a, float b) { return fmaf(a, b, acc); }
  __device__ __forceinline__ static float diag(float a) { return a; }
  __device__ __forceinline__ static float load(const float* p) { return __ldg(p); }
  __device__ __forceinline__ static float shfl_xor(float v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
  __device__ __forceinline__ static float shfl(float v, int src) { return __shfl_sync(0xffffffffu, v, src); }
};

template <> struct Ops<double> {
  static constexpr int VPL = 2;
  static constexpr bool HERM = false;
  __device__ __forceinline__ static double zero() { return 0.0; }
  __device__ __forceinline__ static double nan() { return __longlong_as_double(0x7fffffffffffffffll); }
#if XSYMV_DD_FMA
  // the sums of partial sums (warp reductions, final merge) in the form the
  // FP64 pipe issues fastest; see d_add
  __device__ __forceinline__ static double add(double a, double b) { return d_add(a, b); }
#else
  __device__ __forceinline__ static double add(double a, double b) { return a + b; }
#endif
  __device__ __forceinline__ static double mul(double a, double b) { return a * b; }
  __device__ __forceinline__ static double madd(double acc, double a, double b) { return fma(a, b, acc); }
  __device__ __forceinline__ static double maddc(double acc, double a, double b) { return fma(a, b, acc); }
  __device__ __forceinline__ static double diag(double a) { return a; }
  __device__ __forceinline__ static double load(const double* p) { return __ldg(p); }
  __device__ __forceinline__ static double shfl_xor(double v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
  __device__ __forceinline__ static double shfl(double v, int src) { return __shfl_sync(0xffffffffu, v, src); }
};

template <> struct Ops<c32> {
  static constexpr int VPL = 2;
  static constexpr bool HERM = true;
  __device__ __forceinline__ static c32 zero() { return c32{0.f, 0.f}; }
  __device__ __forceinline__ static c32 nan() { return c32{Ops<float>::nan(), Ops<float>::nan()}; }
  __device__ __forceinline__ static c32 add(c32 a, c32 b) { return c32{a.re + b.re, a.im + b.im}; }
  __device__ __forceinline__ static c32 mul(c32 a, c32 b) {
    return c32{a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
  }
  __device__ __forceinline__ static c32 madd(c32 acc, c32 a, c32 b) {
    acc.re = fmaf(a.re, b.re, acc.re);
    acc.re = fmaf(-a.im, b.im, acc.re);
    acc.im = fmaf(a.re, b.im, acc.im);
    acc.im = fmaf(a.im, b.re, acc.im);
    return acc;
  }
  __device__ __forceinline__ static c32 maddc(c32 acc, c32 a, c32 b) {
    acc.re = fmaf(a.re, b.re, acc.re);
    acc.re = fmaf(a.im, b.im, acc.re);
    acc.im = fmaf(a.re, b.im, acc.im);
    acc.im = fmaf(-a.im, b.re, acc.im);
    return acc;
  }
  // the imaginary part of a Hermitian diagonal is never referenced
  __device__ __forceinline__ static c32 diag(c32 a) { return c32{a.re, 0.f}; }
  // element loads need only the alignment of the component type
  __device__ __forceinline__ static c32 load(const c32* p) {
    const float* f = reinterpret_cast<const float*>(p);
    return c32{__ldg(f), __ldg(f + 1)};
  }
  __device__ __forceinline__ static c32 shfl_xor(c32 v, int m) {
    return c32{__shfl_xor_sync(0xffffffffu, v.re, m), __shfl_xor_sync(0xffffffffu, v.im, m)};
  }
  __device__ __forceinline__ static c32 shfl(c32 v, int s) {
    return c32{__shfl_sync(0xffffffffu, v.re, s), __shfl_sync(0xffffffffu, v.im, s)};
  }
};

template <> struct Ops<c64> {
  static constexpr int VPL = 1;
  static constexpr bool HERM = true;
  __device__ __forceinline__ static c64 zero() { return c64{0.0, 0.0}; }
  __device__ __forceinline__ static c64 nan() { return c64{Ops<double>::nan(), Ops<double>::nan()}; }
  __device__ __forceinline__ static c64 add(c64 a, c64 b) {
    return c64{Ops<double>::add(a.re, b.re), Ops<double>::add(a.im, b.im)};
  }
  __device__ __forceinline__ static c64 mul(c64 a, c64 b) {
    return c64{a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
  }
  __device__ __forceinline__ static c64 madd(c64 acc, c64 a, c64 b) {
    acc.re = fma(a.re, b.re, acc.re);
    acc.re = fma(-a.im, b.im, acc.re);
    acc.im = fma(a.re, b.im, acc.im);
    acc.im = fma(a.im, b.re, acc.im);
    return acc;
  }
  __device__ __forceinline__ static c64 maddc(c64 acc, c64 a, c64 b) {
    acc.re = fma(a.re, b.re, acc.re);
    acc.re = fma(a.im, b.im, acc.re);
    acc.im = fma(a.re, b.im, acc.im);
    acc.im = fma(-a.im, b.re, acc.im);
    return acc;
  }
  __device__ __forceinline__ static c64 diag(c64 a) { return c64{a.re, 0.0}; }
  __device__ __forceinline__ static c64 load(const c64* p) {
    const double* f = reinterpret_cast<const double*>(p);
    return c64{__ldg(f), __ldg(f + 1)};
  }
  __device__ __forceinline__ static c64 shfl_xor(c64 v, int m) {
    return c64{__shfl_xor_sync(0xffffffffu, v.re, m), __shfl_xor_sync(0xffffffffu, v.im, m)};
  }
  __device__ __forceinline__ static c64 shfl(c64 v, int s) {
    return c64{__shfl_sync(0xffffffffu, v.re, s), __shfl_sync(0xffffffffu, v.im, s)};
  }
};

template <> struct Ops<dd> {
  static constexpr int VPL = 1;
  static constexpr bool HERM = false;
  __device__ __forceinline__ static dd zero() { return dd{0.0, 0.0}; }
  __device__ __forceinline__ static dd nan() { return dd{Ops<double>::nan(), Ops<double>::nan()}; }
  __device__ __forceinline__ static dd add(dd a, dd b) { return dd_add(a, b); }
  __device__ __forceinline__ static dd mul(dd a, dd b) { return dd_mul(a, b); }
  __device__ __forceinline__ static dd madd(dd acc, dd a, dd b) { return dd_madd(acc, a, b); }
  __device__ __forceinline__ static dd maddc(dd acc, dd a, dd b) { return dd_madd(acc, a, b); }
  __device__ __forceinline__ static dd diag(dd a) { return a; }
  // inputs are renormalised (QuickTwoSum) as they are read
  __device__ __forceinline__ static dd load(const dd* p) {
    const double* f = reinterpret_cast<const double*>(p);
    return dd_renorm(dd{__ldg(f), __ldg(f + 1)});
  }
  __device__ __forceinline__ static dd shfl_xor(dd v, int m) {
    return dd{__shfl_xor_sync(0xffffffffu, v.hi, m), __shfl_xor_sync(0xffffffffu, v.lo, m)};
  }
  __device__ __forceinline__ static dd shfl(dd v, int s) {
    return dd{__shfl_sync(0xffffffffu, v.hi, s), __shfl_sync(0xffffffffu, v.lo, s)};
  }
};

// ------------------------------------------------ 16-byte streaming loads --
// The stored triangle is read exactly once: bypass L1 and use the read-only
// path.  The address must be 16-byte aligned.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// unpack one 16-byte vector into VPL elements of T
template <class T> struct Unpack;
template <> struct Unpack<float> {
  __device__ __forceinline__ static void run(uint4 v, float* o) {
    o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
  }
};
template <> struct Unpack<double> {
  __device__ __forceinline__ static void run(uint4 v, double* o) {
    o[0] = __hiloint2double((int)v.y, (int)v.x);
    o[1] = __hiloint2double((int)v.w, (int)v.z);
  }
};
template <> struct Unpack<c32> {
  __device__ __forceinline__ static void run(uint4 v, c32* o) {
    o[0] = c32{__uint_as_float(v.x), __uint_as_float(v.y)};
    o[1] = c32{__uint_as_float(v.z), __uint_as_float(v.w)};
  }
};
template <> struct Unpack<c64> {
  __device__ __forceinline__ static void run(uint4 v, c64* o) {
    o[0] = c64{__hiloint2double((int)v.y, (int)v.x), __hiloint2double((int)v.w, (int)v.z)};
  }
};
template <> struct Unpack<dd> {
  __device__ __forceinline__ static void run(uint4 v, dd* o) {
    o[0] = dd_renorm(dd{__hiloint2double((int)v.y, (int)v.x), __hiloint2double((int)v.w, (int)v.z)});
  }
};

}  // namespace xsymv
