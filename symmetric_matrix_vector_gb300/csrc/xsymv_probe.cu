// Probe kernels for the roofline denominators measured in the same run as a
// benchmark: HBM copy and read bandwidth, and FP64 / FP32 FMA throughput.
// The report compares its achieved bandwidth with both the theoretical peak
// and a measured copy rate ("CUDA-xSYMV の実装と評価", §4 and footnote *5,
// bandwidthTest); on GB300 the FP64 rate matters too, because DSYMV, ZHEMV
// and WSYMV need more FP64 operations per byte than the GPU can issue at
// full HBM speed.
#include <cuda_runtime.h>

#include "../../include/xsymv.h"
#include "xsymv_runtime.h"
#include "xsymv_scalar.cuh"

namespace xsymv {
namespace {

__global__ void probe_copy(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// UNR independent 16-byte loads in flight per thread and iteration
template <int UNR>
__global__ void probe_read(const uint4* __restrict__ src, size_t n, unsigned* sink) {
  unsigned acc = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  for (; i + (UNR - 1) * stride < n; i += UNR * stride) {
    uint4 v[UNR];
#pragma unroll
    for (int k = 0; k < UNR; ++k) v[k] = __ldcs(src + i + k * stride);
#pragma unroll
    for (int k = 0; k < UNR; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
  for (; i < n; i += stride) {
    const uint4 v = __ldcs(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u) sink[0] = acc;   // practically never; keeps the loads
}

// The multiplier and addend of the FMA probe, read by an opaque load so
// that they sit in registers: on GB300 an FP64 FMA with an immediate or
// constant-bank operand (as a compile-time constant becomes) issues at
// about 1.68 per clock per SM, one with register operands at 2.0, the
// unit's rate.
static __device__ double g_probe_bc64[2] = {0.999999, 1e-9};
static __device__ float g_probe_bc32[2] = {0.999999f, 1e-9f};
__device__ __forceinline__ double opaque_load(const double* p) {
  double v;
  asm("ld.global.nc.f64 %0, [%1];" : "=d"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float opaque_load(const float* p) {
  float v;
  asm("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
template <class F> struct ProbeBC;
template <> struct ProbeBC<double> { __device__ static const double* p() { return g_probe_bc64; } };
template <> struct ProbeBC<float> { __device__ static const float* p() { return g_probe_bc32; } };

// 8 independent FMA chains per thread, all operands in registers.
template <class F>
__global__ void probe_fma(F* out, int iters) {
  F a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = (F)(threadIdx.x + k) * (F)1e-7;
  const F b = opaque_load(ProbeBC<F>::p()), c = opaque_load(ProbeBC<F>::p() + 1);
#pragma unroll 1
  for (int i = 0; i < iters; ++i)
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = fma(a[k], b, c);
  F s = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += a[k];
  if (s == (F)12345.678) out[0] = s;
}

// out[6i .. 6i+5] = a+b, a-b, a*b with the plain instructions, then the
// same three as the DD code issues them (see d_add, d_sub, d_mul)
__global__ void probe_unit_forms(const double* __restrict__ a, const double* __restrict__ b,
                                 double* __restrict__ out, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const double x = a[i], y = b[i];
    double* o = out + 6 * i;
    o[0] = __dadd_rn(x, y);
    o[1] = __dsub_rn(x, y);
    o[2] = __dmul_rn(x, y);
    o[3] = d_add(x, y);
    o[4] = d_sub(x, y);
    o[5] = d_mul(x, y);
  }
}

float elapsed(cudaEvent_t a, cudaEvent_t b) {
  float ms = 0.f;
  cudaEventElapsedTime(&ms, a, b);
  return ms;
}

}  // namespace
}  // namespace xsymv

using namespace xsymv;

extern "C" XSYMV_API int xsymv_probe_peaks(double* copy_gbs, double* read_gbs,
                                           double* fp64_tflops, double* fp32_tflops) {
  int dev = 0, sms = 0;
  if (!current_device(&dev, &sms)) return XSYMV_ERR_DEVICE;
  cudaStream_t st = current_stream();
  const size_t bytes = (size_t)1 << 30;  // 1 GiB per buffer, far above the L2
  const size_t n16 = bytes / 16;
  void *a = nullptr, *b = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaMalloc(&a, bytes);
  if (e == cudaSuccess) e = cudaMalloc(&b, bytes);
  if (e == cudaSuccess) e = cudaMemsetAsync(a, 1, bytes, st);
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  double best_copy = 0, best_read = 0, best64 = 0, best32 = 0;
  const unsigned grid = (unsigned)sms * 8, block = 256;
  for (int rep = 0; rep < 5 && e == cudaSuccess; ++rep) {
    cudaEventRecord(e0, st);
    probe_copy<<<grid, block, 0, st>>>((const uint4*)a, (uint4*)b, n16);
    cudaEventRecord(e1, st);
    e = cudaEventSynchronize(e1);
    const double c = 2.0 * bytes / (elapsed(e0, e1) * 1e-3) / 1e9;
    if (c > best_copy) best_copy = c;
    // two shapes of the read stream; the faster one counts
    for (int shape = 0; shape < 2 && e == cudaSuccess; ++shape) {
      cudaEventRecord(e0, st);
      if (shape == 0)
        probe_read<4><<<(unsigned)sms * 4, block, 0, st>>>((const uint4*)a, n16, (unsigned*)b);
      else
        probe_read<8><<<(unsigned)sms * 4, block, 0, st>>>((const uint4*)a, n16, (unsigned*)b);
      cudaEventRecord(e1, st);
      e = cudaEventSynchronize(e1);
      const double r = 1.0 * bytes / (elapsed(e0, e1) * 1e-3) / 1e9;
      if (r > best_read) best_read = r;
    }
  }
  const unsigned fgrid = (unsigned)sms * 8;
  const int iters64 = 1 << 12, iters32 = 1 << 15;
  for (int rep = 0; rep < 3 && e == cudaSuccess; ++rep) {
    cudaEventRecord(e0, st);
    probe_fma<double><<<fgrid, block, 0, st>>>((double*)b, iters64);
    cudaEventRecord(e1, st);
    e = cudaEventSynchronize(e1);
    const double f64 = 2.0 * 8 * iters64 * (double)fgrid * block / (elapsed(e0, e1) * 1e-3) / 1e12;
    if (f64 > best64) best64 = f64;
    cudaEventRecord(e0, st);
    probe_fma<float><<<fgrid, block, 0, st>>>((float*)b, iters32);
    cudaEventRecord(e1, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    const double f32 = 2.0 * 8 * iters32 * (double)fgrid * block / (elapsed(e0, e1) * 1e-3) / 1e12;
    if (f32 > best32) best32 = f32;
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (a) cudaFree(a);
  if (b) cudaFree(b);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  if (copy_gbs) *copy_gbs = best_copy;
  if (read_gbs) *read_gbs = best_read;
  if (fp64_tflops) *fp64_tflops = best64;
  if (fp32_tflops) *fp32_tflops = best32;
  note_launches(21);
  return XSYMV_OK;
}

extern "C" XSYMV_API int xsymv_probe_unit_forms(const double* a, const double* b, double* out,
                                               long long n) {
  if (n < 0) return XSYMV_ERR_VALUE;
  if (n == 0) return XSYMV_OK;
  if (!a || !b || !out) return XSYMV_ERR_VALUE;
  int dev = 0, sms = 0;
  if (!current_device(&dev, &sms)) return XSYMV_ERR_DEVICE;
  cudaStream_t st = current_stream();
  long long blocks = (n + 255) / 256;
  if (blocks > (long long)sms * 16) blocks = (long long)sms * 16;
  probe_unit_forms<<<(unsigned)blocks, 256, 0, st>>>(a, b, out, n);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  note_launches(1);
  return XSYMV_OK;
}
