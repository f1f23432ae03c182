// Entry points xgemv_s / xgemv_d: the general product y := alpha*A*x + beta*y
// on the SYMV kernels' loader, for comparing SYMV with GEMV ("CUDA-xSYMV の
// 実装と評価", §1: SYMV halves GEMV's memory traffic).
#include <atomic>

#include "xsymv_entry.cuh"
#include "xsymv_gemv.cuh"

namespace xsymv {
namespace {

template <class T>
struct GemvArgs {
  GemvPlan plan;
  const T* A;
  long long lda;
  const T* x;
  int incx;
  T* Wr;
  bool aligned;
  cudaStream_t stream;
};

template <class T>
struct GemvVariant {
  const char* name;
  int NB;
  int warps;
  cudaError_t (*launch)(const GemvArgs<T>&);
  int (*ctas_per_sm)();
};

template <class T, int VR, int U, int WARPS, int MB>
cudaError_t launch_gemv(const GemvArgs<T>& a) {
  const unsigned grid = (unsigned)((a.plan.W + WARPS - 1) / WARPS);
  if (a.aligned)
    gemv_main<T, VR, U, WARPS, true, MB><<<grid, WARPS * 32, 0, a.stream>>>(a.plan, a.A, a.lda,
                                                                            a.x, a.incx, a.Wr);
  else
    gemv_main<T, VR, U, WARPS, false, MB><<<grid, WARPS * 32, 0, a.stream>>>(a.plan, a.A, a.lda,
                                                                             a.x, a.incx, a.Wr);
  return cudaGetLastError();
}

template <class T, int VR, int U, int WARPS, int MB>
int gemv_ctas_per_sm() {
  static std::atomic<int> cache[kMaxDevices];
  return per_device_count(cache, [] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, gemv_main<T, VR, U, WARPS, true, MB>,
                                                      WARPS * 32, 0) != cudaSuccess)
      b = 0;
    return b;
  });
}

// names: vr<VR>_u<U>_r0_w<WARPS>[_b<MINB>], as for the SYMV register path
#define XGEMV_VARIANT(T, VR, U, W, MB, SUF)                                                 \
  GemvVariant<T> {                                                                          \
    "vr" #VR "_u" #U "_r0_w" #W SUF, 32 * Ops<T>::VPL * (VR), (W),                         \
        &launch_gemv<T, VR, U, W, MB>, &gemv_ctas_per_sm<T, VR, U, W, MB>                   \
  }

const GemvVariant<float> kGemv_s[] = {
    XGEMV_VARIANT(float, 1, 2, 8, 6, "_b6"),
    XGEMV_VARIANT(float, 1, 4, 8, 5, "_b5"),
    XGEMV_VARIANT(float, 1, 4, 8, 0, ""),
    XGEMV_VARIANT(float, 2, 2, 8, 0, ""),
    XGEMV_VARIANT(float, 1, 8, 8, 0, ""),
};
const GemvVariant<double> kGemv_d[] = {
    XGEMV_VARIANT(double, 4, 2, 8, 0, ""),
    XGEMV_VARIANT(double, 2, 2, 8, 0, ""),
    XGEMV_VARIANT(double, 2, 4, 8, 0, ""),
    XGEMV_VARIANT(double, 1, 4, 8, 0, ""),
};
constexpr int kGemvCount_s = (int)(sizeof(kGemv_s) / sizeof(kGemv_s[0]));
constexpr int kGemvCount_d = (int)(sizeof(kGemv_d) / sizeof(kGemv_d[0]));

std::atomic<int> g_gemv_forced[2] = {{-1}, {-1}};

int gemv_type_index(char t) {
  if (t == 's' || t == 'S') return 0;
  if (t == 'd' || t == 'D') return 1;
  return -1;
}

inline int gemv_check_args(int n, int lda, int incx, int incy) {
  if (n < 0) return 1;
  if (lda < (n > 1 ? n : 1)) return 4;
  if (incx == 0) return 6;
  if (incy == 0) return 9;
  return 0;
}

template <class T>
cudaError_t launch_gemv_finalize(const GemvPlan& p, const T* Wr, T alpha, T beta, int mode,
                                 T* y0, long long incy, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.n + kFinCols - 1) / kFinCols));
  cfg.blockDim = dim3(kFinParts * kFinCols);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_finalize<T>, p, Wr, alpha, beta, mode, y0, incy);
}

template <class T>
int gemv_entry(const GemvVariant<T>* table, int count, int tindex, int n, T alpha, const T* A,
               int lda, const T* x, int incx, T beta, T* y, int incy) {
  int info = gemv_check_args(n, lda, incx, incy);
  if (info) return info;
  if (n == 0) return XSYMV_OK;
  const bool az = is_zero(alpha), bz = is_zero(beta);
  if (az && is_one(beta)) return XSYMV_OK;
  cudaStream_t st = current_stream();
  T* y0 = y + (incy < 0 ? (long long)(1 - n) * incy : 0);
  const T* x0 = x + (incx < 0 ? (long long)(1 - n) * incx : 0);
  int dev = 0, sms = 0;
  if (!current_device(&dev, &sms)) return XSYMV_ERR_DEVICE;

  if (az) {  // y := beta*y: neither A nor x is read (the SYMV finaliser's beta-only mode)
    Plan p = plan_make(n, 32, 1, 1);
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

  const int f = g_gemv_forced[tindex].load();
  const GemvVariant<T>* v = &table[(f >= 0 && f < count) ? f : 0];
  const long long wmax = (long long)sms * v->ctas_per_sm() * v->warps;
  const GemvPlan p = gemv_plan_make(n, v->NB, wmax);
  const long long wr_bytes = align_up((long long)p.nb * p.qmax * p.NB * (long long)sizeof(T), 256);
  int status = XSYMV_OK, epoch = 0;
  char* ws = static_cast<char*>(workspace((size_t)(kHeaderBytes + wr_bytes), st, &status, 0, &epoch));
  if (!ws) return status;
  GemvArgs<T> a{p, A, lda, x0, incx, reinterpret_cast<T*>(ws + kHeaderBytes),
                (reinterpret_cast<uintptr_t>(A) % 16 == 0) &&
                    (((long long)lda * (long long)sizeof(T)) % 16 == 0),
                st};
  timing_begin(st);
  cudaError_t e = v->launch(a);
  if (e == cudaSuccess) {
    timing_mid(st);
    e = launch_gemv_finalize<T>(p, a.Wr, alpha, beta, bz ? kBetaZero : kFull, y0, incy, st);
  }
  timing_end(st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return XSYMV_ERR_CUDA;
  }
  note_launches(2);
  note_call_status(st, nullptr, 0);   // nothing in the general product waits
  return XSYMV_OK;
}

}  // namespace
}  // namespace xsymv

extern "C" XSYMV_API int xgemv_s(int n, float alpha, const float* A, int lda, const float* x,
                                 int incx, float beta, float* y, int incy) {
  return xsymv::gemv_entry<float>(xsymv::kGemv_s, xsymv::kGemvCount_s, 0, n, alpha, A, lda, x,
                                  incx, beta, y, incy);
}

extern "C" XSYMV_API int xgemv_d(int n, double alpha, const double* A, int lda, const double* x,
                                 int incx, double beta, double* y, int incy) {
  return xsymv::gemv_entry<double>(xsymv::kGemv_d, xsymv::kGemvCount_d, 1, n, alpha, A, lda, x,
                                   incx, beta, y, incy);
}

extern "C" XSYMV_API int xgemv_variant_count(char type) {
  const int t = xsymv::gemv_type_index(type);
  return t == 0 ? xsymv::kGemvCount_s : t == 1 ? xsymv::kGemvCount_d : XSYMV_ERR_VALUE;
}

extern "C" XSYMV_API const char* xgemv_variant_name(char type, int index) {
  const int t = xsymv::gemv_type_index(type);
  if (t < 0 || index < 0 || index >= xgemv_variant_count(type)) return nullptr;
  return t == 0 ? xsymv::kGemv_s[index].name : xsymv::kGemv_d[index].name;
}

extern "C" XSYMV_API int xgemv_set_variant(char type, int index) {
  const int t = xsymv::gemv_type_index(type);
  if (t < 0 || index < -1 || index >= xgemv_variant_count(type)) return XSYMV_ERR_VALUE;
  xsymv::g_gemv_forced[t].store(index);
  return XSYMV_OK;
}

extern "C" XSYMV_API int xgemv_selected_variant(char type) {
  const int t = xsymv::gemv_type_index(type);
  if (t < 0) return XSYMV_ERR_VALUE;
  const int f = xsymv::g_gemv_forced[t].load();
  return f >= 0 ? f : 0;
}
