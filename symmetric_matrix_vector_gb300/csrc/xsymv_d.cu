// Entry point xsymv_d of the xsymv C ABI and its compiled kernel variants.
#include "xsymv_entry.cuh"

namespace xsymv {
static const Variant<double> kVariants_d[] = {
    XSYMV_REG(double, 4, 2, 8),
    XSYMV_REG(double, 2, 4, 8),
    XSYMV_REG(double, 2, 2, 8),
    XSYMV_REG(double, 1, 4, 8),
    XSYMV_REG_MB(double, 2, 2, 8, 5),
    XSYMV_REG_MB(double, 4, 2, 8, 4),
    XSYMV_TMA(double, 2, 4, 4, 4),
    XSYMV_REG_G(double, 4, 2, 8, 0, 4),
    XSYMV_REG_G(double, 4, 2, 8, 0, 5),
    XSYMV_REG_G(double, 4, 2, 8, 0, 6),
    XSYMV_REG_G(double, 2, 4, 8, 0, 5),
    XSYMV_REG_GC(double, 4, 2, 8, 0, 5, 8),
    XSYMV_REG_GC(double, 4, 2, 8, 0, 5, 4),
    XSYMV_REG_GC(double, 2, 4, 8, 0, 5, 8),
    XSYMV_REG_GC(double, 4, 2, 8, 0, 5, 16),
    XSYMV_REG_GC(double, 4, 2, 8, 0, 4, 8),
    XSYMV_TICKET(double, 4, 2, 8, 0, 5, 8),
    XSYMV_REG_GC(double, 8, 1, 4, 0, 8, 8),
    XSYMV_FUSED(double, 4, 2, 8, 0, 5, 8),
    XSYMV_FUSED(double, 4, 2, 8, 0, 4, 8),
    XSYMV_FUSED(double, 4, 2, 8, 0, 6, 8),
    XSYMV_REG_GC(double, 4, 2, 8, 0, 6, 8),
};
static_assert(sizeof(double) == sizeof(double), "C-ABI type layout");
}  // namespace xsymv

XSYMV_DEFINE_INTROSPECTION(d, double, kVariants_d)
XSYMV_DEFINE_SHARDS(xsymv_d_shard, xsymv_d_reduce, 'd', double, double, xsymv::kVariants_d)

extern "C" XSYMV_API int xsymv_d(char uplo, int n, double alpha, const double* A, int lda, const double* x,
                                int incx, double beta, double* y, int incy) {
  using T = double;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_entry<T>(xsymv::kVariants_d,
                              (int)(sizeof(xsymv::kVariants_d) / sizeof(xsymv::kVariants_d[0])),
                              'd', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                              reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                              incy);
}

extern "C" XSYMV_API int xsymv_d_host(char uplo, int n, double alpha, const double* A, int lda, const double* x,
                                   int incx, double beta, double* y, int incy) {
  using T = double;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_host_entry<T>(xsymv::kVariants_d,
                                   (int)(sizeof(xsymv::kVariants_d) / sizeof(xsymv::kVariants_d[0])),
                                   'd', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                                   reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                                   incy);
}
