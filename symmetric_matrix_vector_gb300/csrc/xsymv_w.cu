// Entry point xsymv_w of the xsymv C ABI and its compiled kernel variants.
#include "xsymv_entry.cuh"

namespace xsymv {
static const Variant<dd> kVariants_w[] = {
    XSYMV_REG(dd, 4, 2, 8),
    XSYMV_REG(dd, 2, 2, 8),
    XSYMV_REG(dd, 4, 1, 8),
    XSYMV_REG_MB(dd, 4, 2, 8, 3),
    XSYMV_TMA(dd, 4, 2, 4, 4),
    XSYMV_REG_G(dd, 4, 2, 8, 0, 4),
    XSYMV_REG_G(dd, 4, 2, 8, 0, 5),
    XSYMV_REG_G(dd, 4, 2, 8, 0, 6),
    XSYMV_REG_GC(dd, 4, 2, 8, 0, 4, 8),
    XSYMV_REG_GC(dd, 4, 2, 8, 0, 4, 4),
    XSYMV_REG_GC(dd, 2, 2, 8, 0, 4, 8),
    XSYMV_REG_GC(dd, 4, 1, 8, 0, 4, 8),
    XSYMV_TICKET(dd, 4, 2, 8, 0, 4, 8),
    XSYMV_REG_GC(dd, 8, 1, 4, 0, 6, 8),
    XSYMV_FUSED(dd, 4, 2, 8, 0, 4, 8),
    XSYMV_REG_GC(dd, 8, 1, 4, 0, 4, 8),
    XSYMV_REG_GC(dd, 8, 1, 4, 0, 5, 8),
    XSYMV_REG_GC(dd, 8, 1, 4, 0, 7, 8),
    XSYMV_REG_GC(dd, 8, 1, 4, 0, 8, 8),
    XSYMV_FUSED(dd, 4, 2, 8, 0, 5, 8),
    XSYMV_FUSED(dd, 4, 2, 8, 0, 6, 8),
    XSYMV_REG_GC(dd, 4, 2, 8, 0, 5, 8),
    XSYMV_REG_GC(dd, 4, 2, 8, 0, 6, 8),
};
static_assert(sizeof(dd) == sizeof(xsymv_dd), "C-ABI type layout");
}  // namespace xsymv

XSYMV_DEFINE_INTROSPECTION(w, xsymv::dd, kVariants_w)
XSYMV_DEFINE_SHARDS(xsymv_w_shard, xsymv_w_reduce, 'w', xsymv_dd, xsymv::dd, xsymv::kVariants_w)

extern "C" XSYMV_API int xsymv_w(char uplo, int n, xsymv_dd alpha, const xsymv_dd* A, int lda, const xsymv_dd* x,
                                int incx, xsymv_dd beta, xsymv_dd* y, int incy) {
  using T = xsymv::dd;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_entry<T>(xsymv::kVariants_w,
                              (int)(sizeof(xsymv::kVariants_w) / sizeof(xsymv::kVariants_w[0])),
                              'w', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                              reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                              incy);
}

extern "C" XSYMV_API int xsymv_w_host(char uplo, int n, xsymv_dd alpha, const xsymv_dd* A, int lda, const xsymv_dd* x,
                                   int incx, xsymv_dd beta, xsymv_dd* y, int incy) {
  using T = xsymv::dd;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_host_entry<T>(xsymv::kVariants_w,
                                   (int)(sizeof(xsymv::kVariants_w) / sizeof(xsymv::kVariants_w[0])),
                                   'w', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                                   reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                                   incy);
}
