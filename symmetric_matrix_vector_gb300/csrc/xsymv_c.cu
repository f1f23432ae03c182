// Entry point xhemv_c of the xsymv C ABI and its compiled kernel variants.
#include "xsymv_entry.cuh"

namespace xsymv {
static const Variant<c32> kVariants_c[] = {
    XSYMV_REG(c32, 1, 4, 8),
    XSYMV_REG(c32, 2, 2, 8),
    XSYMV_REG(c32, 2, 4, 8),
    XSYMV_REG(c32, 1, 8, 8),
    XSYMV_REG_MB(c32, 1, 4, 8, 5),
    XSYMV_REG_MB(c32, 1, 2, 8, 5),
    XSYMV_REG_MB(c32, 2, 2, 8, 5),
    XSYMV_TMA(c32, 1, 8, 4, 4),
    XSYMV_REG_G(c32, 1, 4, 8, 0, 5),
    XSYMV_REG_G(c32, 1, 4, 8, 0, 7),
    XSYMV_REG_G(c32, 2, 2, 8, 0, 7),
    XSYMV_REG_GC(c32, 1, 4, 8, 0, 5, 8),
    XSYMV_REG_GC(c32, 2, 2, 8, 0, 7, 8),
    XSYMV_REG_GC(c32, 1, 4, 8, 0, 7, 8),
    XSYMV_TICKET(c32, 2, 2, 8, 0, 7, 2),
    XSYMV_REG_G(c32, 2, 2, 8, 4, 7),
    XSYMV_REG_G(c32, 2, 2, 8, 4, 9),
    XSYMV_REG_G(c32, 2, 2, 8, 4, 11),
    XSYMV_REG_G(c32, 2, 2, 8, 4, 5),
    XSYMV_REG_G(c32, 2, 2, 8, 4, 10),
    XSYMV_REG_G(c32, 2, 2, 8, 4, 13),
    XSYMV_FUSED(c32, 2, 2, 8, 4, 13, 2),
    XSYMV_FUSED(c32, 2, 2, 8, 4, 11, 2),
    XSYMV_FUSED(c32, 2, 2, 8, 4, 9, 2),
};
static_assert(sizeof(c32) == sizeof(xsymv_c32), "C-ABI type layout");
}  // namespace xsymv

XSYMV_DEFINE_INTROSPECTION(c, xsymv::c32, kVariants_c)
XSYMV_DEFINE_SHARDS(xhemv_c_shard, xhemv_c_reduce, 'c', xsymv_c32, xsymv::c32, xsymv::kVariants_c)

extern "C" XSYMV_API int xhemv_c(char uplo, int n, xsymv_c32 alpha, const xsymv_c32* A, int lda, const xsymv_c32* x,
                                int incx, xsymv_c32 beta, xsymv_c32* y, int incy) {
  using T = xsymv::c32;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_entry<T>(xsymv::kVariants_c,
                              (int)(sizeof(xsymv::kVariants_c) / sizeof(xsymv::kVariants_c[0])),
                              'c', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                              reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                              incy);
}

extern "C" XSYMV_API int xhemv_c_host(char uplo, int n, xsymv_c32 alpha, const xsymv_c32* A, int lda, const xsymv_c32* x,
                                   int incx, xsymv_c32 beta, xsymv_c32* y, int incy) {
  using T = xsymv::c32;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_host_entry<T>(xsymv::kVariants_c,
                                   (int)(sizeof(xsymv::kVariants_c) / sizeof(xsymv::kVariants_c[0])),
                                   'c', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                                   reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                                   incy);
}
