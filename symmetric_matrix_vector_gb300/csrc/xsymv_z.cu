// Entry point xhemv_z of the xsymv C ABI and its compiled kernel variants.
#include "xsymv_entry.cuh"

namespace xsymv {
static const Variant<c64> kVariants_z[] = {
    XSYMV_REG(c64, 4, 2, 8),
    XSYMV_REG(c64, 2, 2, 8),
    XSYMV_REG(c64, 4, 1, 8),
    XSYMV_REG(c64, 2, 4, 8),
    XSYMV_REG_MB(c64, 4, 2, 8, 4),
    XSYMV_TMA(c64, 4, 2, 4, 4),
    XSYMV_REG_G(c64, 4, 2, 8, 0, 4),
    XSYMV_REG_G(c64, 4, 2, 8, 0, 5),
    XSYMV_REG_G(c64, 4, 2, 8, 0, 6),
    XSYMV_REG_GC(c64, 4, 2, 8, 0, 4, 8),
    XSYMV_REG_GC(c64, 4, 2, 8, 0, 4, 4),
    XSYMV_REG_GC(c64, 4, 2, 8, 0, 5, 8),
    XSYMV_REG_GC(c64, 2, 2, 8, 0, 4, 8),
    XSYMV_TICKET(c64, 4, 2, 8, 0, 5, 8),
    XSYMV_FUSED(c64, 4, 2, 8, 0, 5, 8),
    XSYMV_FUSED(c64, 4, 2, 8, 0, 4, 8),
    XSYMV_FUSED(c64, 4, 2, 8, 0, 6, 8),
    XSYMV_REG_GC(c64, 4, 2, 8, 0, 6, 8),
};
static_assert(sizeof(c64) == sizeof(xsymv_c64), "C-ABI type layout");
}  // namespace xsymv

XSYMV_DEFINE_INTROSPECTION(z, xsymv::c64, kVariants_z)
XSYMV_DEFINE_SHARDS(xhemv_z_shard, xhemv_z_reduce, 'z', xsymv_c64, xsymv::c64, xsymv::kVariants_z)

extern "C" XSYMV_API int xhemv_z(char uplo, int n, xsymv_c64 alpha, const xsymv_c64* A, int lda, const xsymv_c64* x,
                                int incx, xsymv_c64 beta, xsymv_c64* y, int incy) {
  using T = xsymv::c64;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_entry<T>(xsymv::kVariants_z,
                              (int)(sizeof(xsymv::kVariants_z) / sizeof(xsymv::kVariants_z[0])),
                              'z', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                              reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                              incy);
}

extern "C" XSYMV_API int xhemv_z_host(char uplo, int n, xsymv_c64 alpha, const xsymv_c64* A, int lda, const xsymv_c64* x,
                                   int incx, xsymv_c64 beta, xsymv_c64* y, int incy) {
  using T = xsymv::c64;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_host_entry<T>(xsymv::kVariants_z,
                                   (int)(sizeof(xsymv::kVariants_z) / sizeof(xsymv::kVariants_z[0])),
                                   'z', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                                   reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                                   incy);
}
