// Entry point xsymv_s of the xsymv C ABI and its compiled kernel variants.
#include "xsymv_entry.cuh"

namespace xsymv {
static const Variant<float> kVariants_s[] = {
    XSYMV_VARIANT(float, 1, 8, 8),
    XSYMV_VARIANT(float, 1, 16, 4),
    XSYMV_VARIANT(float, 2, 4, 8),
    XSYMV_VARIANT(float, 1, 4, 8),
};
static_assert(sizeof(float) == sizeof(float), "C-ABI type layout");
}  // namespace xsymv

XSYMV_DEFINE_INTROSPECTION(s, float, kVariants_s)

extern "C" XSYMV_API int xsymv_s(char uplo, int n, float alpha, const float* A, int lda, const float* x,
                                int incx, float beta, float* y, int incy) {
  using T = float;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_entry<T>(xsymv::kVariants_s,
                              (int)(sizeof(xsymv::kVariants_s) / sizeof(xsymv::kVariants_s[0])),
                              's', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                              reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                              incy);
}

extern "C" XSYMV_API int xsymv_s_host(char uplo, int n, float alpha, const float* A, int lda, const float* x,
                                   int incx, float beta, float* y, int incy) {
  using T = float;
  T a, b;
  memcpy(&a, &alpha, sizeof(T));
  memcpy(&b, &beta, sizeof(T));
  return xsymv::symv_host_entry<T>(xsymv::kVariants_s,
                                   (int)(sizeof(xsymv::kVariants_s) / sizeof(xsymv::kVariants_s[0])),
                                   's', uplo, n, a, reinterpret_cast<const T*>(A), lda,
                                   reinterpret_cast<const T*>(x), incx, b, reinterpret_cast<T*>(y),
                                   incy);
}
