// Online-softmax merge of two finished partials (O, LSE) of the same query row
// ("Context parallelism and ring attention", section "Online softmax": with
// (O, LSE) = (u/z, m + ln z), the running (m, z, u) update reduces to the
// weights below).  Used by the stand-alone merge kernel and by the forward
// kernel's epilogue in merge mode, so both fold partials identically.
#pragma once
#include <cuda_runtime.h>

namespace gb300 {

// M = max(la, lb); if M = -inf both weights are 0 and lnew = -inf, else
// lnew = M + ln(e^(la-M) + e^(lb-M)), ca = e^(la-lnew), cb = e^(lb-lnew).
__device__ __forceinline__ void merge_coeffs(float la, float lb, float& ca, float& cb,
                                             float& lnew) {
  const float M = fmaxf(la, lb);
  ca = 0.f;
  cb = 0.f;
  lnew = -INFINITY;
  if (M != -INFINITY) {
    const float ea = (la == -INFINITY) ? 0.f : expf(la - M);
    const float eb = (lb == -INFINITY) ? 0.f : expf(lb - M);
    const float z = ea + eb;
    lnew = M + logf(z);
    ca = ea / z;
    cb = eb / z;
  }
}

// ca * a + cb * x, where a zero weight drops its operand entirely (an
// accumulator row with LSE -inf may hold anything, even NaN).
__device__ __forceinline__ float merge1(float ca, float cb, float a, float x) {
  return (ca != 0.f ? ca * a : 0.f) + (cb != 0.f ? cb * x : 0.f);
}

__device__ __forceinline__ float4 merge4(float ca, float cb, const float4& a, const float4& x) {
  return make_float4(merge1(ca, cb, a.x, x.x), merge1(ca, cb, a.y, x.y), merge1(ca, cb, a.z, x.z),
                     merge1(ca, cb, a.w, x.w));
}

}  // namespace gb300
