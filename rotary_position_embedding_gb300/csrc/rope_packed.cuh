// Packed 16-bit arithmetic shared by the pipelined kernels.
#pragma once

#include "rope_kernels.cuh"

namespace rope_gb300 {

// ---------------------------------------------------------------------------
// Packed arithmetic for 16-bit storage (float16, bfloat16) on 16-byte units:
// two values per 32-bit word, float32x2 operations (sm_100 and later). Each
// lane of a packed operation rounds exactly as the scalar operation does, so
// the results have the bits of rotate(): a product, then a fused multiply-add
// (-(x1*s) is formed as x1*(-s), which rounds to the same value). Used by the
// pipelined kernels, whose consumers rotate several heads per coefficient
// unpack, and by the SIMT Q/K heads kernel's QK-Norm path; the other SIMT
// paths keep the scalar form, which needs fewer registers and so keeps more
// CTAs resident.
// ---------------------------------------------------------------------------
template <class T>
struct P2;
template <>
struct P2<__half> {
  using w2 = __half2;
  static __device__ __forceinline__ float2 tof(w2 v) { return __half22float2(v); }
  static __device__ __forceinline__ w2 fromf(float2 f) { return __float22half2_rn(f); }
};
template <>
struct P2<__nv_bfloat16> {
  using w2 = __nv_bfloat162;
  static __device__ __forceinline__ float2 tof(w2 v) { return __bfloat1622float2(v); }
  static __device__ __forceinline__ w2 fromf(float2 f) { return __float22bfloat162_rn(f); }
};

template <class T>
struct Unit8 {  // one 16-byte unit of 8 values as 4 packed words
  typename P2<T>::w2 w[4];
};

// Rotation of a unit pair (half split: pair j = (a[j], b[j]); interleaved:
// pair j = elements 2j, 2j+1 of a||b) with unpacked coefficients
// (cf[k] holds the coefficients of pairs 2k and 2k+1).
template <class T, bool INTER>
__device__ __forceinline__ void rotate8p(const Unit8<T>& a, const Unit8<T>& b, const float2 (&cf)[4],
                                         const float2 (&sf)[4], Unit8<T>& ya, Unit8<T>& yb) {
  using P = P2<T>;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 ns = make_float2(-sf[k].x, -sf[k].y);
    if (!INTER) {
      const float2 x0 = P::tof(a.w[k]), x1 = P::tof(b.w[k]);
      ya.w[k] = P::fromf(__ffma2_rn(x0, cf[k], __fmul2_rn(x1, ns)));
      yb.w[k] = P::fromf(__ffma2_rn(x1, cf[k], __fmul2_rn(x0, sf[k])));
    } else {
      // words 2k and 2k+1 of a||b hold pairs 2k and 2k+1
      const float2 f0 = P::tof(k < 2 ? a.w[2 * k] : b.w[2 * k - 4]);
      const float2 f1 = P::tof(k < 2 ? a.w[2 * k + 1] : b.w[2 * k - 3]);
      const float2 x0 = make_float2(f0.x, f1.x), x1 = make_float2(f0.y, f1.y);
      const float2 y0 = __ffma2_rn(x0, cf[k], __fmul2_rn(x1, ns));
      const float2 y1 = __ffma2_rn(x1, cf[k], __fmul2_rn(x0, sf[k]));
      const typename P::w2 p0 = P::fromf(make_float2(y0.x, y1.x));
      const typename P::w2 p1 = P::fromf(make_float2(y0.y, y1.y));
      if (k < 2) {
        ya.w[2 * k] = p0;
        ya.w[2 * k + 1] = p1;
      } else {
        yb.w[2 * k - 4] = p0;
        yb.w[2 * k - 3] = p1;
      }
    }
  }
}

// Coefficient unit unpacked to float32 pairs.
template <class T>
__device__ __forceinline__ void unpack_coef8(const VecT<T, 8>& c, float2 (&cf)[4]) {
  Unit8<T> u;
  __builtin_memcpy(&u, &c, 16);
#pragma unroll
  for (int k = 0; k < 4; ++k) cf[k] = P2<T>::tof(u.w[k]);
}

// z = T(w * T(x * r)) on a unit whose values fx are already unpacked: the
// first product in float32x2, the second on the 16-bit words (the product of
// two 16-bit values is exact in float32, so the 16-bit multiply rounds it just
// as float32-then-round does).
template <class T>
__device__ __forceinline__ Unit8<T> norm8p(const float2 (&fx)[4], float r, const Unit8<T>& w) {
  using P = P2<T>;
  const float2 r2 = make_float2(r, r);
  Unit8<T> z;
#pragma unroll
  for (int k = 0; k < 4; ++k) z.w[k] = __hmul2(P::fromf(__fmul2_rn(fx[k], r2)), w.w[k]);
  return z;
}

}  // namespace rope_gb300
