// On-the-fly RoPE / M-RoPE and the cos/sin cache build for sm_103a.
//
// Definitions followed (web pages, by title and section):
//  - onnxruntime pull request "Add RotaryEmbedding fusion for Qwen3 on-the-fly
//    RoPE patterns": Modeling Code Alignment Check (freqs = inv_freq x
//    positions in float32, cat(freqs, freqs), cos * attention_scaling),
//    Medium Issues 4 (the cache is cos(freqs) * scaling).
//  - "com.microsoft.MRotaryEmbedding" README: Description and Attributes (the
//    three position streams, the scale applied to the cached coefficient).
#pragma once

#include "rope_kernels.cuh"

namespace rope_gb300 {

// ---------------------------------------------------------------------------
// On-the-fly coefficients (float32 angle, double-precision cos/sin rounded to
// float32, times attention scaling in float32, rounded to T). Shared by the
// fused kernel and the cache build so the two agree bit for bit.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void coef_on_the_fly(int64_t pos, float inv, float scaling, float& c,
                                                float& s) {
  const float pf = __ll2float_rn(pos);
  const float theta = __fmul_rn(pf, inv);
  double sd, cd;
  sincos((double)theta, &sd, &cd);
  c = __fmul_rn(__double2float_rn(cd), scaling);
  s = __fmul_rn(__double2float_rn(sd), scaling);
}

// The same coefficients in T's storage, after the whole rounding chain of the
// cached table: T(fl32(fl32(cos theta) * scaling)), and for M-RoPE then
// T(cb * mscale) rounded once (MSCALE). On 16-bit storage most values come
// from float arithmetic, exactly:
//  - sincosf is within 2 ulp of the exact value (CUDA's documented bound for
//    sinf/cosf/sincosf without fast-math), so the exact value lies in
//    [v - e, v + e] with e = |v| * 2^-20 (at least 8 ulp of v), at least 4 ulp
//    inside either end, and so does the double-precision value that
//    coef_on_the_fly rounds to float32;
//  - the chain x -> T(...) is monotone in x (products by a fixed factor and
//    round-to-nearest are), so where the ends of that interval give the same
//    bits, every point inside does, and the result is what coef_on_the_fly
//    gives;
//  - otherwise (about 0.1 % of float16 values: an end lies across a rounding
//    boundary) the value is computed by coef_on_the_fly.
// float32 storage always takes coef_on_the_fly (the chain there keeps the 2-ulp
// uncertainty).
template <class T, bool MSCALE>
__device__ __forceinline__ typename Elem<T>::bits coef_chain(float x, float scaling, float mscale) {
  using E = Elem<T>;
  typename E::bits b = E::fromf(__fmul_rn(x, scaling));
  if (MSCALE) b = E::fromf(E::mul_round(E::tof(b), mscale));
  return b;
}

// ---------------------------------------------------------------------------
// Double-float sine and cosine of a float angle with |theta| < 2^17, for the
// values the float path above leaves open. Methods:
//  - argument reduction of Cody and Waite (W. J. Cody, W. Waite, "Software
//    Manual for the Elementary Functions", 1980): theta = k pi/2 + r with pi/2
//    split into four floats, the first of 7 significant bits, so that k * P1
//    is exact for |k| < 2^17 and theta - k P1 (one fused multiply-add) is exact;
//  - the error-free sum and product of Knuth and Dekker (D. E. Knuth, "The Art
//    of Computer Programming", vol. 2; T. J. Dekker, "A floating-point
//    technique for extending the available precision", 1971) for the remaining
//    parts and for double-float sums and products (as analysed in M. Joldes,
//    J.-M. Muller, V. Popescu, "Tight and rigorous error bounds for basic
//    building blocks of double-word arithmetic", 2017);
//  - the Taylor series of sin and cos on |r| <= pi/4 (plus a rounding of k) to
//    r^15 and r^16, whose truncation is below 2^-53, in double-float Horner
//    steps with the coefficients 1/n! split into two floats.
// The reduction's absolute error is below 2^-46 (the double-float parts of r
// rounded at most about 2^-48 of a value below 1, and the pi/2 tail past the
// fourth part below 2^-68 for |k| < 2^17); each double-float step adds a
// relative error of about 2^-45, about 20 of them. So the exact value lies
// within |v| 2^-36 + 2^-44 of the double-float result v.
// ---------------------------------------------------------------------------
struct FFloat {
  float h, l;
};

__device__ __forceinline__ FFloat ff_two_sum(float a, float b) {  // a + b = h + l exactly
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FFloat ff_fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FFloat ff_two_prod(float a, float b) {  // a * b = h + l exactly
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
// sums with no cancellation (the Horner steps below: |z acc| < |c| / 10)
__device__ __forceinline__ FFloat ff_add(FFloat a, FFloat b) {
  const FFloat s = ff_two_sum(a.h, b.h);
  return ff_fast_two_sum(s.h, __fadd_rn(s.l, __fadd_rn(a.l, b.l)));
}
__device__ __forceinline__ FFloat ff_mul(FFloat a, FFloat b) {
  const FFloat p = ff_two_prod(a.h, b.h);
  return ff_fast_two_sum(p.h, __fmaf_rn(a.h, b.l, __fmaf_rn(a.l, b.h, p.l)));
}

__device__ __forceinline__ void ff_sincos(float theta, FFloat& sv, FFloat& cv) {
  const float k = rintf(__fmul_rn(theta, 0x1.45f306p-1f));  // nearest k of theta * 2/pi
  // pi/2 = P1 + P2 + P3 + P4 + (below 2^-85)
  constexpr float P1 = 0x1.94p+0f, P2 = -0x1.e04abcp-8f, P3 = 0x1.0b4612p-34f, P4 = -0x1.676734p-60f;
  const float r1 = __fmaf_rn(-k, P1, theta);  // exact
  FFloat p = ff_two_prod(k, P2);
  const FFloat s1 = ff_two_sum(r1, -p.h);
  float lo = __fsub_rn(s1.l, p.l);
  p = ff_two_prod(k, P3);
  const FFloat s2 = ff_two_sum(s1.h, -p.h);
  lo = __fadd_rn(lo, __fsub_rn(s2.l, p.l));
  lo = __fmaf_rn(-k, P4, lo);
  const FFloat r = ff_two_sum(s2.h, lo);
  const FFloat z = ff_mul(r, r);
  // (-1)^j / (2j+1)!, j = 7 .. 1, and (-1)^j / (2j)!, j = 8 .. 1, as high + low floats
  constexpr float SN[7][2] = {{-0x1.ae7f3ep-41f, -0x1.ccee08p-67f}, {0x1.612462p-33f, -0x1.8af25ep-58f},
                              {-0x1.ae6456p-26f, -0x1.fd5138p-52f}, {0x1.71de3ap-19f, 0x1.55b1ccp-45f},
                              {-0x1.a01a02p-13f, 0x1.7f97fap-39f}, {0x1.111112p-7f, -0x1.dddddep-32f},
                              {-0x1.555556p-3f, 0x1.555556p-28f}};
  constexpr float CS[8][2] = {{0x1.ae7f3ep-45f, 0x1.ccee08p-71f}, {-0x1.93974ap-37f, -0x1.180f94p-62f},
                              {0x1.1eed8ep-29f, 0x1.ff1b12p-54f}, {-0x1.27e4fcp-22f, 0x1.10ec14p-47f},
                              {0x1.a01a02p-16f, -0x1.7f97fap-42f}, {-0x1.6c16c2p-10f, 0x1.27d27ep-35f},
                              {0x1.555556p-5f, -0x1.555556p-30f}, {-0x1p-1f, 0.0f}};
  FFloat a = {SN[0][0], SN[0][1]};
#pragma unroll
  for (int j = 1; j < 7; ++j) a = ff_add({SN[j][0], SN[j][1]}, ff_mul(z, a));
  a = ff_add({1.0f, 0.0f}, ff_mul(z, a));
  const FFloat sr = ff_mul(r, a);  // sin r
  FFloat c = {CS[0][0], CS[0][1]};
#pragma unroll
  for (int j = 1; j < 8; ++j) c = ff_add({CS[j][0], CS[j][1]}, ff_mul(z, c));
  const FFloat cr = ff_add({1.0f, 0.0f}, ff_mul(z, c));  // cos r
  const FFloat nsr = {-sr.h, -sr.l}, ncr = {-cr.h, -cr.l};
  switch ((int)k & 3) {  // theta = k pi/2 + r
    case 0: sv = sr; cv = cr; break;
    case 1: sv = cr; cv = nsr; break;
    case 2: sv = nsr; cv = ncr; break;
    default: sv = ncr; cv = sr; break;
  }
}

// The chain's bits if [v - e, v + e] (v = h + l) cannot tell them apart.
template <class T, bool MSCALE>
__device__ __forceinline__ bool coef_decided(FFloat v, float e, float scaling, float mscale,
                                             typename Elem<T>::bits& out) {
  const auto b0 = coef_chain<T, MSCALE>(__fadd_rd(v.h, __fsub_rd(v.l, e)), scaling, mscale);
  const auto b1 = coef_chain<T, MSCALE>(__fadd_ru(v.h, __fadd_ru(v.l, e)), scaling, mscale);
  out = b0;
  return b0 == b1;
}

// FF: values the float path leaves open go through ff_sincos before binary64.
// On GB300 one lane's double-float chain takes about as long as one lane's
// binary64 sincos, so a latency-bound launch (the fused kernel) gains nothing;
// a throughput-bound one (the cache build, whose warps share the narrow FP64
// pipe) does.
template <class T, bool MSCALE, bool FF = false>
__device__ __forceinline__ void coef_on_the_fly_bits(int64_t pos, float inv, float scaling, float mscale,
                                                     typename Elem<T>::bits& cb, typename Elem<T>::bits& sb) {
  if constexpr (sizeof(typename Elem<T>::bits) == 2) {
    const float theta = __fmul_rn(__ll2float_rn(pos), inv);
    float sf, cf;
    sincosf(theta, &sf, &cf);
    const float ec = __fmaf_ru(fabsf(cf), 0x1p-20f, 0x1p-100f);
    const float es = __fmaf_ru(fabsf(sf), 0x1p-20f, 0x1p-100f);
    if (coef_decided<T, MSCALE>({cf, 0.0f}, ec, scaling, mscale, cb) &&
        coef_decided<T, MSCALE>({sf, 0.0f}, es, scaling, mscale, sb))
      return;
    if (FF && fabsf(theta) < 0x1p17f) {
      FFloat sv, cv;
      ff_sincos(theta, sv, cv);
      const float fc = __fmaf_ru(fabsf(cv.h), 0x1p-36f, 0x1p-44f);
      const float fs = __fmaf_ru(fabsf(sv.h), 0x1p-36f, 0x1p-44f);
      if (coef_decided<T, MSCALE>(cv, fc, scaling, mscale, cb) && coef_decided<T, MSCALE>(sv, fs, scaling, mscale, sb))
        return;
    }
  }
  float c, s;
  coef_on_the_fly(pos, inv, scaling, c, s);
  cb = coef_chain<T, MSCALE>(c, 1.0f, mscale);
  sb = coef_chain<T, MSCALE>(s, 1.0f, mscale);
}

// Fused rotation: per tile of TTs tokens the CTA first fills a shared-memory
// table of the tile's rd/2 coefficients (coef_on_the_fly_bits once per token
// and index, not per head), then every thread rotates its unit from it.
// MROPE: index i takes the position of its stream (t, h or w, from the stream
// map), and the coefficient is then scaled and rounded to T as the cached
// M-RoPE path does ("com.microsoft.MRotaryEmbedding" README, Description and
// Attributes/scale), so the result equals M-RoPE over rope_cache_build's
// table wherever the positions are inside that table.
template <class T, int V, bool INTER, bool RANK4, bool MROPE>
__global__ void __launch_bounds__(kMaxRowThreads) rope_fused_kernel(const KParams p) {
  using E = Elem<T>;
  using VT = VecT<T, V>;
  using bits = typename E::bits;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  bits* sc = reinterpret_cast<bits*>(smem_raw);
  bits* ss = sc + (size_t)p.TTs * p.h;

  const int tid = threadIdx.x;
  const int per_tok = p.NG * p.Ublk;
  const int slot = tid / per_tok;
  const int r = tid - slot * per_tok;
  const int ng = r / p.Ublk;
  const int k0 = r - ng * p.Ublk;
  const int64_t n = (int64_t)blockIdx.y * p.NG + ng;
  const bool active = slot < p.TTs && n < p.N;

  // x and y may be the same buffer (in place), so neither is __restrict__
  const bits* x = static_cast<const bits*>(p.x);
  bits* y = static_cast<bits*>(p.y);
  const int items = p.TTs * p.h;
  pdl_launch_dependents();
  pdl_wait();

  for (int64_t tile0 = (int64_t)blockIdx.x * p.TTs; tile0 < p.ntok; tile0 += p.step_tok) {
    const int64_t tok = tile0 + slot;
    const bool mine = active && tok < p.ntok;
    int64_t row = 0;
    if (mine) {
      if (RANK4) {
        const int64_t b = tok / p.S, s = tok - (tok / p.S) * p.S;
        row = ((b * p.N + n) * p.S + s) * p.H;
      } else {
        row = (tok * p.N + n) * p.H;
      }
    }
    const bits* xr = x + row;
    bits* yr = y + row;
    // The thread's first pair unit is loaded before the table is built, so its
    // DRAM latency overlaps the coefficients' computation.
    const bool pre = mine && k0 < p.nP;
    int pa = 0, pb = 0;
    VT a0{}, b0{};
    if (pre) {
      unit_offsets<V, INTER>(k0, p.h, pa, pb);
      a0 = ld_stream(reinterpret_cast<const VT*>(xr + pa));
      b0 = ld_stream(reinterpret_cast<const VT*>(xr + pb));
    }
    __syncthreads();  // the previous tile's readers are done with the table
    for (int it = tid; it < items; it += blockDim.x) {
      const int ls = it / p.h;
      const int i = it - ls * p.h;
      const int64_t t = tile0 + ls;
      if (t < p.ntok) {
        int64_t pp;
        if (MROPE) {
          const int st = (int)((p.smap[i >> 4] >> ((i & 15) * 2)) & 3u);
          pp = __ldg(p.pos + st * p.ntok + t);
        } else {
          pp = __ldg(p.pos + t);
        }
        bits cb, sb;
        if (MROPE && !p.mscale_is_one)
          coef_on_the_fly_bits<T, true>(pp, __ldg(p.inv_freq + i), p.scale, p.mscale, cb, sb);
        else
          coef_on_the_fly_bits<T, false>(pp, __ldg(p.inv_freq + i), p.scale, 1.0f, cb, sb);
        sc[it] = cb;
        ss[it] = sb;
      }
    }
    __syncthreads();
    if (!mine) continue;
    for (int k = k0; k < p.U; k += p.Ublk) {
      if (k >= p.nP) {
        const int off = p.rd + (k - p.nP) * V;
        st_stream(reinterpret_cast<VT*>(yr + off), ld_stream(reinterpret_cast<const VT*>(xr + off)));
        continue;
      }
      int oa, ob;
      unit_offsets<V, INTER>(k, p.h, oa, ob);
      VT a, bv;
      if (k == k0) {  // loaded before the table
        a = a0;
        bv = b0;
      } else {
        a = ld_stream(reinterpret_cast<const VT*>(xr + oa));
        bv = ld_stream(reinterpret_cast<const VT*>(xr + ob));
      }
      const VT c = *reinterpret_cast<const VT*>(sc + slot * p.h + k * V);
      const VT sn = *reinterpret_cast<const VT*>(ss + slot * p.h + k * V);
      VT ya, yb;
      rotate_unit<T, V, INTER>(a, bv, c, sn, ya, yb);
      st_stream(reinterpret_cast<VT*>(yr + oa), ya);
      st_stream(reinterpret_cast<VT*>(yr + ob), yb);
    }
  }
}

// (rows, half) cos/sin tables: row p = on-the-fly coefficients of position p,
// through the same coef_on_the_fly_bits as the fused kernel (with the
// double-float step, which gives the same bits).
template <class T>
__global__ void __launch_bounds__(256) rope_cache_build_kernel(const float* __restrict__ inv,
                                                               int32_t half, int64_t rows,
                                                               float scaling, void* cos_out,
                                                               void* sin_out) {
  using E = Elem<T>;
  using bits = typename E::bits;
  bits* co = static_cast<bits*>(cos_out);
  bits* so = static_cast<bits*>(sin_out);
  const int64_t total = rows * half;
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pr = idx / half;
    const int i = (int)(idx - pr * half);
    bits cb, sb;
    coef_on_the_fly_bits<T, false, true>(pr, __ldg(inv + i), scaling, 1.0f, cb, sb);
    co[idx] = cb;
    so[idx] = sb;
  }
}

}  // namespace rope_gb300
