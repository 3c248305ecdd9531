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

template <class T, bool MSCALE>
__device__ __forceinline__ void coef_on_the_fly_bits(int64_t pos, float inv, float scaling, float mscale,
                                                     typename Elem<T>::bits& cb, typename Elem<T>::bits& sb) {
  if constexpr (sizeof(typename Elem<T>::bits) == 2) {
    const float theta = __fmul_rn(__ll2float_rn(pos), inv);
    float sf, cf;
    sincosf(theta, &sf, &cf);
    const float ec = __fmaf_ru(fabsf(cf), 0x1p-20f, 0x1p-100f);
    const float es = __fmaf_ru(fabsf(sf), 0x1p-20f, 0x1p-100f);
    const auto c0 = coef_chain<T, MSCALE>(__fsub_rd(cf, ec), scaling, mscale);
    const auto c1 = coef_chain<T, MSCALE>(__fadd_ru(cf, ec), scaling, mscale);
    const auto s0 = coef_chain<T, MSCALE>(__fsub_rd(sf, es), scaling, mscale);
    const auto s1 = coef_chain<T, MSCALE>(__fadd_ru(sf, es), scaling, mscale);
    if (c0 == c1 && s0 == s1) {
      cb = c0;
      sb = s0;
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
// through the same coef_on_the_fly_bits as the fused kernel.
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
    coef_on_the_fly_bits<T, false>(pr, __ldg(inv + i), scaling, 1.0f, cb, sb);
    co[idx] = cb;
    so[idx] = sb;
  }
}

}  // namespace rope_gb300
