// Rotary position embedding kernels for sm_103a (GB300).
//
// The operation is a streaming, HBM-bound gather/rotate/copy: every element of
// X is read once and every element of Y written once; the cos/sin rows are a
// few percent of the traffic and are shared by all heads of a token. No tensor
// cores: nothing here is a contraction.
//
// Definitions followed (web pages, by title and section):
//  - "ai.onnx.RotaryEmbedding" WebGPU manifest: inputs/X (rank 3
//    (B, S, N*H), rank 4 (B, N, S, H)), inputs/cos_cache and position_ids (2-D
//    table gathered at position_ids[b, s], or a (B, S, rd/2) table),
//    attributeDescriptions/interleaved and rotary_embedding_dim (pairing,
//    partial rotation with pass-through tail).
//  - "com.microsoft.MRotaryEmbedding" README: Inputs/positionIds (three
//    streams, out-of-range pairs copied through), Attributes/mrope_section,
//    mrope_layout, scale, Implementation variants/pairs4 (scaled coefficient
//    rounded to the storage type).
//  - onnxruntime pull request "Add RotaryEmbedding fusion for Qwen3 on-the-fly
//    RoPE patterns": Modeling Code Alignment Check (apply_rotary_pos_emb,
//    rotate_half; cos/sin from inv_freq times attention_scaling), Medium
//    Issues 4 (cache = cos(freqs) * scaling).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "rope_internal.h"

namespace rope_gb300 {

// ---------------------------------------------------------------------------
// Element types: values are carried as their storage bits and converted to
// float32 for arithmetic.
// ---------------------------------------------------------------------------
template <class T>
struct Elem;

template <>
struct Elem<float> {
  using bits = float;
  static __device__ __forceinline__ float tof(float v) { return v; }
  static __device__ __forceinline__ float fromf(float v) { return v; }
  // T(a * b) rounded once from the exact product: a float32 product is
  // already that.
  static __device__ __forceinline__ float mul_round(float a, float b) { return __fmul_rn(a, b); }
};

template <>
struct Elem<__half> {
  using bits = unsigned short;
  static __device__ __forceinline__ float tof(unsigned short v) {
    return __half2float(__ushort_as_half(v));
  }
  static __device__ __forceinline__ unsigned short fromf(float v) {
    return __half_as_ushort(__float2half_rn(v));
  }
  // float16(a * b) rounded once from the exact product. The float32 product
  // is formed with round-to-odd (truncate, then set the last bit if the
  // truncation was inexact); rounding a round-to-odd value with at least two
  // extra bits to nearest-even gives the correctly rounded result (Boldo and
  // Melquiond, "Emulation of FMA and correctly rounded sums: proved
  // algorithms using rounding to odd", IEEE Trans. Computers 57(4), 2008).
  static __device__ __forceinline__ float mul_round(float a, float b) {
    float t = __fmul_rz(a, b);
    float lo = __fmul_rd(a, b);
    float hi = __fmul_ru(a, b);
    if (lo != hi && isfinite(t)) t = __int_as_float(__float_as_int(t) | 1);
    return __half2float(__float2half_rn(t));
  }
};

// bfloat16 (storage beyond the pages' float32 / float16): the top 16 bits of
// a float32.
template <>
struct Elem<__nv_bfloat16> {
  using bits = unsigned short;
  static __device__ __forceinline__ float tof(unsigned short v) { return __uint_as_float((unsigned int)v << 16); }
  static __device__ __forceinline__ unsigned short fromf(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  // bfloat16(a * b) rounded once from the exact product: round-to-odd float32
  // product (16 spare bits), then nearest-even (Boldo and Melquiond, as for
  // float16 above).
  static __device__ __forceinline__ float mul_round(float a, float b) {
    float t = __fmul_rz(a, b);
    float lo = __fmul_rd(a, b);
    float hi = __fmul_ru(a, b);
    if (lo != hi && isfinite(t)) t = __int_as_float(__float_as_int(t) | 1);
    return tof(fromf(t));
  }
};

template <class T, int V>
struct alignas(V * sizeof(typename Elem<T>::bits)) VecT {
  typename Elem<T>::bits v[V];
};

template <int BYTES>
struct Raw;
template <>
struct Raw<16> {
  using t = uint4;
};
template <>
struct Raw<8> {
  using t = uint2;
};
template <>
struct Raw<4> {
  using t = unsigned int;
};
template <>
struct Raw<2> {
  using t = unsigned short;
};

// X is read exactly once: streaming load (evict-first).
template <class VT>
__device__ __forceinline__ VT ld_stream(const VT* p) {
  using R = typename Raw<sizeof(VT)>::t;
  R r = __ldcs(reinterpret_cast<const R*>(p));
  VT v;
  __builtin_memcpy(&v, &r, sizeof(VT));
  return v;
}

// Y is written exactly once: streaming store.
template <class VT>
__device__ __forceinline__ void st_stream(VT* p, const VT& v) {
  using R = typename Raw<sizeof(VT)>::t;
  R r;
  __builtin_memcpy(&r, &v, sizeof(VT));
  __stcs(reinterpret_cast<R*>(p), r);
}

// cos/sin rows and positions are shared by every head of a token: read-only
// path, cached in L1.
template <class VT>
__device__ __forceinline__ VT ld_shared_ro(const VT* p) {
  using R = typename Raw<sizeof(VT)>::t;
  R r = __ldg(reinterpret_cast<const R*>(p));
  VT v;
  __builtin_memcpy(&v, &r, sizeof(VT));
  return v;
}

// One rotation pair in float32: y0 = x0*c - x1*s, y1 = x1*c + x0*s.
__device__ __forceinline__ void rotate(float x0, float x1, float c, float s, float& y0,
                                       float& y1) {
  y0 = __fmaf_rn(x0, c, -__fmul_rn(x1, s));
  y1 = __fmaf_rn(x1, c, __fmul_rn(x0, s));
}

// Pair j of a unit: half-split pairs a[j] with b[j]; interleaved pairs
// elements 2j and 2j+1 of the 2V-element run a||b. Coefficient index j.
template <class T, int V, bool INTER>
struct Pairs {
  using E = Elem<T>;
  using VT = VecT<T, V>;
  static __device__ __forceinline__ typename E::bits get(const VT& a, const VT& b, int q) {
    return q < V ? a.v[q] : b.v[q - V];
  }
  static __device__ __forceinline__ void set(VT& a, VT& b, int q, typename E::bits v) {
    if (q < V)
      a.v[q] = v;
    else
      b.v[q - V] = v;
  }
  static __device__ __forceinline__ int i0(int j) { return INTER ? 2 * j : j; }
  static __device__ __forceinline__ int i1(int j) { return INTER ? 2 * j + 1 : j + V; }
};

// Rotate all V pairs of a unit with coefficient vectors c, s.
template <class T, int V, bool INTER>
struct RotateUnit {
  static __device__ __forceinline__ void run(const VecT<T, V>& a, const VecT<T, V>& b,
                                             const VecT<T, V>& c, const VecT<T, V>& s,
                                             VecT<T, V>& ya, VecT<T, V>& yb) {
    using E = Elem<T>;
    using P = Pairs<T, V, INTER>;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      float x0 = E::tof(P::get(a, b, P::i0(j)));
      float x1 = E::tof(P::get(a, b, P::i1(j)));
      float y0, y1;
      rotate(x0, x1, E::tof(c.v[j]), E::tof(s.v[j]), y0, y1);
      P::set(ya, yb, P::i0(j), E::fromf(y0));
      P::set(ya, yb, P::i1(j), E::fromf(y1));
    }
  }
};

// float16 x 8: the same arithmetic on packed half2 words (two conversions and
// one rounding pack per two values instead of one each).
__device__ __forceinline__ void unpack8(const VecT<__half, 8>& v, __half2 (&w)[4]) {
  __builtin_memcpy(&w, &v, 16);
}
__device__ __forceinline__ void pack8(VecT<__half, 8>& v, const __half2 (&w)[4]) {
  __builtin_memcpy(&v, &w, 16);
}

template <>
struct RotateUnit<__half, 8, false> {
  static __device__ __forceinline__ void run(const VecT<__half, 8>& a, const VecT<__half, 8>& b,
                                             const VecT<__half, 8>& c, const VecT<__half, 8>& s,
                                             VecT<__half, 8>& ya, VecT<__half, 8>& yb) {
    __half2 aw[4], bw[4], cw[4], sw[4], y0w[4], y1w[4];
    unpack8(a, aw);
    unpack8(b, bw);
    unpack8(c, cw);
    unpack8(s, sw);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 x0 = __half22float2(aw[w]);
      const float2 x1 = __half22float2(bw[w]);
      const float2 cf = __half22float2(cw[w]);
      const float2 sf = __half22float2(sw[w]);
      float2 y0, y1;
      rotate(x0.x, x1.x, cf.x, sf.x, y0.x, y1.x);
      rotate(x0.y, x1.y, cf.y, sf.y, y0.y, y1.y);
      y0w[w] = __floats2half2_rn(y0.x, y0.y);
      y1w[w] = __floats2half2_rn(y1.x, y1.y);
    }
    pack8(ya, y0w);
    pack8(yb, y1w);
  }
};

template <>
struct RotateUnit<__half, 8, true> {
  // a||b holds pairs 0..7 as consecutive (even, odd) halves; pair j uses coefficient j.
  static __device__ __forceinline__ void run(const VecT<__half, 8>& a, const VecT<__half, 8>& b,
                                             const VecT<__half, 8>& c, const VecT<__half, 8>& s,
                                             VecT<__half, 8>& ya, VecT<__half, 8>& yb) {
    __half2 aw[4], bw[4], cw[4], sw[4], yaw[4], ybw[4];
    unpack8(a, aw);
    unpack8(b, bw);
    unpack8(c, cw);
    unpack8(s, sw);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 cf = __half22float2(cw[w]);  // coefficients of pairs 2w, 2w+1
      const float2 sf = __half22float2(sw[w]);
      const float2 p0 = __half22float2(w < 2 ? aw[2 * w] : bw[2 * w - 4]);
      const float2 p1 = __half22float2(w < 2 ? aw[2 * w + 1] : bw[2 * w - 3]);
      float2 q0, q1;
      rotate(p0.x, p0.y, cf.x, sf.x, q0.x, q0.y);
      rotate(p1.x, p1.y, cf.y, sf.y, q1.x, q1.y);
      const __half2 h0 = __floats2half2_rn(q0.x, q0.y);
      const __half2 h1 = __floats2half2_rn(q1.x, q1.y);
      if (w < 2) {
        yaw[2 * w] = h0;
        yaw[2 * w + 1] = h1;
      } else {
        ybw[2 * w - 4] = h0;
        ybw[2 * w - 3] = h1;
      }
    }
    pack8(ya, yaw);
    pack8(yb, ybw);
  }
};

template <class T, int V, bool INTER>
__device__ __forceinline__ void rotate_unit(const VecT<T, V>& a, const VecT<T, V>& b,
                                            const VecT<T, V>& c, const VecT<T, V>& s,
                                            VecT<T, V>& ya, VecT<T, V>& yb) {
  RotateUnit<T, V, INTER>::run(a, b, c, s, ya, yb);
}

// ---------------------------------------------------------------------------
// M-RoPE stream merge. A unit's V coefficient indices each follow one of the
// three position streams; instead of choosing per element, the three gathered
// coefficient vectors are merged word by word with bit masks that depend only
// on the unit (so each thread builds them once).
// ---------------------------------------------------------------------------
template <int V>
__device__ __forceinline__ void unit_mask(uint32_t sel, uint32_t (&m)[4]) {
  constexpr int ES = 16 / V;  // bytes per element
  constexpr uint32_t ONES = ES >= 4 ? 0xffffffffu : ((1u << (8 * ES)) - 1u);
#pragma unroll
  for (int w = 0; w < 4; ++w) m[w] = 0;
#pragma unroll
  for (int j = 0; j < V; ++j)
    if ((sel >> j) & 1u) m[(j * ES) / 4] |= ONES << (((j * ES) % 4) * 8);
}

// m0 / m1 select the elements driven by stream 0 / stream 1 (the rest: 2).
template <int V>
__device__ __forceinline__ void stream_masks(uint32_t um, uint32_t (&m0)[4], uint32_t (&m1)[4]) {
  uint32_t s0 = 0, s1 = 0;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const uint32_t st = (um >> (2 * j)) & 3u;
    s0 |= (st == 0u ? 1u : 0u) << j;
    s1 |= (st == 1u ? 1u : 0u) << j;
  }
  unit_mask<V>(s0, m0);
  unit_mask<V>(s1, m1);
}

// Element-wise m0 ? c0 : (m1 ? c1 : c2) on 16-byte vectors.
template <class VT>
__device__ __forceinline__ VT merge3(const VT& c0, const VT& c1, const VT& c2, const uint32_t (&m0)[4],
                                     const uint32_t (&m1)[4]) {
  static_assert(sizeof(VT) == 16, "16-byte units");
  uint32_t a[4], b[4], c[4], r[4];
  __builtin_memcpy(a, &c0, 16);
  __builtin_memcpy(b, &c1, 16);
  __builtin_memcpy(c, &c2, 16);
#pragma unroll
  for (int w = 0; w < 4; ++w) r[w] = (a[w] & m0[w]) | (((b[w] & m1[w]) | (c[w] & ~m1[w])) & ~m0[w]);
  VT out;
  __builtin_memcpy(&out, r, 16);
  return out;
}

// Masks of the output elements of a unit whose pair follows one of the
// streams in `streams` (bit k = stream k). Half split: pair j is element j of
// a and of b; interleaved: pair j is elements 2j, 2j+1 of the run a||b.
template <int V, bool INTER>
__device__ __forceinline__ void pair_masks(uint32_t um, uint32_t streams, uint32_t (&ma)[4],
                                           uint32_t (&mb)[4]) {
  uint32_t sa = 0, sb = 0;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const uint32_t on = (streams >> ((um >> (2 * j)) & 3u)) & 1u;
    if (!INTER) {
      sa |= on << j;
      sb |= on << j;
    } else if (2 * j < V) {
      sa |= (on * 3u) << (2 * j);
    } else {
      sb |= (on * 3u) << (2 * j - V);
    }
  }
  unit_mask<V>(sa, ma);
  unit_mask<V>(sb, mb);
}

// y = m ? y : x, word-wise (restores the pass-through elements).
template <class VT>
__device__ __forceinline__ void blend(VT& y, const VT& x, const uint32_t (&m)[4]) {
  uint32_t a[4], b[4];
  __builtin_memcpy(a, &y, 16);
  __builtin_memcpy(b, &x, 16);
#pragma unroll
  for (int w = 0; w < 4; ++w) a[w] = (a[w] & m[w]) | (b[w] & ~m[w]);
  __builtin_memcpy(&y, a, 16);
}

// The scaled coefficient rounded to T (M-RoPE attribute scale), element-wise.
template <class T, int V>
__device__ __forceinline__ void scale_round(VecT<T, V>& c, float scale) {
  using E = Elem<T>;
#pragma unroll
  for (int j = 0; j < V; ++j) c.v[j] = E::fromf(E::mul_round(E::tof(c.v[j]), scale));
}

// M-RoPE unit with per-element stream choice and per-pair copy-through of
// out-of-range streams (the general path: any V, any validity). Kept out of
// line: it runs only for units that touch an out-of-range position, and
// inlining it would cost the common path registers.
template <class T, int V, bool INTER>
__device__ __noinline__ void mrope_unit_general(const VecT<T, V>& a, const VecT<T, V>& bv,
                                                   const VecT<T, V> (&cs)[3], const VecT<T, V> (&ss)[3],
                                                   uint32_t um, uint32_t valid, bool scaled, float scale,
                                                   VecT<T, V>& ya, VecT<T, V>& yb) {
  using E = Elem<T>;
  using P = Pairs<T, V, INTER>;
  using bits = typename E::bits;
  ya = a;
  yb = bv;
#pragma unroll
  for (int jj = 0; jj < V; ++jj) {
    const int stream = (um >> (2 * jj)) & 3;
    if (!((valid >> stream) & 1u)) continue;  // out-of-range stream: the pair stays
    const bits cb = stream == 0 ? cs[0].v[jj] : (stream == 1 ? cs[1].v[jj] : cs[2].v[jj]);
    const bits sb = stream == 0 ? ss[0].v[jj] : (stream == 1 ? ss[1].v[jj] : ss[2].v[jj]);
    float c = E::tof(cb), sv = E::tof(sb);
    if (scaled) {
      c = E::mul_round(c, scale);
      sv = E::mul_round(sv, scale);
    }
    float y0, y1;
    rotate(E::tof(P::get(a, bv, P::i0(jj))), E::tof(P::get(a, bv, P::i1(jj))), c, sv, y0, y1);
    P::set(ya, yb, P::i0(jj), E::fromf(y0));
    P::set(ya, yb, P::i1(jj), E::fromf(y1));
  }
}

// Offsets (elements, within a head row) of a pair unit's two X vectors.
template <int V, bool INTER>
__device__ __forceinline__ void unit_offsets(int k, int h, int& oa, int& ob) {
  if (INTER) {
    oa = 2 * k * V;
    ob = oa + V;
  } else {
    oa = k * V;
    ob = h + k * V;
  }
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (a no-op when the kernel was
// not launched as a dependent), and let the next kernel be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void flag_oor(int32_t* flag) {
  if (flag) atomicOr(flag, 1);
}

// ---------------------------------------------------------------------------
// Cached RoPE and M-RoPE: coefficients read straight from the table. Each
// thread keeps one (token slot, head, unit) role for its whole life, so there
// is no per-element index arithmetic and no barrier; the 32+ threads of a
// token that need the same cos/sin bytes hit in L1.
// ---------------------------------------------------------------------------
template <class T, int V, bool INTER, bool RANK4, Coef MODE>
__global__ void __launch_bounds__(kMaxRowThreads) rope_rows_kernel(const KParams p) {
  using E = Elem<T>;
  using VT = VecT<T, V>;
  using bits = typename E::bits;
  const int tid = threadIdx.x;
  const int per_tok = p.NG * p.Ublk;
  const int slot = tid / per_tok;
  const int r = tid - slot * per_tok;
  const int ng = r / p.Ublk;
  const int k0 = r - ng * p.Ublk;
  const int64_t n = (int64_t)blockIdx.y * p.NG + ng;
  pdl_launch_dependents();
  pdl_wait();
  if (slot >= p.TTs || n >= p.N) return;  // no barrier below

  // x and y may be the same buffer (in place), so neither is __restrict__
  const bits* x = static_cast<const bits*>(p.x);
  bits* y = static_cast<bits*>(p.y);
  const bits* __restrict__ cosb = static_cast<const bits*>(p.cos);
  const bits* __restrict__ sinb = static_cast<const bits*>(p.sin);

  int64_t tok = (int64_t)blockIdx.x * p.TTs + slot;
  int64_t b = 0, s = 0;
  if (RANK4) {
    b = tok / p.S;
    s = tok - b * p.S;
  }
  for (; tok < p.ntok; tok += p.step_tok) {
    const int64_t row = RANK4 ? ((b * p.N + n) * p.S + s) * p.H : (tok * p.N + n) * p.H;
    const bits* xr = x + row;
    bits* yr = y + row;
    for (int k = k0; k < p.U; k += p.Ublk) {
      if (k >= p.nP) {  // tail unit: bit copy
        const int off = p.rd + (k - p.nP) * V;
        st_stream(reinterpret_cast<VT*>(yr + off), ld_stream(reinterpret_cast<const VT*>(xr + off)));
        continue;
      }
      int oa, ob;
      unit_offsets<V, INTER>(k, p.h, oa, ob);
      const int oc = k * V;
      const VT a = ld_stream(reinterpret_cast<const VT*>(xr + oa));
      const VT bv = ld_stream(reinterpret_cast<const VT*>(xr + ob));
      VT ya, yb;
      if (MODE == Coef::kCache2D || MODE == Coef::kCache3D) {
        int64_t crow;
        if (MODE == Coef::kCache2D) {
          const int64_t pp = __ldg(p.pos + tok);
          if ((uint64_t)pp >= (uint64_t)p.cache_rows) {  // negative or past the table
            if (ng == 0 && k == 0) flag_oor(p.oor_flag);
            st_stream(reinterpret_cast<VT*>(yr + oa), a);
            st_stream(reinterpret_cast<VT*>(yr + ob), bv);
            continue;
          }
          crow = pp * p.h;
        } else {
          crow = tok * p.h;
        }
        const VT c = ld_shared_ro(reinterpret_cast<const VT*>(cosb + crow + oc));
        const VT sn = ld_shared_ro(reinterpret_cast<const VT*>(sinb + crow + oc));
        rotate_unit<T, V, INTER>(a, bv, c, sn, ya, yb);
      } else {  // M-RoPE
        const uint32_t word = p.smap[oc >> 4];
        const uint32_t um = (word >> ((oc & 15) * 2)) & (uint32_t)((1ull << (2 * V)) - 1);
        uint32_t present = 0;
#pragma unroll
        for (int j = 0; j < V; ++j) present |= 1u << ((um >> (2 * j)) & 3);
        uint32_t valid = 0;
        VT cs[3], ss[3];
#pragma unroll
        for (int st = 0; st < 3; ++st) {
          cs[st] = VT{};
          ss[st] = VT{};
          if (present & (1u << st)) {
            const int64_t ps = __ldg(p.pos + st * p.ntok + tok);
            if ((uint64_t)ps < (uint64_t)p.cache_rows) {
              valid |= 1u << st;
              cs[st] = ld_shared_ro(reinterpret_cast<const VT*>(cosb + ps * p.h + oc));
              ss[st] = ld_shared_ro(reinterpret_cast<const VT*>(sinb + ps * p.h + oc));
            } else if (ng == 0) {
              flag_oor(p.oor_flag);
            }
          }
        }
        if constexpr (V * sizeof(bits) == 16) {
          // merge the streams, rotate once, restore pairs of out-of-range streams
          uint32_t m0[4], m1[4];
          stream_masks<V>(um, m0, m1);
          VT c = merge3(cs[0], cs[1], cs[2], m0, m1);
          VT sn = merge3(ss[0], ss[1], ss[2], m0, m1);
          if (!p.scale_is_one) {
            scale_round<T, V>(c, p.scale);
            scale_round<T, V>(sn, p.scale);
          }
          rotate_unit<T, V, INTER>(a, bv, c, sn, ya, yb);
          if (present & ~valid) {
            uint32_t ma[4], mb[4];
            pair_masks<V, INTER>(um, valid, ma, mb);
            blend(ya, a, ma);
            blend(yb, bv, mb);
          }
        } else {
          mrope_unit_general<T, V, INTER>(a, bv, cs, ss, um, valid, !p.scale_is_one, p.scale, ya, yb);
        }
      }
      st_stream(reinterpret_cast<VT*>(yr + oa), ya);
      st_stream(reinterpret_cast<VT*>(yr + ob), yb);
    }
    if (RANK4) {
      s += p.step_s;
      b += p.step_b;
      if (s >= p.S) {
        s -= p.S;
        ++b;
      }
    }
  }
}

}  // namespace rope_gb300
