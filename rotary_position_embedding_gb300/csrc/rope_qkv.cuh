// Q and K rotation for grouped-query attention in one launch, with the
// optional key/value cache append.
//
// Definitions followed (web pages, by title and section):
//  - "com.microsoft.SparseAttention" README: Description (grouped-query heads,
//    separate or packed [Q|K|V] input, partial or full rotary embedding in
//    NeoX or interleaved layout, past key/value updated in place), Inputs
//    (query (B, S, Nq*H) or packed (B, S, (Nq + 2*Nkv)*H); key, value
//    (B, S, Nkv*H); past_key, past_value (B, Nkv, max_cache_len, H)),
//    Attributes (do_rotary: Q and K rotated before K enters the cache;
//    kv_num_heads divides num_heads).
//  - onnxruntime pull request "Add RotaryEmbedding fusion for Qwen3 on-the-fly
//    RoPE patterns": Verification and Qwen3 Architecture (RoPE on both the Q
//    and the K path, GQA with fewer K/V heads; QK-Norm: RMSNorm on Q and K
//    after the projection and before RoPE).
// Every Q and K head is rotated exactly as rope_rows_kernel rotates one head of
// a rank-3 X (same tables, positions, pairing, rotary width and out-of-range
// rule); V heads are copied bit for bit. With NORM, each Q and K head is first
// RMS-normalised: z = T(w * T(x * r)), r = 1/sqrt(mean(x^2) + eps) over the
// head (the products rounded once to T), and z is what gets rotated.
#pragma once

#include "rope_kernels.cuh"

namespace rope_gb300 {

__device__ __forceinline__ void flag_cache_row(int32_t* flag) {
  if (flag) atomicOr(flag, 4);
}

template <class T, int V>
__device__ __forceinline__ float sum_squares(const VecT<T, V>& x) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float v = Elem<T>::tof(x.v[j]);
    s = __fmaf_rn(v, v, s);
  }
  return s;
}

// z_j = T(w_j * T(x_j * r)). Both products are float32 products rounded to
// T; w * n is exact in float32 for float16 data, and x * r (r itself a
// float32 approximation of the exact scale) may land on a float16 midpoint
// only where the exact product is within 2^-24 of it -- inside the one-ulp
// flips that r's own error already allows.
template <class T, int V>
__device__ __forceinline__ VecT<T, V> norm_weight(const VecT<T, V>& x, float r, const VecT<T, V>& w) {
  using E = Elem<T>;
  VecT<T, V> z;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float n = E::tof(E::fromf(__fmul_rn(E::tof(x.v[j]), r)));
    z.v[j] = E::fromf(__fmul_rn(n, E::tof(w.v[j])));
  }
  return z;
}

// The kernel sees each token as N = Nq + Nkv (+ Nkv in cache mode) head rows
// in the packed [Q|K|V] order and keeps rope_rows_kernel's fixed thread roles
// (KParams): a thread's head row -- and with it its source, its destination and
// whether it rotates -- never changes, so the routing is decided once.
// Register cap. A token's 48 head rows (Qwen3-8B shape) make 384-thread CTAs;
// uncapped the kernel takes 58 registers, so only 2 CTAs fit an SM. At 48
// registers 3 fit (a few bytes of spills): the prefill workload runs 41.0 us
// instead of 45.1 us (40 registers: 4 CTAs but heavier spills, 43.0 us).
#ifndef ROPE_QKV_MAXNREG
#define ROPE_QKV_MAXNREG 48
#endif
// With RMSNorm a lane also holds the weights and its cos/sin while the
// head's mean is formed: 56 registers (still 3 CTAs of 384 threads per SM).
#ifndef ROPE_QKV_NORM_MAXNREG
#define ROPE_QKV_NORM_MAXNREG 56
#endif
#ifndef ROPE_QKV_NORM_HOIST
#define ROPE_QKV_NORM_HOIST 1
#endif
// M-RoPE heads gather three coefficient rows per unit and merge them: their
// own cap. 80 registers keep two CTAs of 384 threads per SM, as 64 do, without
// spills (M-RoPE QK-Norm decode, 256 tokens: 5.2 us from a graph; 5.9 us at 64).
#ifndef ROPE_QKV_MROPE_MAXNREG
#define ROPE_QKV_MROPE_MAXNREG 80
#endif
#define ROPE_QKV_BOUNDS \
  __maxnreg__(MROPE ? ROPE_QKV_MROPE_MAXNREG : (NORM ? ROPE_QKV_NORM_MAXNREG : ROPE_QKV_MAXNREG))

// M-RoPE rotation of one unit of a Q or K head ("com.microsoft.MRotaryEmbedding"
// README, Inputs/positionIds and Attributes): each of the unit's V coefficient
// indices follows its stream's position pos3[stream, token]; a pair whose
// position is outside the table is copied through (and reported in *oor);
// the gathered coefficients are scaled and rounded to T first. 128-bit units
// merge the three streams by bit masks; single-element units take the general
// per-pair form (mrope_unit_general).
template <class T, int V, bool INTER>
__device__ __forceinline__ void mrope_qkv_unit(const KParams& p, int64_t tok, int k, const VecT<T, V>& a,
                                               const VecT<T, V>& bv, VecT<T, V>& ya, VecT<T, V>& yb,
                                               bool& oor) {
  using VT = VecT<T, V>;
  using bits = typename Elem<T>::bits;
  const int oc = k * V;
  const uint32_t word = p.smap[oc >> 4];
  const uint32_t um = (word >> ((oc & 15) * 2)) & (uint32_t)((1ull << (2 * V)) - 1);
  uint32_t present = 0, valid = 0;
#pragma unroll
  for (int j = 0; j < V; ++j) present |= 1u << ((um >> (2 * j)) & 3);
  const bits* cosb = static_cast<const bits*>(p.cos);
  const bits* sinb = static_cast<const bits*>(p.sin);
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
      }
    }
  }
  if (present & ~valid) oor = true;
  if constexpr (V * sizeof(bits) == 16) {
    // 128-bit units: merge the streams with bit masks, rotate once, restore
    // the pairs of out-of-range streams (as rope_rows_kernel does)
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

template <class T, int V, bool INTER, bool IMPLICIT, bool NORM, bool MROPE = false>
__global__ void ROPE_QKV_BOUNDS rope_qkv_kernel(const KParams p, const QKVParams a) {
  using VT = VecT<T, V>;
  using bits = typename Elem<T>::bits;
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

  // role 0: Q head, 1: K head, 2: V head (cache mode only)
  const int role = n < a.Nq ? 0 : (n < a.Nq + a.Nkv ? 1 : 2);
  const int64_t hd = role == 0 ? n : (role == 1 ? n - a.Nq : n - a.Nq - a.Nkv);
  const int64_t H = p.H;
  const bits* src;
  int64_t sstride;  // elements between the rows of consecutive tokens
  if (a.packed) {
    src = static_cast<const bits*>(p.x) + n * H;
    sstride = (int64_t)(a.Nq + 2 * a.Nkv) * H;
  } else {
    const void* base = role == 0 ? p.x : (role == 1 ? a.k : a.v);
    src = static_cast<const bits*>(base) + hd * H;
    sstride = (int64_t)(role == 0 ? a.Nq : a.Nkv) * H;
  }
  const bool to_cache = role != 0 && a.cache;
  bits* dst;
  int64_t dstride = 0;
  if (role == 0) {
    dst = static_cast<bits*>(p.y) + hd * H;
    dstride = (int64_t)a.Nq * H;
  } else if (!a.cache) {
    dst = static_cast<bits*>(a.k_out) + hd * H;
    dstride = (int64_t)a.Nkv * H;
  } else {
    dst = static_cast<bits*>(role == 1 ? a.k_cache : a.v_cache) + hd * a.max_len * H;
  }
  const bool rotates = role != 2;
  const bits* __restrict__ cosb = static_cast<const bits*>(p.cos);
  const bits* __restrict__ sinb = static_cast<const bits*>(p.sin);
  // NORM: a row's Ublk lanes (a power of two <= 32, one unit each) are an
  // aligned group of its warp; they add up the row's squares with shuffles.
  unsigned gmask = 0u;
  if (NORM) {
    const unsigned lane = threadIdx.x & 31u;
    gmask = p.Ublk >= 32 ? 0xffffffffu : (((1u << p.Ublk) - 1u) << (lane & ~(unsigned)(p.Ublk - 1)));
  }

  int64_t tok = (int64_t)blockIdx.x * p.TTs + slot;
  int64_t b = tok / p.S;
  int64_t s = tok - b * p.S;
  for (; tok < p.ntok; tok += p.step_tok) {
    const int64_t past = a.past ? (int64_t)__ldg(a.past + b) : 0;
    const bits* xr = src + tok * sstride;
    bits* yr = nullptr;
    if (to_cache) {
      const int64_t row = past + s;
      if (row >= 0 && row < a.max_len) {
        yr = dst + (b * a.Nkv * a.max_len + row) * H;
      } else if (role == 1 && hd == 0 && k0 == 0) {
        flag_cache_row(p.oor_flag);
      }
    } else {
      yr = dst + tok * dstride;
    }
    if (yr) {
      bool valid = false;
      int64_t crow = 0;
      if (rotates && !MROPE) {
        const int64_t pp = IMPLICIT ? past + s : __ldg(p.pos + tok);
        valid = (uint64_t)pp < (uint64_t)p.cache_rows;
        if (!valid && role == 0 && hd == 0 && k0 == 0) flag_oor(p.oor_flag);
        crow = pp * p.h;
      }
      if (MROPE) valid = rotates;  // out-of-range streams are handled pair by pair
      bool oor = false;
      if (NORM && rotates) {
        // at most one unit per lane; lanes past the row's units add zeros
        const bool has = k0 < p.U;
        const bool tail = k0 >= p.nP;
        int oa = 0, ob = 0;
        if (tail)
          oa = p.rd + (k0 - p.nP) * V;
        else
          unit_offsets<V, INTER>(k0, p.h, oa, ob);
        // every load that does not depend on the mean goes out before the
        // reduction, so their latencies overlap X's
        VT xa{}, xb{}, wa{}, wb{}, c{}, sn{};
        const bits* w = static_cast<const bits*>(role == 0 ? a.qw : a.kw);
        if (has) {
          xa = ld_stream(reinterpret_cast<const VT*>(xr + oa));
          if (!tail) xb = ld_stream(reinterpret_cast<const VT*>(xr + ob));
#if ROPE_QKV_NORM_HOIST
          wa = ld_shared_ro(reinterpret_cast<const VT*>(w + oa));
          if (!tail) {
            wb = ld_shared_ro(reinterpret_cast<const VT*>(w + ob));
            if (valid && !MROPE) {
              const int oc = k0 * V;
              c = ld_shared_ro(reinterpret_cast<const VT*>(cosb + crow + oc));
              sn = ld_shared_ro(reinterpret_cast<const VT*>(sinb + crow + oc));
            }
          }
#endif
        }
        float ss = sum_squares<T, V>(xa) + sum_squares<T, V>(xb);
        for (int o = p.Ublk >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(gmask, ss, o);
        const float r = 1.0f / sqrtf(ss / (float)H + a.eps);
#if !ROPE_QKV_NORM_HOIST
        if (has) {
          wa = ld_shared_ro(reinterpret_cast<const VT*>(w + oa));
          if (!tail) {
            wb = ld_shared_ro(reinterpret_cast<const VT*>(w + ob));
            if (valid && !MROPE) {
              const int oc = k0 * V;
              c = ld_shared_ro(reinterpret_cast<const VT*>(cosb + crow + oc));
              sn = ld_shared_ro(reinterpret_cast<const VT*>(sinb + crow + oc));
            }
          }
        }
#endif
        if (has) {
          const VT za = norm_weight<T, V>(xa, r, wa);
          if (tail) {
            st_stream(reinterpret_cast<VT*>(yr + oa), za);
          } else {
            const VT zb = norm_weight<T, V>(xb, r, wb);
            if (valid) {
              VT ya, yb;
              if (MROPE)
                mrope_qkv_unit<T, V, INTER>(p, tok, k0, za, zb, ya, yb, oor);
              else
                rotate_unit<T, V, INTER>(za, zb, c, sn, ya, yb);
              st_stream(reinterpret_cast<VT*>(yr + oa), ya);
              st_stream(reinterpret_cast<VT*>(yr + ob), yb);
            } else {  // out-of-range position: the normalised head passes through
              st_stream(reinterpret_cast<VT*>(yr + oa), za);
              st_stream(reinterpret_cast<VT*>(yr + ob), zb);
            }
          }
        }
      } else {
        for (int k = k0; k < p.U; k += p.Ublk) {
          if (k >= p.nP) {  // tail unit: bit copy
            const int off = p.rd + (k - p.nP) * V;
            st_stream(reinterpret_cast<VT*>(yr + off), ld_stream(reinterpret_cast<const VT*>(xr + off)));
            continue;
          }
          int oa, ob;
          unit_offsets<V, INTER>(k, p.h, oa, ob);
          const VT xa = ld_stream(reinterpret_cast<const VT*>(xr + oa));
          const VT xb = ld_stream(reinterpret_cast<const VT*>(xr + ob));
          if (!valid) {  // V head, or an out-of-range position: copied through
            st_stream(reinterpret_cast<VT*>(yr + oa), xa);
            st_stream(reinterpret_cast<VT*>(yr + ob), xb);
            continue;
          }
          VT ya, yb;
          if (MROPE) {
            mrope_qkv_unit<T, V, INTER>(p, tok, k, xa, xb, ya, yb, oor);
          } else {
            const int oc = k * V;
            const VT c = ld_shared_ro(reinterpret_cast<const VT*>(cosb + crow + oc));
            const VT sn = ld_shared_ro(reinterpret_cast<const VT*>(sinb + crow + oc));
            rotate_unit<T, V, INTER>(xa, xb, c, sn, ya, yb);
          }
          st_stream(reinterpret_cast<VT*>(yr + oa), ya);
          st_stream(reinterpret_cast<VT*>(yr + ob), yb);
        }
      }
      if (MROPE && oor && role == 0) flag_oor(p.oor_flag);
    }
    s += p.step_s;
    b += p.step_b;
    if (s >= p.S) {
      s -= p.S;
      ++b;
    }
  }
}

}  // namespace rope_gb300
