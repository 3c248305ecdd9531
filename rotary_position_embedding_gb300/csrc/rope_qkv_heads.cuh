// Q and K rotation with the key/value cache append (and the optional
// QK-RMSNorm), SIMT, several heads per thread, for sm_103a.
//
// The operation of rope_qkv_kernel (rope_qkv.cuh) on the 128-bit path: every Q
// and K head rotated as rope_rows_kernel rotates one head of a rank-3 X, V
// heads copied, K and V appended to the caches at rows past[b] + s; with NORM
// each Q and K head is RMS-normalised first. Here a thread owns unit k of HPT
// heads of one role (Q, K or V) for its whole life: it issues the X loads of
// all its heads first (2*HPT 16-byte loads in flight), then loads the unit's
// cos/sin (and norm weights) once and rotates every head with them. With NORM
// a head's U units are an aligned power-of-two lane group that adds up each of
// its heads' squares with shuffles, HPT reductions side by side; on 16-bit
// data the normalisation and rotation take the packed float32x2 form of
// rope_packed.cuh (faster at the sizes this kernel gets the norm), otherwise
// the scalar one; both round every value alike. KParams:
// NG = head groups per token (ceil(Nq/HPT) + ceil(Nkv/HPT) [+ ceil(Nkv/HPT)
// with caches]; with RAGGED a role's last group may hold fewer heads, without
// it HPT divides both head counts), U = units per head row, Ublk = U.
//
// Definitions followed (web pages, by title and section): "com.microsoft.
// SparseAttention" README (Description, Inputs, Attributes do_rotary,
// kv_num_heads); onnxruntime pull request "Add RotaryEmbedding fusion for
// Qwen3 on-the-fly RoPE patterns" (Verification, Qwen3 Architecture: QK-Norm
// before RoPE). Same arithmetic as rope_qkv_kernel, whose helpers it uses.
#pragma once

#include "rope_packed.cuh"
#include "rope_qkv.cuh"

namespace rope_gb300 {

template <class T, int V, bool INTER, bool IMPLICIT, bool NORM, int HPT, bool RAGGED>
__global__ void __launch_bounds__(kMaxRowThreads) rope_qkv_heads_kernel(const KParams p, const QKVParams a) {
  using VT = VecT<T, V>;
  using bits = typename Elem<T>::bits;
  static_assert(V * sizeof(bits) == 16, "128-bit units only");
  const int tid = threadIdx.x;
  const int U = p.U;
  const int per_tok = p.NG * U;
  const int slot = tid / per_tok;
  const int r = tid - slot * per_tok;
  const int grp = r / U;
  const int k = r - grp * U;
  pdl_launch_dependents();
  pdl_wait();
  if (slot >= p.TTs) return;  // a whole token slot: no head group is split

  // role 0: Q heads, 1: K heads, 2: V heads (cache mode only); a role's last
  // group holds the remainder of its heads (nh of them)
  const int gq = (a.Nq + HPT - 1) / HPT, gk = (a.Nkv + HPT - 1) / HPT;
  const int role = grp < gq ? 0 : (grp < gq + gk ? 1 : 2);
  const int64_t hd0 = (int64_t)(role == 0 ? grp : (role == 1 ? grp - gq : grp - gq - gk)) * HPT;
  // heads of the group: HPT unless RAGGED and the role's last group is short
  const int nh = RAGGED ? (int)min((int64_t)HPT, (role == 0 ? a.Nq : a.Nkv) - hd0) : HPT;
  const int64_t H = p.H;
  const bits* src;
  int64_t sstride;  // elements between the rows of consecutive tokens
  if (a.packed) {
    const int64_t n0 = role == 0 ? hd0 : (role == 1 ? a.Nq + hd0 : (int64_t)a.Nq + a.Nkv + hd0);
    src = static_cast<const bits*>(p.x) + n0 * H;
    sstride = (int64_t)(a.Nq + 2 * a.Nkv) * H;
  } else {
    const void* base = role == 0 ? p.x : (role == 1 ? a.k : a.v);
    src = static_cast<const bits*>(base) + hd0 * H;
    sstride = (int64_t)(role == 0 ? a.Nq : a.Nkv) * H;
  }
  const bool to_cache = role != 0 && a.cache;
  bits* dst;
  int64_t dstride = 0;   // destination elements between consecutive tokens
  int64_t dhead = H;     // destination elements between heads j and j+1 of the group
  if (role == 0) {
    dst = static_cast<bits*>(p.y) + hd0 * H;
    dstride = (int64_t)a.Nq * H;
  } else if (!a.cache) {
    dst = static_cast<bits*>(a.k_out) + hd0 * H;
    dstride = (int64_t)a.Nkv * H;
  } else {
    dst = static_cast<bits*>(role == 1 ? a.k_cache : a.v_cache) + hd0 * a.max_len * H;
    dhead = a.max_len * H;
  }
  const bool rotates = role != 2;
  const bool pair = k < p.nP;
  int oa = 0, ob = 0;
  if (pair)
    unit_offsets<V, INTER>(k, p.h, oa, ob);
  else
    oa = p.rd + (k - p.nP) * V;
  const int oc = k * V;
  const bits* __restrict__ cosb = static_cast<const bits*>(p.cos);
  const bits* __restrict__ sinb = static_cast<const bits*>(p.sin);
  // NORM: the row's U lanes (a power of two <= 32) are an aligned group of the warp
  unsigned gmask = 0u;
  VT wa{}, wb{};
  if (NORM) {
    const unsigned lane = threadIdx.x & 31u;
    gmask = U >= 32 ? 0xffffffffu : (((1u << U) - 1u) << (lane & ~(unsigned)(U - 1)));
    if (rotates) {  // the role's channel weights: the same for every head of the group
      const bits* w = static_cast<const bits*>(role == 0 ? a.qw : a.kw);
      wa = ld_shared_ro(reinterpret_cast<const VT*>(w + oa));
      if (pair) wb = ld_shared_ro(reinterpret_cast<const VT*>(w + ob));
    }
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
      } else if (role == 1 && hd0 == 0 && k == 0) {
        flag_cache_row(p.oor_flag);
      }
    } else {
      yr = dst + tok * dstride;
    }
    if (yr) {  // the same for every lane of a head group (one token, one role)
      VT xa[HPT], xb[HPT];
#pragma unroll
      for (int j = 0; j < HPT; ++j) {  // a short group reads its last head again
        const bits* xj = xr + (j < nh ? j : nh - 1) * H;
        xa[j] = ld_stream(reinterpret_cast<const VT*>(xj + oa));
        xb[j] = VT{};
        if (pair) xb[j] = ld_stream(reinterpret_cast<const VT*>(xj + ob));
      }
      bool valid = false;
      VT c{}, sn{};
      if (rotates) {
        const int64_t pp = IMPLICIT ? past + s : __ldg(p.pos + tok);
        valid = (uint64_t)pp < (uint64_t)p.cache_rows;
        if (!valid && role == 0 && hd0 == 0 && k == 0) flag_oor(p.oor_flag);
        if (valid && pair) {
          c = ld_shared_ro(reinterpret_cast<const VT*>(cosb + pp * p.h + oc));
          sn = ld_shared_ro(reinterpret_cast<const VT*>(sinb + pp * p.h + oc));
        }
      }
      if constexpr (NORM && sizeof(bits) == 2) {
        // 16-bit data: the packed form (float32x2 products, coefficients
        // unpacked once per unit), which rounds every lane as the scalar form
        // below does
        if (rotates) {
          using P = P2<T>;
          float2 fa[HPT][4], fb[HPT][4];
          float ss[HPT];
#pragma unroll
          for (int j = 0; j < HPT; ++j) {
            Unit8<T> ua, ub;
            __builtin_memcpy(&ua, &xa[j], 16);
            __builtin_memcpy(&ub, &xb[j], 16);
            float sa = 0.f, sb = 0.f;  // sum_squares' order: a's eight values, then b's
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              fa[j][q] = P::tof(ua.w[q]);
              fb[j][q] = P::tof(ub.w[q]);
              sa = __fmaf_rn(fa[j][q].x, fa[j][q].x, sa);
              sa = __fmaf_rn(fa[j][q].y, fa[j][q].y, sa);
              sb = __fmaf_rn(fb[j][q].x, fb[j][q].x, sb);
              sb = __fmaf_rn(fb[j][q].y, fb[j][q].y, sb);
            }
            ss[j] = sa + sb;
          }
          for (int o = U >> 1; o > 0; o >>= 1) {
#pragma unroll
            for (int j = 0; j < HPT; ++j) ss[j] += __shfl_xor_sync(gmask, ss[j], o);
          }
          float2 cf[4], sf[4];
          if (valid && pair) {
            unpack_coef8<T>(c, cf);
            unpack_coef8<T>(sn, sf);
          }
          Unit8<T> wua, wub;
          __builtin_memcpy(&wua, &wa, 16);
          __builtin_memcpy(&wub, &wb, 16);
#pragma unroll
          for (int j = 0; j < HPT; ++j) {
            if (j >= nh) break;
            const float rr = 1.0f / sqrtf(ss[j] / (float)H + a.eps);
            const Unit8<T> za = norm8p<T>(fa[j], rr, wua);
            bits* yj = yr + j * dhead;
            if (!pair) {
              st_stream(reinterpret_cast<VT*>(yj + oa), *reinterpret_cast<const VT*>(&za));
              continue;
            }
            const Unit8<T> zb = norm8p<T>(fb[j], rr, wub);
            if (valid) {
              Unit8<T> ya, yb;
              rotate8p<T, INTER>(za, zb, cf, sf, ya, yb);
              st_stream(reinterpret_cast<VT*>(yj + oa), *reinterpret_cast<const VT*>(&ya));
              st_stream(reinterpret_cast<VT*>(yj + ob), *reinterpret_cast<const VT*>(&yb));
            } else {  // out-of-range position: the normalised head passes through
              st_stream(reinterpret_cast<VT*>(yj + oa), *reinterpret_cast<const VT*>(&za));
              st_stream(reinterpret_cast<VT*>(yj + ob), *reinterpret_cast<const VT*>(&zb));
            }
          }
        } else {  // V heads: copied
#pragma unroll
          for (int j = 0; j < HPT; ++j) {
            if (j >= nh) break;
            bits* yj = yr + j * dhead;
            st_stream(reinterpret_cast<VT*>(yj + oa), xa[j]);
            if (pair) st_stream(reinterpret_cast<VT*>(yj + ob), xb[j]);
          }
        }
      } else if (NORM && rotates) {
        float ss[HPT];
#pragma unroll
        for (int j = 0; j < HPT; ++j) ss[j] = sum_squares<T, V>(xa[j]) + sum_squares<T, V>(xb[j]);
        for (int o = U >> 1; o > 0; o >>= 1) {
#pragma unroll
          for (int j = 0; j < HPT; ++j) ss[j] += __shfl_xor_sync(gmask, ss[j], o);
        }
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
          if (j >= nh) break;
          const float rr = 1.0f / sqrtf(ss[j] / (float)H + a.eps);
          const VT za = norm_weight<T, V>(xa[j], rr, wa);
          bits* yj = yr + j * dhead;
          if (!pair) {
            st_stream(reinterpret_cast<VT*>(yj + oa), za);
            continue;
          }
          const VT zb = norm_weight<T, V>(xb[j], rr, wb);
          if (valid) {
            VT ya, yb;
            rotate_unit<T, V, INTER>(za, zb, c, sn, ya, yb);
            st_stream(reinterpret_cast<VT*>(yj + oa), ya);
            st_stream(reinterpret_cast<VT*>(yj + ob), yb);
          } else {  // out-of-range position: the normalised head passes through
            st_stream(reinterpret_cast<VT*>(yj + oa), za);
            st_stream(reinterpret_cast<VT*>(yj + ob), zb);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
          if (j >= nh) break;
          bits* yj = yr + j * dhead;
          if (pair && valid) {
            VT ya, yb;
            rotate_unit<T, V, INTER>(xa[j], xb[j], c, sn, ya, yb);
            st_stream(reinterpret_cast<VT*>(yj + oa), ya);
            st_stream(reinterpret_cast<VT*>(yj + ob), yb);
          } else {  // V head, tail unit or out-of-range position: copied through
            st_stream(reinterpret_cast<VT*>(yj + oa), xa[j]);
            if (pair) st_stream(reinterpret_cast<VT*>(yj + ob), xb[j]);
          }
        }
      }
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
