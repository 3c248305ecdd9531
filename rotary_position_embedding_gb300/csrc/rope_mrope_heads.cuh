// Cached M-RoPE on the SIMT path, several heads per thread, for sm_103a.
//
// Thread roles: token slot, head group g (heads g*HPT .. g*HPT + HPT-1) and
// unit k of the head row. A pair-unit thread first issues the X loads of all
// its heads (so a thread keeps 2*HPT 16-byte loads in flight), then loads the
// token's stream positions and the in-range rows' coefficient pieces for unit
// k, merges them once by the stream map's element masks, applies the scale
// step and rotates every head with them, putting back the pairs of
// out-of-range streams. The coefficients are gathered and merged once per HPT
// heads, with no barrier and no shared memory. Tail units copy their heads'
// elements past the rotary width. KParams: NG = head groups per token,
// Ublk = U (every unit of a row has its thread).
//
// The rotation is the scalar form: float32x2 rotation with coefficients
// unpacked once measured the same at 4 heads per thread and erratic at 7 or 8
// (bfloat16 up to 1.5x slower at the 128-register cap).
//
// Definitions followed: "com.microsoft.MRotaryEmbedding" README (Description,
// Inputs/positionIds, Attributes mrope_section, mrope_layout, scale) -- the
// same arithmetic as the rows kernel and the TMA pipeline, which this file
// shares through rope_kernels.cuh.
#pragma once

#include "rope_kernels.cuh"

namespace rope_gb300 {

template <class T, int V, bool INTER, bool RANK4, int HPT>
__global__ void __launch_bounds__(kMaxRowThreads) rope_mrope_heads_kernel(const KParams p) {
  using E = Elem<T>;
  using VT = VecT<T, V>;
  using bits = typename E::bits;
  static_assert(V * sizeof(bits) == 16, "128-bit units only");
  const int tid = threadIdx.x;
  const int per_tok = p.NG * p.U;
  const int slot = tid / per_tok;
  const int r = tid - slot * per_tok;
  const int grp = r / p.U;
  const int k = r - grp * p.U;
  const int64_t n0 = (int64_t)grp * HPT;
  if (slot >= p.TTs || n0 >= p.N) return;  // no barrier below
  const int nP = p.nP;

  // x and y may be the same buffer (in place), so neither is __restrict__
  const bits* x = static_cast<const bits*>(p.x);
  bits* y = static_cast<bits*>(p.y);
  const bits* __restrict__ cosb = static_cast<const bits*>(p.cos);
  const bits* __restrict__ sinb = static_cast<const bits*>(p.sin);
  pdl_launch_dependents();
  pdl_wait();

  // the unit's stream map and element masks, fixed for the thread's life
  int oa = 0, ob = 0;
  uint32_t um = 0, present = 0;
  uint32_t m0[4] = {0, 0, 0, 0}, m1[4] = {0, 0, 0, 0};  // elements of stream 0 / 1 (the rest: 2)
  if (k < nP) {
    unit_offsets<V, INTER>(k, p.h, oa, ob);
    const int oc = k * V;
    const uint32_t word = p.smap[oc >> 4];
    um = (word >> ((oc & 15) * 2)) & (uint32_t)((1ull << (2 * V)) - 1);
#pragma unroll
    for (int j = 0; j < V; ++j) present |= 1u << ((um >> (2 * j)) & 3u);
    stream_masks<V>(um, m0, m1);
  }
  const int64_t hstride = RANK4 ? p.S * p.H : p.H;  // elements between heads n and n+1 of a token
  for (int64_t tok = (int64_t)blockIdx.x * p.TTs + slot; tok < p.ntok; tok += p.step_tok) {
    int64_t row0;  // element offset of head n0 of the token
    if (RANK4) {
      const int64_t b = tok / p.S, s = tok - b * p.S;
      row0 = ((b * p.N + n0) * p.S + s) * p.H;
    } else {
      row0 = (tok * p.N + n0) * p.H;
    }
    if (k >= nP) {  // tail unit: bit copy of every head's elements [rd + (k-nP)*V, ...)
      const int off = p.rd + (k - nP) * V;
#pragma unroll
      for (int j = 0; j < HPT; ++j) {
        if (n0 + j >= p.N) break;
        const int64_t o = row0 + j * hstride + off;
        st_stream(reinterpret_cast<VT*>(y + o), ld_stream(reinterpret_cast<const VT*>(x + o)));
      }
      continue;
    }
    VT a[HPT], bv[HPT];
#pragma unroll
    for (int j = 0; j < HPT; ++j) {
      if (n0 + j < p.N) {
        a[j] = ld_stream(reinterpret_cast<const VT*>(x + row0 + j * hstride + oa));
        bv[j] = ld_stream(reinterpret_cast<const VT*>(x + row0 + j * hstride + ob));
      }
    }
    const int oc = k * V;
    int64_t ps[3];
#pragma unroll
    for (int st = 0; st < 3; ++st) ps[st] = (present & (1u << st)) ? __ldg(p.pos + st * p.ntok + tok) : -1;
    uint32_t valid = 0;
    uint32_t cw[4] = {0, 0, 0, 0}, sw[4] = {0, 0, 0, 0};
#pragma unroll
    for (int st = 0; st < 3; ++st) {
      if ((present & (1u << st)) && (uint64_t)ps[st] < (uint64_t)p.cache_rows) {
        valid |= 1u << st;
        const VT cv = ld_shared_ro(reinterpret_cast<const VT*>(cosb + ps[st] * p.h + oc));
        const VT sv2 = ld_shared_ro(reinterpret_cast<const VT*>(sinb + ps[st] * p.h + oc));
        uint32_t cu[4], su[4];
        __builtin_memcpy(cu, &cv, 16);
        __builtin_memcpy(su, &sv2, 16);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t m = st == 0 ? m0[w] : (st == 1 ? m1[w] : ~(m0[w] | m1[w]));
          cw[w] |= cu[w] & m;
          sw[w] |= su[w] & m;
        }
      }
    }
    if ((present & ~valid) && grp == 0) flag_oor(p.oor_flag);
    VT c, sn;
    __builtin_memcpy(&c, cw, 16);
    __builtin_memcpy(&sn, sw, 16);
    if (!p.scale_is_one) {
      scale_round<T, V>(c, p.scale);
      scale_round<T, V>(sn, p.scale);
    }
    const bool blend_on = (present & ~valid) != 0;
    uint32_t ma[4] = {0, 0, 0, 0}, mb[4] = {0, 0, 0, 0};
    if (blend_on) pair_masks<V, INTER>(um, valid, ma, mb);
#pragma unroll
    for (int j = 0; j < HPT; ++j) {
      if (n0 + j >= p.N) break;
      VT ya, yb;
      rotate_unit<T, V, INTER>(a[j], bv[j], c, sn, ya, yb);
      if (blend_on) {  // pairs of out-of-range streams keep their input
        blend(ya, a[j], ma);
        blend(yb, bv[j], mb);
      }
      st_stream(reinterpret_cast<VT*>(y + row0 + j * hstride + oa), ya);
      st_stream(reinterpret_cast<VT*>(y + row0 + j * hstride + ob), yb);
    }
  }
}

}  // namespace rope_gb300
