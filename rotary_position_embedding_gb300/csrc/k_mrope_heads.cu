// MRotaryEmbedding, SIMT path with several heads per thread: kernel instances
// for 2 and 4 heads per thread ("com.microsoft.MRotaryEmbedding" README:
// three position streams, section select, scale, out-of-range copy-through).
#include "rope_mrope_heads.cuh"

namespace rope_gb300 {

namespace {
template <class T, int V, int HPT>
const void* pick_heads(bool inter, bool rank4) {
  if (inter)
    return rank4 ? (const void*)rope_mrope_heads_kernel<T, V, true, true, HPT>
                 : (const void*)rope_mrope_heads_kernel<T, V, true, false, HPT>;
  return rank4 ? (const void*)rope_mrope_heads_kernel<T, V, false, true, HPT>
               : (const void*)rope_mrope_heads_kernel<T, V, false, false, HPT>;
}

template <int HPT>
const void* pick_dtype(int dtype, bool inter, bool rank4) {
  if (dtype == 0) return pick_heads<float, 4, HPT>(inter, rank4);
  if (dtype == 1) return pick_heads<__half, 8, HPT>(inter, rank4);
  if (dtype == 2) return pick_heads<__nv_bfloat16, 8, HPT>(inter, rank4);
  return nullptr;
}
}  // namespace

const void* rope_kernel_mrope_heads(int dtype, bool inter, bool rank4, int hpt) {
  if (hpt == 2) return pick_dtype<2>(dtype, inter, rank4);
  if (hpt == 4) return pick_dtype<4>(dtype, inter, rank4);
  return nullptr;
}

}  // namespace rope_gb300
