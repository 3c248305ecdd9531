// On-the-fly RoPE and M-RoPE (cos/sin from inv_freq) and the cos/sin cache
// build (the onnxruntime Qwen3 on-the-fly RoPE fusion pull request: Modeling
// Code Alignment Check, Medium Issues 4; "com.microsoft.MRotaryEmbedding"
// README for the three position streams).
#include "rope_fused.cuh"

namespace rope_gb300 {

namespace {
template <class T, int V, bool MROPE>
const void* pick(bool inter, bool rank4) {
  if (inter)
    return rank4 ? (const void*)rope_fused_kernel<T, V, true, true, MROPE>
                 : (const void*)rope_fused_kernel<T, V, true, false, MROPE>;
  return rank4 ? (const void*)rope_fused_kernel<T, V, false, true, MROPE>
               : (const void*)rope_fused_kernel<T, V, false, false, MROPE>;
}

template <bool MROPE>
const void* pick_dtype(int dtype, bool vec, bool inter, bool rank4) {
  if (dtype == 0) return vec ? pick<float, 4, MROPE>(inter, rank4) : pick<float, 1, MROPE>(inter, rank4);
  if (dtype == 1) return vec ? pick<__half, 8, MROPE>(inter, rank4) : pick<__half, 1, MROPE>(inter, rank4);
  if (dtype == 2) return vec ? pick<__nv_bfloat16, 8, MROPE>(inter, rank4) : pick<__nv_bfloat16, 1, MROPE>(inter, rank4);
  return nullptr;
}
}  // namespace

const void* fused_kernel(int dtype, bool vec, bool inter, bool rank4, bool mrope) {
  return mrope ? pick_dtype<true>(dtype, vec, inter, rank4) : pick_dtype<false>(dtype, vec, inter, rank4);
}

const void* cache_build_kernel(int dtype) {
  if (dtype == 0) return (const void*)rope_cache_build_kernel<float>;
  if (dtype == 1) return (const void*)rope_cache_build_kernel<__half>;
  if (dtype == 2) return (const void*)rope_cache_build_kernel<__nv_bfloat16>;
  return nullptr;
}

}  // namespace rope_gb300
