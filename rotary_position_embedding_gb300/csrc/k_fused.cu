// On-the-fly RoPE (cos/sin from inv_freq) and the cos/sin cache build (the
// onnxruntime Qwen3 on-the-fly RoPE fusion pull request: Modeling Code
// Alignment Check, Medium Issues 4).
#include "rope_kernels.cuh"

namespace rope_gb300 {

namespace {
template <class T, int V>
const void* pick(bool inter, bool rank4) {
  if (inter)
    return rank4 ? (const void*)rope_fused_kernel<T, V, true, true>
                 : (const void*)rope_fused_kernel<T, V, true, false>;
  return rank4 ? (const void*)rope_fused_kernel<T, V, false, true>
               : (const void*)rope_fused_kernel<T, V, false, false>;
}
}  // namespace

const void* fused_kernel(int dtype, bool vec, bool inter, bool rank4) {
  if (dtype == 0) return vec ? pick<float, 4>(inter, rank4) : pick<float, 1>(inter, rank4);
  if (dtype == 1) return vec ? pick<__half, 8>(inter, rank4) : pick<__half, 1>(inter, rank4);
  return nullptr;
}

const void* cache_build_kernel(int dtype) {
  if (dtype == 0) return (const void*)rope_cache_build_kernel<float>;
  if (dtype == 1) return (const void*)rope_cache_build_kernel<__half>;
  return nullptr;
}

}  // namespace rope_gb300
