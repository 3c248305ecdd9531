// M-RoPE Q/K rotation with grouped-query heads and the key/value cache append
// (SIMT instances): "com.microsoft.MRotaryEmbedding" README (Description,
// Inputs, Attributes) and "com.microsoft.SparseAttention" README (Description,
// Inputs).
#include "rope_qkv.cuh"

namespace rope_gb300 {

namespace {
template <class T, int V, bool NORM>
const void* pick(bool inter) {
  return inter ? (const void*)rope_qkv_kernel<T, V, true, false, NORM, true>
               : (const void*)rope_qkv_kernel<T, V, false, false, NORM, true>;
}

template <bool NORM>
const void* pick_dtype(int dtype, bool vec, bool inter) {
  if (dtype == 0) return vec ? pick<float, 4, NORM>(inter) : pick<float, 1, NORM>(inter);
  if (dtype == 1) return vec ? pick<__half, 8, NORM>(inter) : pick<__half, 1, NORM>(inter);
  if (dtype == 2) return vec ? pick<__nv_bfloat16, 8, NORM>(inter) : pick<__nv_bfloat16, 1, NORM>(inter);
  return nullptr;
}
}  // namespace

const void* mrope_qkv_kernel(int dtype, bool vec, bool inter, bool rms_norm) {
  return rms_norm ? pick_dtype<true>(dtype, vec, inter) : pick_dtype<false>(dtype, vec, inter);
}

}  // namespace rope_gb300
