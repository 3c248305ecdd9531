// Pipelined M-RoPE Q/K rotation with the key/value cache append (and
// QK-RMSNorm): kernel instances ("com.microsoft.MRotaryEmbedding" README,
// Description, Inputs, Attributes; "com.microsoft.SparseAttention" README,
// Description and Inputs).
#include "rope_qkv_tma.cuh"

namespace rope_gb300 {

namespace {
template <class T, bool NORM>
const void* pick(bool inter) {
  return inter ? (const void*)rope_qkv_tma_kernel<T, true, false, NORM, true>
               : (const void*)rope_qkv_tma_kernel<T, false, false, NORM, true>;
}

template <bool NORM>
const void* pick_dtype(int dtype, bool inter) {
  if (dtype == 0) return pick<float, NORM>(inter);
  if (dtype == 1) return pick<__half, NORM>(inter);
  if (dtype == 2) return pick<__nv_bfloat16, NORM>(inter);
  return nullptr;
}
}  // namespace

const void* mrope_qkv_tma_kernel(int dtype, bool inter, bool rms_norm) {
  return rms_norm ? pick_dtype<true>(dtype, inter) : pick_dtype<false>(dtype, inter);
}

}  // namespace rope_gb300
