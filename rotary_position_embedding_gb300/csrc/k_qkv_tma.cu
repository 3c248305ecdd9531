// Pipelined Q/K rotation with the key/value cache append (and QK-RMSNorm):
// kernel instances ("com.microsoft.SparseAttention" README, Description and
// Inputs; onnxruntime PR "Add RotaryEmbedding fusion for Qwen3 on-the-fly RoPE
// patterns", Qwen3 Architecture).
#include "rope_qkv_tma.cuh"

namespace rope_gb300 {

namespace {
template <class T, bool NORM>
const void* pick(bool inter, bool implicit_pos) {
  if (inter)
    return implicit_pos ? (const void*)rope_qkv_tma_kernel<T, true, true, NORM>
                        : (const void*)rope_qkv_tma_kernel<T, true, false, NORM>;
  return implicit_pos ? (const void*)rope_qkv_tma_kernel<T, false, true, NORM>
                      : (const void*)rope_qkv_tma_kernel<T, false, false, NORM>;
}

template <bool NORM>
const void* pick_dtype(int dtype, bool inter, bool implicit_pos) {
  if (dtype == 0) return pick<float, NORM>(inter, implicit_pos);
  if (dtype == 1) return pick<__half, NORM>(inter, implicit_pos);
  if (dtype == 2) return pick<__nv_bfloat16, NORM>(inter, implicit_pos);
  return nullptr;
}
}  // namespace

const void* qkv_tma_kernel(int dtype, bool inter, bool implicit_pos, bool rms_norm) {
  return rms_norm ? pick_dtype<true>(dtype, inter, implicit_pos) : pick_dtype<false>(dtype, inter, implicit_pos);
}

}  // namespace rope_gb300
