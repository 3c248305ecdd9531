// rope_qkv_heads_kernel instances: Q/K rotation with the cache append (and
// QK-RMSNorm), SIMT, several heads per thread ("com.microsoft.SparseAttention"
// README; the onnxruntime Qwen3 on-the-fly RoPE fusion pull request).
#include "rope_qkv_heads.cuh"

namespace rope_gb300 {

namespace {
template <class T, bool NORM, int HPT, bool RAGGED>
const void* pick(bool inter, bool implicit_pos) {
  constexpr int V = 16 / (int)sizeof(typename Elem<T>::bits);
  if (inter)
    return implicit_pos ? (const void*)rope_qkv_heads_kernel<T, V, true, true, NORM, HPT, RAGGED>
                        : (const void*)rope_qkv_heads_kernel<T, V, true, false, NORM, HPT, RAGGED>;
  return implicit_pos ? (const void*)rope_qkv_heads_kernel<T, V, false, true, NORM, HPT, RAGGED>
                      : (const void*)rope_qkv_heads_kernel<T, V, false, false, NORM, HPT, RAGGED>;
}

// RoPE: groups of 2 or 4 heads; RMSNorm: groups of 2 (each also with a short last group)
template <class T>
const void* pick_shape(bool norm, int hpt, bool ragged, bool inter, bool implicit_pos) {
  if (norm) {
    if (hpt != 2) return nullptr;
    return ragged ? pick<T, true, 2, true>(inter, implicit_pos) : pick<T, true, 2, false>(inter, implicit_pos);
  }
  if (hpt == 2) return ragged ? pick<T, false, 2, true>(inter, implicit_pos) : pick<T, false, 2, false>(inter, implicit_pos);
  if (hpt == 4) return ragged ? pick<T, false, 4, true>(inter, implicit_pos) : pick<T, false, 4, false>(inter, implicit_pos);
  return nullptr;
}
}  // namespace

const void* qkv_heads_kernel(int dtype, bool inter, bool implicit_pos, bool rms_norm, int hpt, bool ragged) {
  if (dtype == 0) return pick_shape<float>(rms_norm, hpt, ragged, inter, implicit_pos);
  if (dtype == 1) return pick_shape<__half>(rms_norm, hpt, ragged, inter, implicit_pos);
  if (dtype == 2) return pick_shape<__nv_bfloat16>(rms_norm, hpt, ragged, inter, implicit_pos);
  return nullptr;
}

}  // namespace rope_gb300
