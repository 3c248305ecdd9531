// RotaryEmbedding kernel instances: 2-D cache gathered at position_ids, and
// the per-token 3-D cache ("ai.onnx.RotaryEmbedding" WebGPU manifest, the four
// variants rank3/rank4 x with/without position_ids).
#include "rope_kernels.cuh"

namespace rope_gb300 {

namespace {
template <class T, int V, Coef M>
const void* pick(bool inter, bool rank4) {
  if (inter)
    return rank4 ? (const void*)rope_rows_kernel<T, V, true, true, M>
                 : (const void*)rope_rows_kernel<T, V, true, false, M>;
  return rank4 ? (const void*)rope_rows_kernel<T, V, false, true, M>
               : (const void*)rope_rows_kernel<T, V, false, false, M>;
}

template <Coef M>
const void* pick_dtype(int dtype, bool vec, bool inter, bool rank4) {
  if (dtype == 0) return vec ? pick<float, 4, M>(inter, rank4) : pick<float, 1, M>(inter, rank4);
  if (dtype == 1) return vec ? pick<__half, 8, M>(inter, rank4) : pick<__half, 1, M>(inter, rank4);
  if (dtype == 2) return vec ? pick<__nv_bfloat16, 8, M>(inter, rank4) : pick<__nv_bfloat16, 1, M>(inter, rank4);
  return nullptr;
}
}  // namespace

const void* rope_kernel_cached(int dtype, bool vec, bool inter, bool rank4, Coef mode) {
  if (mode == Coef::kCache2D) return pick_dtype<Coef::kCache2D>(dtype, vec, inter, rank4);
  if (mode == Coef::kCache3D) return pick_dtype<Coef::kCache3D>(dtype, vec, inter, rank4);
  return nullptr;
}

}  // namespace rope_gb300
