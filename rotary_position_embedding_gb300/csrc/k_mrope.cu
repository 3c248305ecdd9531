// MRotaryEmbedding kernel instances ("com.microsoft.MRotaryEmbedding" README:
// three position streams, section select, scale, out-of-range copy-through).
#include "rope_kernels.cuh"

namespace rope_gb300 {

namespace {
template <class T, int V>
const void* pick(bool inter, bool rank4) {
  if (inter)
    return rank4 ? (const void*)rope_rows_kernel<T, V, true, true, Coef::kMRope>
                 : (const void*)rope_rows_kernel<T, V, true, false, Coef::kMRope>;
  return rank4 ? (const void*)rope_rows_kernel<T, V, false, true, Coef::kMRope>
               : (const void*)rope_rows_kernel<T, V, false, false, Coef::kMRope>;
}

}  // namespace

const void* rope_kernel_mrope(int dtype, bool vec, bool inter, bool rank4) {
  if (dtype == 0) return vec ? pick<float, 4>(inter, rank4) : pick<float, 1>(inter, rank4);
  if (dtype == 1) return vec ? pick<__half, 8>(inter, rank4) : pick<__half, 1>(inter, rank4);
  if (dtype == 2) return vec ? pick<__nv_bfloat16, 8>(inter, rank4) : pick<__nv_bfloat16, 1>(inter, rank4);
  return nullptr;
}

}  // namespace rope_gb300
