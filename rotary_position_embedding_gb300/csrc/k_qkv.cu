// Q/K rotation with grouped-query heads and the key/value cache append: kernel
// instances ("com.microsoft.SparseAttention" README, Description and Inputs).
#include "rope_qkv.cuh"

namespace rope_gb300 {

namespace {
template <class T, int V, bool NORM>
const void* pick(bool inter, bool implicit_pos) {
  if (inter)
    return implicit_pos ? (const void*)rope_qkv_kernel<T, V, true, true, NORM>
                        : (const void*)rope_qkv_kernel<T, V, true, false, NORM>;
  return implicit_pos ? (const void*)rope_qkv_kernel<T, V, false, true, NORM>
                      : (const void*)rope_qkv_kernel<T, V, false, false, NORM>;
}

template <bool NORM>
const void* pick_dtype(int dtype, bool vec, bool inter, bool implicit_pos) {
  if (dtype == 0)
    return vec ? pick<float, 4, NORM>(inter, implicit_pos) : pick<float, 1, NORM>(inter, implicit_pos);
  if (dtype == 1)
    return vec ? pick<__half, 8, NORM>(inter, implicit_pos) : pick<__half, 1, NORM>(inter, implicit_pos);
  if (dtype == 2)
    return vec ? pick<__nv_bfloat16, 8, NORM>(inter, implicit_pos) : pick<__nv_bfloat16, 1, NORM>(inter, implicit_pos);
  return nullptr;
}
}  // namespace

const void* qkv_kernel(int dtype, bool vec, bool inter, bool implicit_pos, bool rms_norm) {
  return rms_norm ? pick_dtype<true>(dtype, vec, inter, implicit_pos)
                  : pick_dtype<false>(dtype, vec, inter, implicit_pos);
}

}  // namespace rope_gb300
