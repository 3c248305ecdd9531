// Q/K rotation with grouped-query heads and the key/value cache append: kernel
// instances ("com.microsoft.SparseAttention" README, Description and Inputs).
#include "rope_qkv.cuh"

namespace rope_gb300 {

namespace {
template <class T, int V>
const void* pick(bool inter, bool implicit_pos) {
  if (inter)
    return implicit_pos ? (const void*)rope_qkv_kernel<T, V, true, true>
                        : (const void*)rope_qkv_kernel<T, V, true, false>;
  return implicit_pos ? (const void*)rope_qkv_kernel<T, V, false, true>
                      : (const void*)rope_qkv_kernel<T, V, false, false>;
}
}  // namespace

const void* qkv_kernel(int dtype, bool vec, bool inter, bool implicit_pos) {
  if (dtype == 0) return vec ? pick<float, 4>(inter, implicit_pos) : pick<float, 1>(inter, implicit_pos);
  if (dtype == 1) return vec ? pick<__half, 8>(inter, implicit_pos) : pick<__half, 1>(inter, implicit_pos);
  return nullptr;
}

}  // namespace rope_gb300
