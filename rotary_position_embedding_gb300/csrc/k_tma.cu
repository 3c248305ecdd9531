// TMA-pipelined kernel instances (RotaryEmbedding with a 2-D or 3-D cache,
// MRotaryEmbedding) for the 128-bit vector path.
#include "rope_tma.cuh"

namespace rope_gb300 {

namespace {
template <class T, Coef M>
const void* pick(bool inter, bool rank4) {
  if (inter)
    return rank4 ? (const void*)rope_tma_kernel<T, true, true, M>
                 : (const void*)rope_tma_kernel<T, true, false, M>;
  return rank4 ? (const void*)rope_tma_kernel<T, false, true, M>
               : (const void*)rope_tma_kernel<T, false, false, M>;
}

template <class T>
const void* pick_mode(bool inter, bool rank4, Coef mode) {
  switch (mode) {
    case Coef::kCache2D:
      return pick<T, Coef::kCache2D>(inter, rank4);
    case Coef::kCache3D:
      return pick<T, Coef::kCache3D>(inter, rank4);
    case Coef::kMRope:
      return pick<T, Coef::kMRope>(inter, rank4);
  }
  return nullptr;
}
}  // namespace

const void* tma_kernel(int dtype, bool inter, bool rank4, Coef mode) {
  if (dtype == 0) return pick_mode<float>(inter, rank4, mode);
  if (dtype == 1) return pick_mode<__half>(inter, rank4, mode);
  if (dtype == 2) return pick_mode<__nv_bfloat16>(inter, rank4, mode);
  return nullptr;
}

}  // namespace rope_gb300
