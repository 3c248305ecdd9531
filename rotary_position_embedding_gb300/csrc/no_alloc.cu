// rope_apply_no_alloc: RotaryEmbedding for callers that cannot allocate device
// memory, not even the few bytes of scratch rope_apply's dynamic tile schedule
// takes. Examples: code running inside CUDA stream capture (where device
// allocation is not allowed), plugins and runtimes that hand out only
// pre-sized buffers for inputs and outputs, and callers without a device
// allocator of their own. This entry point takes its scratch from a fixed
// array that lives in the library's own device memory instead.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "rope.h"
#include "rope_internal.h"

namespace {

// The schedule's scratch, shared by every call on a device. Fixed size: the
// pipelined kernel's counter pair needs 16 of these bytes whatever the shapes,
// so no input can need more. Device memory of the library image: every GPU
// that loads the library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = 256;
static_assert(ROPE_SCRATCH_BYTES <= kNoAllocScratchBytes, "static scratch smaller than the schedule needs");
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_no_alloc_scratch, per device

// Failures are reported through rope_last_error(), like every other entry point.
rope_status fail(rope_status st, const char* what, cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, e == cudaSuccess ? "" : cudaGetErrorString(e));
  rope_gb300::set_last_error(msg);
  return st;
}

// Set-up, once per device, with that device current: the array's device
// address (in host code the symbol is only a host-side stand-in) and a cleared
// array. It runs inside the first call on the device, which is why that first
// call must not be made while the stream is being captured.
rope_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ROPE_ERR_CUDA, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices)
    return fail(ROPE_ERR_UNSUPPORTED, "device ordinal beyond the 64 devices rope_apply_no_alloc serves",
                cudaSuccess);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_no_alloc_scratch);
    if (e != cudaSuccess || !ptr) return fail(ROPE_ERR_CUDA, "cudaGetSymbolAddress(static scratch)", e);
    e = cudaMemset(ptr, 0, kNoAllocScratchBytes);  // the schedule's counters start at zero
    if (e != cudaSuccess) return fail(ROPE_ERR_CUDA, "clearing the static scratch", e);
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return ROPE_OK;
}

}  // namespace

extern "C" {

rope_status rope_apply_no_alloc(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape,
                                const void* x, void* y, int32_t cache_rank,
                                const int64_t* cache_shape, const void* cos_cache,
                                const void* sin_cache, const int64_t* position_ids,
                                int32_t interleaved, int32_t rotary_embedding_dim,
                                int32_t num_heads, int32_t* oor_flag, rope_stream_t stream) {
  void* scratch = nullptr;
  const rope_status st = scratch_for_current_device(&scratch);
  if (st != ROPE_OK) return st;
  // Each launch leaves the counters at zero again when it completes, so the
  // next call (in this stream or after it) starts from a cleared array.
  return rope_apply(dtype, x_rank, x_shape, x, y, cache_rank, cache_shape, cos_cache, sin_cache,
                    position_ids, interleaved, rotary_embedding_dim, num_heads, oor_flag, scratch,
                    stream);
}

}  // extern "C"
