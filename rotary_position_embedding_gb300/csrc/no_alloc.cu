// rope_apply_no_alloc: RotaryEmbedding for callers that cannot allocate device
// memory, not even the few bytes of scratch rope_apply's dynamic tile schedule
// takes. Examples: code running inside CUDA stream capture (where device
// allocation is not allowed), plugins and runtimes that hand out only
// pre-sized buffers for inputs and outputs, and callers without a device
// allocator of their own. This entry point takes its scratch from a fixed
// array that lives in the library's own device memory instead.
#include <cuda.h>  // CUcontext; the two driver calls are fetched at run time
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "rope.h"
#include "rope_internal.h"

namespace {

// The schedule's scratch, shared by every call on a device. Fixed size: the
// pipelined kernel's counter pair needs 16 of these bytes whatever the shapes,
// so no input can need more. Device memory of the library image: every GPU
// that loads the library holds it until the process exits. It is zero when
// the module is loaded, and every launch that uses it leaves it zero again.
constexpr size_t kNoAllocScratchBytes = 256;
static_assert(ROPE_SCRATCH_BYTES <= kNoAllocScratchBytes, "static scratch smaller than the schedule needs");
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// The array's device address as seen from one context. A context's unique id
// (cuCtxGetId) is never reused within the process, so a reset device or a
// different context on the same device never matches an old entry.
struct ScratchAddr {
  unsigned long long ctx_id = 0;  // 0: not set up
  void* ptr = nullptr;
};
std::mutex g_mu;
ScratchAddr g_scratch_addr[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Failures are reported through rope_last_error(), like every other entry point.
rope_status fail(rope_status st, const char* what, cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s%s%s", what, e == cudaSuccess ? "" : ": ",
           e == cudaSuccess ? "" : cudaGetErrorString(e));
  rope_gb300::set_last_error(msg);
  return st;
}

// Unique id of the calling thread's current context, or 0 when none is
// current yet (the runtime makes the device's primary context current on its
// first call that needs one).
bool current_context_id(unsigned long long* id) {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return false;
  return true;
}

// Set-up, once per device and context, with that device current: the array's
// device address (in host code the symbol is only a host-side stand-in, not
// an address a kernel may be given). It runs inside the first call on the
// device, which is why that first call must not be made while the stream is
// being captured.
rope_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ROPE_ERR_CUDA, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices)
    return fail(ROPE_ERR_UNSUPPORTED, "device ordinal beyond the 64 devices rope_apply_no_alloc serves",
                cudaSuccess);
  unsigned long long id = 0;
  if (!current_context_id(&id))
    return fail(ROPE_ERR_CUDA, "cannot identify the current CUDA context (cuCtxGetCurrent / cuCtxGetId)",
                cudaSuccess);
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  if (id == 0 || a.ctx_id != id) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_no_alloc_scratch);
    if (e != cudaSuccess || !ptr) return fail(ROPE_ERR_CUDA, "cudaGetSymbolAddress(static scratch)", e);
    if (id == 0 && !current_context_id(&id)) id = 0;  // the lookup made the primary context current
    a.ptr = ptr;
    a.ctx_id = id;
  }
  *out = a.ptr;
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
