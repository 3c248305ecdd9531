// Internal interface between the C-ABI layer (rope_api.cu) and the kernel
// translation units. Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rope_gb300 {

enum class Coef : int {
  kCache2D = 0,  // (rows, rd/2) table gathered at position_ids[b, s]
  kCache3D = 1,  // (B, S, rd/2) table, row (b, s)
  kMRope = 2,    // (rows, rd/2) table gathered per pair at one of three streams
};

// Most threads per CTA of the SIMT kernels (their register budget follows).
constexpr int kMaxRowThreads = 512;

// Largest half-rotary width the M-RoPE stream map (2 bits per index) holds.
constexpr int kMaxMRopeHalf = 1024;

// Everything a kernel needs, passed by value (kernel parameter space).
//
// Work decomposition. A head row of H elements is split into U "units":
//   nP pair units, each covering V rotation pairs (V = 16 bytes / sizeof(T) on
//   the vector path, 1 on the scalar path), then (H - rd) / V tail units that
//   copy V elements each. A CTA owns TTs tokens ("token slots") times NG heads
//   times Ublk units; thread t has the fixed role
//     slot = t / (NG*Ublk), head = blockIdx.y*NG + (t / Ublk) % NG, unit = t % Ublk
//   and walks tokens slot + blockIdx.x*TTs, + step_tok, ... (and units
//   unit, unit + Ublk, ... when a row has more than Ublk units).
struct KParams {
  const void* x;
  void* y;
  const void* cos;
  const void* sin;
  const int64_t* pos;
  int32_t* oor_flag;
  const float* inv_freq;
  float scale;           // M-RoPE coefficient scale, or on-the-fly attention scaling
  int32_t scale_is_one;  // M-RoPE: skip the scale-and-round step
  int64_t ntok;          // B*S tokens
  int64_t S, N, H;       // sequence length, heads, head size (elements)
  int64_t cache_rows;    // rows of a 2-D table (range check)
  int32_t h, rd;         // half rotary width, rotary width (elements)
  int32_t U, nP, Ublk;
  int32_t NG, TTs;
  int64_t step_tok;      // gridDim.x * TTs
  int64_t step_b, step_s;  // step_tok = step_b * S + step_s
  uint32_t smap[kMaxMRopeHalf / 16];  // M-RoPE: 2-bit stream of each coefficient index
  unsigned long long* sched;  // TMA path: tile counter pair for the dynamic schedule, or null
  float mscale;          // on-the-fly M-RoPE: the M-RoPE scale (scale holds attention scaling)
  int32_t mscale_is_one;
};

// Q/K rotation with the key/value cache append (rope_qkv_kernel): the routing
// that KParams does not carry. KParams.x is the query (or packed [Q|K|V])
// tensor, KParams.y the rotated Q, KParams.N = Nq + Nkv (+ Nkv in cache mode).
struct QKVParams {
  const void* k;         // key (B, S, Nkv*H), or null when x is packed
  const void* v;         // value (B, S, Nkv*H), or null
  void* k_out;           // no-cache mode: rotated K (B, S, Nkv*H)
  void* k_cache;         // cache mode: (B, Nkv, max_len, H); token s of batch b -> row past[b] + s
  void* v_cache;
  const int32_t* past;   // (B) rows already cached (implicit positions, cache rows), or null
  int64_t max_len;
  int32_t Nq, Nkv;
  int32_t packed;        // x is packed [Q|K|V]
  int32_t cache;         // cache mode
  const void* qw;        // RMSNorm: head-size weights of Q and K heads (null: no norm)
  const void* kw;
  float eps;
};

// Kernel entry points for cudaLaunchKernel / occupancy queries. `vec` selects
// the 128-bit vector path. Return nullptr for unsupported combinations.
const void* rope_kernel_cached(int dtype, bool vec, bool interleaved, bool rank4, Coef mode);
const void* rope_kernel_mrope(int dtype, bool vec, bool interleaved, bool rank4);
// Cached M-RoPE with hpt (2 or 4) heads per thread (128-bit path only); its
// launch takes (KParams) with NG = head groups, Ublk = U, no shared memory.
const void* rope_kernel_mrope_heads(int dtype, bool interleaved, bool rank4, int hpt);
const void* fused_kernel(int dtype, bool vec, bool interleaved, bool rank4, bool mrope = false);
const void* cache_build_kernel(int dtype);
// rope_qkv_kernel instance; its launch takes (KParams, QKVParams).
const void* qkv_kernel(int dtype, bool vec, bool interleaved, bool implicit_pos, bool rms_norm);
// The M-RoPE instance of rope_qkv_kernel (positions (3, B, S), KParams.smap /
// scale as for mrope_apply); same launch.
const void* mrope_qkv_kernel(int dtype, bool vec, bool interleaved, bool rms_norm);
// rope_qkv_heads_kernel (128-bit path, RoPE): hpt heads of one role per thread
// (RoPE: 2 or 4, RMSNorm: 2); ragged: a role's head count need not be a
// multiple of hpt. Same launch, KParams.NG = head groups, Ublk = U; nullptr
// for a shape not instantiated.
const void* qkv_heads_kernel(int dtype, bool interleaved, bool implicit_pos, bool rms_norm, int hpt, bool ragged);
// Records the message rope_last_error() returns on the calling thread.
void set_last_error(const char* msg);

// TMA-pipelined variant (vector path, head size <= 256 elements); its launch
// takes (KParams, TParams, CUtensorMap x, CUtensorMap y).
const void* tma_kernel(int dtype, bool interleaved, bool rank4, Coef mode);

// TMA-pipelined Q/K rotation with the cache append (vector path); its launch
// takes (KParams, QKVParams, QTParams, QKVMaps).
const void* qkv_tma_kernel(int dtype, bool interleaved, bool implicit_pos, bool rms_norm);
// Its M-RoPE instances (positions (3, B, S)).
const void* mrope_qkv_tma_kernel(int dtype, bool interleaved, bool rms_norm);

}  // namespace rope_gb300
