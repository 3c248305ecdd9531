// C ABI of librope_gb300.so: argument validation (the operators' shape and
// attribute contracts), variant selection and launch geometry. Kernels live
// in k_rope.cu, k_mrope.cu and k_fused.cu.
//
// Contracts followed (web pages, by title and section):
//  - "ai.onnx.RotaryEmbedding" WebGPU manifest, "derive": rank3Contract,
//    rank4Contract, rank3PosContract, rank4PosContract; attributeConstraints
//    (interleaved in {0, 1}); typeConstraints (T in {float32, float16}).
//  - "com.microsoft.MRotaryEmbedding" README, Attributes: mrope_section (three
//    non-negative counts summing to rd/2), mrope_layout (0 chunked, 1
//    interleaved), is_packed_batching (only 0), rotary_embedding_dim (even,
//    may leave an odd head size), num_heads.
// The library allocates nothing, keeps no per-call state and never
// synchronises; host-side failures return before any launch.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is fetched from the driver at run time
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <tuple>

#include "rope.h"
#include "rope_internal.h"
#include "rope_qkv_tma.cuh"
#include "rope_tma.cuh"

// Launch-shape defaults (threads a CTA aims for; resident-CTA waves in the
// persistent grid). Overridable at compile time.
#ifndef ROPE_TARGET_THREADS
#define ROPE_TARGET_THREADS 256
#endif
#ifndef ROPE_GRID_WAVES
#define ROPE_GRID_WAVES 1
#endif
// The rank-3 cached RoPE / M-RoPE rows kernel launches five times the resident
// CTAs (one or two tokens per CTA at the float16 prefill shapes), so that CTAs
// that finish early are replaced instead of the last wave draining unevenly:
// measured 22.1 -> 20.7 us on (4, 2048, 32 x 128) float16, 84.5 -> 79.4 us on
// (4, 8192, 32 x 128), 43.1 -> 40.5 us in float32. Rank 4 keeps one wave (its
// strided rows measured 5-6 % slower with more).
#ifndef ROPE_ROWS_WAVES_RANK3
#define ROPE_ROWS_WAVES_RANK3 5
#endif
// M-RoPE on the 128-bit path. The SIMT kernel takes several heads per thread
// (rope_mrope_heads_kernel): 2 below ROPE_MROPE_HEADS4_MIN_TOKENS tokens (more
// threads for decode-sized calls), 4 from there. Measured on GB300, float16,
// 28 heads of 128, from a CUDA graph (2 / 4 heads per thread; the per-thread
// merge of rope_rows_kernel): 256 tokens 2.95 / 3.39 us (3.46); 1024 tokens
// 5.51 / 4.40 us (7.98); 16384 tokens 45.6 / 38.8 us (80.6). The TMA pipeline
// (38.2 us there) stays the automatic choice from 8 MiB of X where its tile
// reaches ROPE_MROPE_TMA_MIN_TILE bytes: the three coefficient rows a token
// gathers cap its tokens per tile, and with few heads the tiles shrink (16
// heads: 20 KB tiles, 25.7 us against 24.0 us for the SIMT kernel; 4 heads:
// 5 KB, 20.9 against 8.3 us; 32 heads: 32 KB, 43.0 against 43.0 us).
#ifndef ROPE_MROPE_HEADS4_MIN_TOKENS
#define ROPE_MROPE_HEADS4_MIN_TOKENS 512
#endif
#ifndef ROPE_MROPE_TMA_MIN_TILE
#define ROPE_MROPE_TMA_MIN_TILE (24 * 1024)
#endif
// TMA pipeline: bytes of one X tile, shared-memory budget of the stage ring,
// smallest X (bytes) sent down the pipeline, most stages.
#ifndef ROPE_TMA_TILE_BYTES
#define ROPE_TMA_TILE_BYTES 32768
#endif
// The budget is half an SM's shared memory less the per-CTA reserve, so two
// CTAs fit per SM; at 112 KB the rank-4 tiles (32 KB of X and 4 KB of rows)
// get a third stage: measured 80.4 -> 80.0 us per launch from a graph and
// 85.5 -> 84.5 us alone on (8, 32, 4096, 128) float16 with rd 64 (110 KB
// gave two); M-RoPE keeps three either way.
#ifndef ROPE_TMA_SMEM_BUDGET
#define ROPE_TMA_SMEM_BUDGET (112 * 1024)
#endif
#ifndef ROPE_TMA_MIN_BYTES
#define ROPE_TMA_MIN_BYTES (8 << 20)
#endif
#ifndef ROPE_TMA_MAX_STAGES
#define ROPE_TMA_MAX_STAGES 8
#endif
// Pipelined Q/K kernel: largest tile (bytes of NG heads x TS tokens) and most
// tokens per tile.
#ifndef ROPE_QKV_TMA_TILE_BYTES
#define ROPE_QKV_TMA_TILE_BYTES 32768
#endif
#ifndef ROPE_QKV_TMA_MAX_TS
#define ROPE_QKV_TMA_MAX_TS 16
#endif
// Its shared-memory budget per CTA (two CTAs per SM): three stages of a
// 32 KB tile with its cos/sin rows.
#ifndef ROPE_QKV_TMA_SMEM_BUDGET
#define ROPE_QKV_TMA_SMEM_BUDGET (112 * 1024)
#endif

using namespace rope_gb300;

#define ROPE_TRY(expr)               \
  do {                               \
    rope_status _s = (expr);         \
    if (_s != ROPE_OK) return _s;    \
  } while (0)

namespace {

thread_local std::string g_last_error;
thread_local const char* g_last_kernel = "";
std::atomic<int> g_variant{ROPE_VARIANT_AUTO};

rope_status fail(rope_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

rope_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ROPE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int elem_size(rope_dtype dt) { return dt == ROPE_F32 ? 4 : 2; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Multiply non-negative sizes; false on int64 overflow.
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a == 0 || b == 0) {
    *out = 0;
    return true;
  }
  if (a > INT64_MAX / b) return false;
  *out = a * b;
  return true;
}

// ---------------------------------------------------------------------------
// Device facts, cached per device (SM count) and per kernel configuration
// (resident CTAs per SM).
// ---------------------------------------------------------------------------
std::mutex g_mu;
std::map<int, int> g_sm_count;
std::map<std::tuple<int, const void*, int, size_t>, int> g_occupancy;
std::set<std::pair<int, const void*>> g_smem_raised;

rope_status device_facts(const void* fn, int threads, size_t smem, int* sms, int* per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_sm_count.find(dev);
  if (it == g_sm_count.end()) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    it = g_sm_count.emplace(dev, n).first;
  }
  *sms = it->second;
  // Kernels that take more than 48 KB of dynamic shared memory get the
  // device's opt-in maximum once (a per-call value could later lower it below
  // what an earlier, cached configuration launches with).
  if (smem > 48 * 1024 && !g_smem_raised.count(std::make_pair(dev, fn))) {
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(shared memory opt-in)");
    if ((size_t)optin < smem) return fail(ROPE_ERR_UNSUPPORTED, "needs %zu bytes of shared memory", smem);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
    g_smem_raised.insert(std::make_pair(dev, fn));
  }
  auto key = std::make_tuple(dev, fn, threads, smem);
  auto oc = g_occupancy.find(key);
  if (oc == g_occupancy.end()) {
    int b = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (b < 1) b = 1;
    oc = g_occupancy.emplace(key, b).first;
  }
  *per_sm = oc->second;
  return ROPE_OK;
}

// ---------------------------------------------------------------------------
// X geometry.
// ---------------------------------------------------------------------------
struct Geom {
  int64_t B = 0, S = 0, N = 0, H = 0, ntok = 0, numel = 0;
  int64_t rd = 0, h = 0;
};

// RotaryEmbedding manifest, inputs/X and attributeDescriptions/num_heads:
// rank 3 is (B, S, num_heads*H) and needs num_heads; rank 4 is (B, N, S, H).
rope_status x_geometry(int32_t rank, const int64_t* xs, int32_t num_heads, Geom* g) {
  if (!xs) return fail(ROPE_ERR_INVALID_ARG, "x_shape is NULL");
  if (rank != 3 && rank != 4) return fail(ROPE_ERR_INVALID_ARG, "X must be rank 3 or 4, got %d", rank);
  for (int i = 0; i < rank; ++i)
    if (xs[i] < 0) return fail(ROPE_ERR_INVALID_ARG, "x_shape[%d] = %lld is negative", i, (long long)xs[i]);
  if (rank == 3) {
    if (num_heads < 1)
      return fail(ROPE_ERR_INVALID_ARG, "num_heads must be >= 1 for rank-3 X (got %d)", num_heads);
    if (xs[2] % num_heads != 0)
      return fail(ROPE_ERR_INVALID_ARG, "hidden size %lld is not a multiple of num_heads %d",
                  (long long)xs[2], num_heads);
    g->B = xs[0];
    g->S = xs[1];
    g->N = num_heads;
    g->H = xs[2] / num_heads;
  } else {
    if (num_heads != 0 && num_heads != xs[1])
      return fail(ROPE_ERR_INVALID_ARG, "num_heads %d does not match rank-4 X dim 1 (%lld)", num_heads,
                  (long long)xs[1]);
    g->B = xs[0];
    g->N = xs[1];
    g->S = xs[2];
    g->H = xs[3];
  }
  int64_t t;
  if (!mul_ok(g->B, g->S, &g->ntok) || !mul_ok(g->ntok, g->N, &t) || !mul_ok(t, g->H, &g->numel))
    return fail(ROPE_ERR_INVALID_ARG, "X has more than 2^63 elements");
  return ROPE_OK;
}

// rotary_embedding_dim: 0 = the whole head; else even, 0 < rd <= H.
rope_status rotary_width(int32_t rde, bool odd_head_ok, Geom* g) {
  if (rde < 0) return fail(ROPE_ERR_INVALID_ARG, "rotary_embedding_dim %d is negative", rde);
  if (rde > g->H)
    return fail(ROPE_ERR_INVALID_ARG, "rotary_embedding_dim %d exceeds the head size %lld", rde,
                (long long)g->H);
  if (!odd_head_ok && g->H % 2)
    return fail(ROPE_ERR_INVALID_ARG, "head size %lld must be even", (long long)g->H);
  g->rd = rde ? rde : g->H;
  if (g->rd % 2)
    return fail(ROPE_ERR_INVALID_ARG, "rotary width %lld must be even (a head size of %lld needs an "
                "even rotary_embedding_dim)", (long long)g->rd, (long long)g->H);
  g->h = g->rd / 2;
  return ROPE_OK;
}

// ---------------------------------------------------------------------------
// Launch geometry: fixed thread roles (see KParams).
// ---------------------------------------------------------------------------
struct Launch {
  dim3 grid, block;
  size_t smem = 0;
};

// unit_groups: a row's units go to a power-of-two group of at most 32 lanes,
// one unit per lane (kernels that reduce over a row with warp shuffles).
rope_status plan(const Geom& g, int es, bool vec, const void* fn, bool smem_table, KParams* kp,
                 Launch* L, bool unit_groups = false, int waves = ROPE_GRID_WAVES) {
  const int V = vec ? 16 / es : 1;
  const int64_t nP = g.h / V;
  const int64_t nT = (g.H - g.rd) / V;
  const int64_t U = nP + nT;
  if (U < 1) return fail(ROPE_ERR_INVALID_ARG, "empty head");
  int64_t Ublk = U < kMaxRowThreads ? U : kMaxRowThreads;
  if (unit_groups) {
    Ublk = 1;
    while (Ublk < U) Ublk *= 2;
    if (Ublk > 32)
      return fail(ROPE_ERR_UNSUPPORTED,
                  "a head of %lld %d-element units does not fit one 32-lane group (RMSNorm needs head_size "
                  "<= 256 float16 / 128 float32 elements on the 16-byte path, or 32 on the scalar path)",
                  (long long)U, V);
  }
  int64_t NG = g.N;
  if (NG * Ublk > kMaxRowThreads) {
    NG = kMaxRowThreads / Ublk;
    if (NG < 1) NG = 1;
  }
  const int64_t per_tok = NG * Ublk;
  int64_t TTs = ROPE_TARGET_THREADS / per_tok;
  if (TTs < 1) TTs = 1;
  if (TTs * per_tok > kMaxRowThreads) TTs = kMaxRowThreads / per_tok;
  if (TTs > g.ntok) TTs = g.ntok;
  const int threads = (int)(TTs * per_tok);
  const size_t smem = smem_table ? (size_t)2 * TTs * g.h * es : 0;
  int sms = 0, per_sm = 0;
  rope_status st = device_facts(fn, threads, smem, &sms, &per_sm);
  if (st != ROPE_OK) return st;
  const int64_t tiles = (g.ntok + TTs - 1) / TTs;
  int64_t gx = (int64_t)sms * per_sm * waves;
  if (gx > tiles) gx = tiles;
  if (gx > 0x7fffffff) gx = 0x7fffffff;
  const int64_t gy = (g.N + NG - 1) / NG;
  if (gy > 65535) return fail(ROPE_ERR_UNSUPPORTED, "too many head groups (%lld)", (long long)gy);

  kp->ntok = g.ntok;
  kp->S = g.S;
  kp->N = g.N;
  kp->H = g.H;
  kp->h = (int32_t)g.h;
  kp->rd = (int32_t)g.rd;
  kp->U = (int32_t)U;
  kp->nP = (int32_t)nP;
  kp->Ublk = (int32_t)Ublk;
  kp->NG = (int32_t)NG;
  kp->TTs = (int32_t)TTs;
  kp->step_tok = gx * TTs;
  kp->step_b = g.S ? kp->step_tok / g.S : 0;
  kp->step_s = g.S ? kp->step_tok % g.S : 0;
  L->grid = dim3((unsigned)gx, (unsigned)gy, 1);
  L->block = dim3((unsigned)threads, 1, 1);
  L->smem = smem;
  return ROPE_OK;
}

// rope_mrope_heads_kernel: HPT heads per thread, one thread per (token slot,
// head group, unit); ROPE_ERR_UNSUPPORTED when a token's threads exceed a CTA.
rope_status plan_heads(const Geom& g, int es, const void* fn, int hpt, KParams* kp, Launch* L, int waves) {
  const int V = 16 / es;
  const int64_t nP = g.h / V;
  const int64_t U = nP + (g.H - g.rd) / V;
  const int64_t G = (g.N + hpt - 1) / hpt;
  const int64_t per_tok = G * U;
  if (per_tok < 1 || per_tok > kMaxRowThreads) return ROPE_ERR_UNSUPPORTED;
  int64_t TTs = ROPE_TARGET_THREADS / per_tok;
  if (TTs < 1) TTs = 1;
  if (TTs * per_tok > kMaxRowThreads) TTs = kMaxRowThreads / per_tok;
  if (TTs > g.ntok) TTs = g.ntok;
  const int threads = (int)(TTs * per_tok);
  int sms = 0, per_sm = 0;
  ROPE_TRY(device_facts(fn, threads, 0, &sms, &per_sm));
  const int64_t tiles = (g.ntok + TTs - 1) / TTs;
  int64_t gx = (int64_t)sms * per_sm * waves;
  if (gx > tiles) gx = tiles;
  if (gx > 0x7fffffff) gx = 0x7fffffff;
  kp->ntok = g.ntok;
  kp->S = g.S;
  kp->N = g.N;
  kp->H = g.H;
  kp->h = (int32_t)g.h;
  kp->rd = (int32_t)g.rd;
  kp->U = (int32_t)U;
  kp->nP = (int32_t)nP;
  kp->Ublk = (int32_t)U;
  kp->NG = (int32_t)G;
  kp->TTs = (int32_t)TTs;
  kp->step_tok = gx * TTs;
  L->grid = dim3((unsigned)gx, 1, 1);
  L->block = dim3((unsigned)threads, 1, 1);
  L->smem = 0;
  return ROPE_OK;
}

// rope_qkv_heads_kernel: hpt heads of one role per thread, one thread per
// (token slot, head group, unit); ROPE_ERR_UNSUPPORTED when a token's threads
// exceed a CTA or (RMSNorm) a row's units are not a power-of-two lane group.
rope_status plan_qkv_heads(const Geom& g, int es, const void* fn, int hpt, int64_t nq, int64_t nkv, bool cache,
                           bool norm, KParams* kp, Launch* L) {
  const int V = 16 / es;
  const int64_t nP = g.h / V;
  const int64_t U = nP + (g.H - g.rd) / V;
  if (U < 1) return ROPE_ERR_UNSUPPORTED;
  if (norm && (U > 32 || (U & (U - 1)))) return ROPE_ERR_UNSUPPORTED;
  const int64_t G = (nq + hpt - 1) / hpt + (cache ? 2 : 1) * ((nkv + hpt - 1) / hpt);
  const int64_t per_tok = G * U;
  if (per_tok > kMaxRowThreads) return ROPE_ERR_UNSUPPORTED;
  int64_t TTs = ROPE_TARGET_THREADS / per_tok;
  if (TTs < 1) TTs = 1;
  if (TTs * per_tok > kMaxRowThreads) TTs = kMaxRowThreads / per_tok;
  if (TTs > g.ntok) TTs = g.ntok;
  const int threads = (int)(TTs * per_tok);
  int sms = 0, per_sm = 0;
  ROPE_TRY(device_facts(fn, threads, 0, &sms, &per_sm));
  const int64_t tiles = (g.ntok + TTs - 1) / TTs;
  int64_t gx = (int64_t)sms * per_sm;
  if (gx > tiles) gx = tiles;
  if (gx > 0x7fffffff) gx = 0x7fffffff;
  kp->ntok = g.ntok;
  kp->S = g.S;
  kp->N = g.N;
  kp->H = g.H;
  kp->h = (int32_t)g.h;
  kp->rd = (int32_t)g.rd;
  kp->U = (int32_t)U;
  kp->nP = (int32_t)nP;
  kp->Ublk = (int32_t)U;
  kp->NG = (int32_t)G;
  kp->TTs = (int32_t)TTs;
  kp->step_tok = gx * TTs;
  kp->step_b = g.S ? kp->step_tok / g.S : 0;
  kp->step_s = g.S ? kp->step_tok % g.S : 0;
  L->grid = dim3((unsigned)gx, 1, 1);
  L->block = dim3((unsigned)threads, 1, 1);
  L->smem = 0;
  return ROPE_OK;
}

// ---------------------------------------------------------------------------
// TMA pipeline planning (see rope_tma.cuh).
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// The automatic choice, from measurements on GB300 (kernel and chained step
// times of both paths over rank 3/4, both pairings, fp16/fp32, full and
// partial rotation, 34 MB to 545 MB): the TMA pipeline wins where the SIMT
// kernels do extra work per element -- partial rotation (its consumers never
// touch the tail; 17-36 % faster) and M-RoPE (the three streams' merge runs
// once per tile column; 1.9x) -- and loses on full rotation (SIMT 2-8 %
// faster at rank 3, 36-127 % at rank 4), where a SIMT thread's 128-bit loads
// already keep enough bytes in flight.
bool tma_eligible(const Geom& g, int es, bool vec, bool mrope) {
  const int variant = g_variant.load(std::memory_order_relaxed);
  if (variant == ROPE_VARIANT_SIMT) return false;
  if (!vec || g.H > 256) return false;
  const int64_t nP = g.h / (16 / es);
  if (nP < 1 || nP > kTmaConsumers) return false;
  if (g.ntok > INT32_MAX || g.N > INT32_MAX || g.S > INT32_MAX || g.B > INT32_MAX) return false;
  if (variant == ROPE_VARIANT_AUTO &&
      (g.numel * es < (int64_t)ROPE_TMA_MIN_BYTES || (!mrope && g.rd == g.H)))
    return false;
  return encode_tiled() != nullptr;
}

struct TmaLaunch {
  TParams tp;
  CUtensorMap mx;  // the type carries the alignment TMA needs
  CUtensorMap my;
  Launch L;
};

rope_status encode_x_map(CUtensorMap* m, rope_dtype dt, const Geom& g, int rank, int es, const void* base,
                         const TParams& tp) {
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  cuuint32_t r;
  if (rank == 3) {
    r = 3;
    dims[0] = g.H, dims[1] = g.N, dims[2] = g.ntok;
    strides[0] = g.H * es, strides[1] = g.N * g.H * es;
    box[0] = (cuuint32_t)g.H, box[1] = tp.NG, box[2] = tp.TS;
  } else {
    r = 4;
    dims[0] = g.H, dims[1] = g.S, dims[2] = g.N, dims[3] = g.B;
    strides[0] = g.H * es, strides[1] = g.S * g.H * es, strides[2] = g.N * g.S * g.H * es;
    box[0] = (cuuint32_t)g.H, box[1] = tp.TS, box[2] = tp.NG, box[3] = 1;
  }
  const CUtensorMapDataType ty = dt == ROPE_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dt == ROPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult e = encode_tiled()(m, ty,
                              r, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (e != CUDA_SUCCESS) return fail(ROPE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)e);
  return ROPE_OK;
}

// Persistent grid of the pipelined kernels: one CTA per resident slot (at
// most one per tile). Measured: shrinking the grid so that every CTA takes
// the same number of round-robin tiles gained nothing on M-RoPE or rank 4
// and cost the Q/K workloads 1-3 us.
int64_t pipeline_grid(int64_t slots, int64_t ntiles) { return slots < ntiles ? slots : ntiles; }

// Fills kp's geometry and the TMA launch; ROPE_ERR_UNSUPPORTED (no message)
// when the shape does not fit the pipeline, in which case the caller falls
// back to the register-path kernel.
rope_status plan_tma(rope_dtype dt, const Geom& g, int es, int rank, int slots, const void* fn, const void* x,
                     void* y, KParams* kp, TmaLaunch* T) {
  const int V = 16 / es;
  TParams& tp = T->tp;
  memset(&tp, 0, sizeof(tp));
  int64_t TS, NG;
  if (rank == 3) {
    NG = g.N < 256 ? g.N : 256;
    TS = ROPE_TMA_TILE_BYTES / (NG * g.H * es);
    if (TS < 1) TS = 1;
    if (TS > 32) TS = 32;
    if (TS > g.ntok) TS = g.ntok;
  } else {
    TS = g.S < 32 ? g.S : 32;
    NG = ROPE_TMA_TILE_BYTES / (TS * g.H * es);
    if (NG < 1) NG = 1;
    if (NG > g.N) NG = g.N;
    if (NG > 256) NG = 256;
  }
  // Consumer columns (token, pair unit) must fit the consumer threads, each
  // thread covers at most kMaxHeads heads of its column, and the gather
  // warp's 32 lanes gather at most kMaxGather 16-byte cos/sin pieces each.
  const int64_t nPu = g.h / V;
  const int64_t pieces_per_tok = (int64_t)slots * 2 * (g.h * es / 16);
  auto fits = [&](int64_t ts, int64_t ng) {
    if (ts * nPu > kTmaConsumers) return false;
    if (ts * pieces_per_tok > 32 * kMaxGather) return false;
    return ng <= kMaxHeads * (kTmaConsumers / (ts * nPu));
  };
  while (!fits(TS, NG) && TS > 1) --TS;
  while (!fits(TS, NG) && NG > 1) --NG;
  if (!fits(TS, NG)) return ROPE_ERR_UNSUPPORTED;
  tp.head_groups = (int32_t)((g.N + NG - 1) / NG);
  if (rank == 3) {
    tp.ntiles = ((g.ntok + TS - 1) / TS) * tp.head_groups;
  } else {
    tp.s_tiles = (int32_t)((g.S + TS - 1) / TS);
    tp.ntiles = g.B * tp.head_groups * (int64_t)tp.s_tiles;
  }
  if (tp.ntiles >= INT32_MAX) return ROPE_ERR_UNSUPPORTED;
  tp.TS = (int32_t)TS;
  tp.NG = (int32_t)NG;
  tp.slots = slots;
  tp.x_bytes = (uint32_t)(TS * NG * g.H * es);
  tp.coef_off = tp.x_bytes;
  tp.flag_off = tp.coef_off + (uint32_t)(TS * slots * 2 * g.h * es);
  tp.pos_off = (tp.flag_off + (uint32_t)TS * 4 + 15) / 16 * 16;
  tp.hdr_off = (tp.pos_off + (uint32_t)TS * slots * 8 + 15) / 16 * 16;
  tp.stage_bytes = (tp.hdr_off + 16 + 1023) / 1024 * 1024;
  tp.bar_bytes = 1024;
  int64_t K = (ROPE_TMA_SMEM_BUDGET - tp.bar_bytes) / tp.stage_bytes;
  if (K > ROPE_TMA_MAX_STAGES) K = ROPE_TMA_MAX_STAGES;
  if (K < 2) return ROPE_ERR_UNSUPPORTED;
  tp.K = (int32_t)K;
  const size_t smem = tp.bar_bytes + (size_t)K * tp.stage_bytes;

  kp->ntok = g.ntok;
  kp->S = g.S;
  kp->N = g.N;
  kp->H = g.H;
  kp->h = (int32_t)g.h;
  kp->rd = (int32_t)g.rd;
  kp->nP = (int32_t)(g.h / V);
  kp->U = kp->nP;
  kp->Ublk = kp->nP;

  int sms = 0, per_sm = 0;
  rope_status st = device_facts(fn, kTmaThreads, smem, &sms, &per_sm);
  if (st != ROPE_OK) return st;
  const int64_t gx = pipeline_grid((int64_t)sms * per_sm, tp.ntiles);
  T->L.grid = dim3((unsigned)gx, 1, 1);
  T->L.block = dim3(kTmaThreads, 1, 1);
  T->L.smem = smem;
  ROPE_TRY(encode_x_map(&T->mx, dt, g, rank, es, x, tp));
  ROPE_TRY(encode_x_map(&T->my, dt, g, rank, es, y, tp));
  return ROPE_OK;
}

// ---------------------------------------------------------------------------
// Pipelined Q/K planning (see rope_qkv_tma.cuh).
// ---------------------------------------------------------------------------
struct QkvTmaLaunch {
  QTParams tp;
  QKVMaps maps;
  Launch L;
};

// Multiply-shift constants for dividing values below 2^31 by d (see Div).
Div div_of(int64_t d) {
  if (d < 1) d = 1;  // empty roles: never divided by
  int l = 0;
  while (((int64_t)1 << l) < d) ++l;
  Div r;
  r.m = (uint32_t)((((uint64_t)1 << (31 + l)) + (uint64_t)d - 1) / (uint64_t)d);
  r.shift = 31 + l;
  return r;
}

// One 4-D tiled tensor map: dims and strides innermost first (strides in
// bytes, dims[1..3]), box (bx0..bx3).
rope_status encode4(CUtensorMap* m, rope_dtype dt, const void* base, const cuuint64_t (&dims)[4],
                    const cuuint64_t (&strides)[3], const cuuint32_t (&box)[4]) {
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = dt == ROPE_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dt == ROPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult e = encode_tiled()(m, ty, 4, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (e != CUDA_SUCCESS) return fail(ROPE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)e);
  return ROPE_OK;
}

// The pipelined Q/K kernel takes the 128-bit path with head sizes up to 256
// elements; with RMSNorm, full rotation whose pair units fill a power-of-two
// lane group. The automatic choice sends it the calls whose packed Q/K/V are
// at least ROPE_TMA_MIN_BYTES (smaller ones are launch-bound either way).
bool qkv_tma_eligible(const Geom& g, int es, bool vec, bool norm, int64_t n_all, int64_t max_len,
                      int64_t qkv_bytes) {
  const int variant = g_variant.load(std::memory_order_relaxed);
  if (variant == ROPE_VARIANT_SIMT) return false;
  if (!vec || g.H > 256) return false;
  const int64_t nP = g.h / (16 / es);
  if (nP < 1 || nP > 32) return false;
  if (norm && (g.rd != g.H || (nP & (nP - 1)))) return false;
  if (g.S > INT32_MAX || g.B > INT32_MAX || n_all > INT32_MAX || max_len > INT32_MAX) return false;
  if (variant == ROPE_VARIANT_AUTO && qkv_bytes < (int64_t)ROPE_TMA_MIN_BYTES) return false;
  return encode_tiled() != nullptr;
}

// Tile shape, stage layout, grid and tensor maps; ROPE_ERR_UNSUPPORTED (no
// message) when the shape does not fit, and the caller takes the SIMT kernel.
rope_status plan_qkv_tma(rope_dtype dt, const Geom& g, int es, const QKVParams& a, const void* query,
                         const void* q_out, const void* fn, bool mrope, QkvTmaLaunch* T) {
  const int V = 16 / es;
  const int64_t nP = g.h / V;
  const int64_t slots = mrope ? 3 : 1;  // cos/sin rows per token: one per position stream
  QTParams& tp = T->tp;
  memset(&tp, 0, sizeof(tp));
  memset(&T->maps, 0, sizeof(T->maps));
  const int64_t heads[3] = {a.Nq, a.Nkv, a.cache ? a.Nkv : 0};
  const int nroles = a.cache ? 3 : 2;
  const int64_t ts_cap = g.S < ROPE_QKV_TMA_MAX_TS ? g.S : ROPE_QKV_TMA_MAX_TS;
  const int64_t coef_row = g.h * es;  // bytes of one cos or sin row
  auto blk_of = [&](int64_t TS) { return (TS * g.H * es + 127) / 128 * 128; };
  // the stage's tail: per-token flags, M-RoPE positions and the header, for up to 32 tokens
  const int64_t tail = 32 * 4 + (mrope ? 32 * slots * 8 : 0) + 64;
  int64_t TSr[3] = {0, 0, 0}, NGr[3] = {0, 0, 0};
  // Stage layout for the roles' shapes: each role's NG blocks and then its
  // cos/sin rows; the flags, positions and header after the largest of those.
  // Returns the stages that fit the budget, or -1 when the tile counts overflow.
  auto layout = [&]() -> int64_t {
    int64_t end_max = 0, ts_max = 0, first = 0;
    for (int r = 0; r < 3; ++r) {
      QRole& R = tp.r[r];
      R.TS = (int32_t)TSr[r];
      R.NG = (int32_t)NGr[r];
      R.G = (int32_t)(heads[r] / NGr[r]);
      R.s_tiles = (int32_t)((g.S + TSr[r] - 1) / TSr[r]);
      if (g.B * (int64_t)R.s_tiles >= INT32_MAX) return -1;
      R.nt_tiles = (int32_t)(g.B * R.s_tiles);
      R.blk_bytes = (uint32_t)blk_of(TSr[r]);
      R.x_bytes = (uint32_t)(NGr[r] * TSr[r] * g.H * es);
      R.coef_off = (uint32_t)NGr[r] * R.blk_bytes;
      R.by_nt = div_of(R.nt_tiles);
      R.by_s = div_of(R.s_tiles);
      R.cols = (int32_t)(TSr[r] * nP);
      if (R.cols > kTmaConsumers) return -1;
      R.tpc = kTmaConsumers / R.cols;
      R.hpt = (R.NG + R.tpc - 1) / R.tpc;
      R.by_cols = div_of(R.cols);
      R.first = first;
      first += (int64_t)R.nt_tiles * R.G;
      if (r < nroles) {
        const int64_t end = R.coef_off + (r < 2 ? TSr[r] * slots * 2 * coef_row : 0);
        if (end > end_max) end_max = end;
        if (TSr[r] > ts_max) ts_max = TSr[r];
      }
    }
    tp.ntiles = a.cache ? first : tp.r[2].first;
    if (!a.cache) tp.r[2].first = tp.ntiles;  // no V tiles
    if (tp.ntiles >= INT32_MAX) return -1;
    tp.flag_off = (uint32_t)((end_max + 15) / 16 * 16);
    tp.pos_off = (tp.flag_off + (uint32_t)ts_max * 4 + 15) / 16 * 16;
    tp.hdr_off = (tp.pos_off + (uint32_t)(mrope ? ts_max * slots * 8 : 0) + 15) / 16 * 16;
    tp.stage_bytes = (tp.hdr_off + 16 + 1023) / 1024 * 1024;
    tp.bar_bytes = 1024;
    tp.by_nP = div_of(nP);
    return (ROPE_QKV_TMA_SMEM_BUDGET - tp.bar_bytes) / tp.stage_bytes;
  };
  int64_t K = 0;
  if (!mrope) {
    // One tile shape for every role: TS tokens, each gather lane holding one
    // token's position and copying at most kMaxGather cos/sin rows; NG a
    // divisor of Nkv (so of Nq) that each column's threads cover with at most
    // kMaxHeads heads apiece, within the tile budget. Fewer tokens while
    // fewer than three stages fit.
    int64_t TS = ts_cap;
    while (TS > 1 && TS * slots * 2 > 32 * kMaxGather) --TS;
    for (;;) {
      if (TS < 1 || TS > 32 || TS * nP > kTmaConsumers) return ROPE_ERR_UNSUPPORTED;
      const int64_t tpc = kTmaConsumers / (TS * nP);
      int64_t NG = 1;
      for (int64_t d = 1; d <= a.Nkv; ++d) {
        if (a.Nkv % d) continue;
        if (d > kMaxHeads * tpc) break;
        if (d > 1 && d * TS * g.H * es > ROPE_QKV_TMA_TILE_BYTES) break;
        NG = d;
      }
      for (int r = 0; r < 3; ++r) TSr[r] = TS, NGr[r] = NG;
      K = layout();
      if (K < 0) return ROPE_ERR_UNSUPPORTED;
      if (K >= 3 || TS <= 4) break;
      TS -= 4;
    }
  } else {
    // Per role: the most heads a tile can take (a token's three coefficient
    // rows are gathered once per tile, so a Q tile of all 32 heads gathers a
    // quarter of what four tiles of 8 do), then the most tokens that keep the
    // tile within the tile budget and its stage within a third of the shared
    // memory, so that three stages are in flight.
    const int64_t stage_cap = (ROPE_QKV_TMA_SMEM_BUDGET - 1024) / 3 / 1024 * 1024 - tail;
    for (int r = 0; r < nroles; ++r) {
      const int64_t coef_tok = r < 2 ? slots * 2 * coef_row : 0;  // V tiles gather nothing
      for (int64_t d = heads[r]; d >= 1 && !TSr[r]; --d) {
        if (heads[r] % d) continue;
        for (int64_t TS = ts_cap; TS >= 1; --TS) {
          if (TS > 32 || TS * nP > kTmaConsumers) continue;
          if (d > kMaxHeads * (kTmaConsumers / (TS * nP))) continue;
          if (d * TS * g.H * es > ROPE_QKV_TMA_TILE_BYTES && !(d == 1 && TS == 1)) continue;
          if (d * blk_of(TS) + TS * coef_tok > stage_cap) continue;
          TSr[r] = TS, NGr[r] = d;
          break;
        }
      }
      if (!TSr[r]) return ROPE_ERR_UNSUPPORTED;
    }
    if (!a.cache) TSr[2] = TSr[1], NGr[2] = NGr[1];
    K = layout();
    if (K < 0) return ROPE_ERR_UNSUPPORTED;
  }
  tp.nT = (int32_t)((g.H - g.rd) / V);
  if (K > ROPE_TMA_MAX_STAGES) K = ROPE_TMA_MAX_STAGES;
  if (K < 2) return ROPE_ERR_UNSUPPORTED;
  tp.K = (int32_t)K;
  const bool packed = a.packed != 0;
  const int64_t n_all = (int64_t)a.Nq + 2 * a.Nkv;
  tp.r[0].head_off = 0;
  tp.r[1].head_off = packed ? a.Nq : 0;
  tp.r[2].head_off = packed ? a.Nq + a.Nkv : 0;
  // pipes pipelines per CTA, each with its own barriers and stages
  const int pipes_per_cta = qkv_pipes(mrope);
  const size_t smem = pipes_per_cta * (tp.bar_bytes + (size_t)K * tp.stage_bytes);
  const int threads = kTmaThreads * pipes_per_cta;

  int sms = 0, per_sm = 0;
  rope_status st = device_facts(fn, threads, smem, &sms, &per_sm);
  if (st != ROPE_OK) return st;
  const int64_t pipes = pipeline_grid((int64_t)sms * per_sm * pipes_per_cta, tp.ntiles);
  T->L.grid = dim3((unsigned)((pipes + pipes_per_cta - 1) / pipes_per_cta), 1, 1);
  T->L.block = dim3(threads, 1, 1);
  T->L.smem = smem;

  // maps: sources (H, heads, S, B) and q_out / k_out (H, heads, S, B) with a
  // TS x NG-head box (Q, K without caches) or a one-head box (K and V into the
  // caches); caches (H, max_len, Nkv, B), TS rows of one head -- TS and NG
  // those of the map's role
  const cuuint64_t H = (cuuint64_t)g.H, S = (cuuint64_t)g.S, B = (cuuint64_t)g.B, E = (cuuint64_t)es;
  auto seq_map = [&](CUtensorMap* m, const void* base, int64_t heads_all, int r, bool wide) {
    const cuuint64_t n = (cuuint64_t)heads_all;
    const cuuint64_t dims[4] = {H, n, S, B};
    const cuuint64_t strides[3] = {H * E, n * H * E, S * n * H * E};
    const cuuint32_t box[4] = {(cuuint32_t)g.H, wide ? (cuuint32_t)tp.r[r].NG : 1u, (cuuint32_t)tp.r[r].TS, 1};
    return encode4(m, dt, base, dims, strides, box);
  };
  auto cache_map = [&](CUtensorMap* m, const void* base, int r) {
    const cuuint64_t L = (cuuint64_t)a.max_len, n = (cuuint64_t)a.Nkv;
    const cuuint64_t dims[4] = {H, L, n, B};
    const cuuint64_t strides[3] = {H * E, L * H * E, n * L * H * E};
    const cuuint32_t box[4] = {(cuuint32_t)g.H, (cuuint32_t)tp.r[r].TS, 1, 1};
    return encode4(m, dt, base, dims, strides, box);
  };
  const bool kv_wide = !a.cache;
  ROPE_TRY(seq_map(&T->maps.src[0], query, packed ? n_all : a.Nq, 0, true));
  ROPE_TRY(seq_map(&T->maps.src[1], packed ? query : a.k, packed ? n_all : a.Nkv, 1, kv_wide));
  if (a.cache) ROPE_TRY(seq_map(&T->maps.src[2], packed ? query : a.v, packed ? n_all : a.Nkv, 2, false));
  ROPE_TRY(seq_map(&T->maps.dst[0], q_out, a.Nq, 0, true));
  if (a.cache) {
    ROPE_TRY(cache_map(&T->maps.dst[1], a.k_cache, 1));
    ROPE_TRY(cache_map(&T->maps.dst[2], a.v_cache, 2));
  } else {
    ROPE_TRY(seq_map(&T->maps.dst[1], a.k_out, a.Nkv, 1, true));
  }
  return ROPE_OK;
}

// Every kernel is launched with programmatic stream serialization: it may be
// scheduled while the previous kernel in the stream finishes, sets up its
// shared memory and barriers, and waits (griddepcontrol.wait) before its
// first read of global memory, so the stream's ordering is unchanged.
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, rope_stream_t stream,
                       void** args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

rope_status launch_tma(const void* fn, TmaLaunch* T, KParams* kp, rope_stream_t stream) {
  void* args[] = {kp, &T->tp, &T->mx, &T->my};
  cudaError_t e = launch_pdl(fn, T->L.grid, T->L.block, T->L.smem, stream, args);
  if (e != cudaSuccess) return cuda_fail(e, "TMA kernel launch");
  g_last_kernel = "rope_tma_kernel";
  return ROPE_OK;
}

rope_status launch(const void* fn, const Launch& L, KParams* kp, rope_stream_t stream,
                   const char* family = "rope_rows_kernel") {
  void* args[] = {kp};
  cudaError_t e = launch_pdl(fn, L.grid, L.block, L.smem, stream, args);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  g_last_kernel = family;
  return ROPE_OK;
}

bool vector_ok(const Geom& g, int es, std::initializer_list<const void*> ptrs) {
  const int V = 16 / es;
  if (g.H % V || g.h % V) return false;
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return false;
  return true;
}

rope_status check_dtype(rope_dtype dt) {
  if (dt != ROPE_F32 && dt != ROPE_F16 && dt != ROPE_BF16)
    return fail(ROPE_ERR_UNSUPPORTED, "dtype %d: only float32 (0), float16 (1) and bfloat16 (2) are implemented",
                (int)dt);
  return ROPE_OK;
}

rope_status check_elem_ptr(const void* p, const char* name, size_t align) {
  if (!p) return fail(ROPE_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, align))
    return fail(ROPE_ERR_INVALID_ARG, "%s is not aligned to %zu bytes", name, align);
  return ROPE_OK;
}

// Interleaved stream map: walk t, h, w cyclically, skipping streams whose
// section count is used up, so every stream gets exactly its section count.
rope_status build_stream_map(const int32_t* sec, int32_t layout, int64_t half, uint8_t* map) {
  if (!sec) return fail(ROPE_ERR_INVALID_ARG, "mrope_section is NULL");
  int64_t total = 0;
  for (int k = 0; k < 3; ++k) {
    if (sec[k] < 0) return fail(ROPE_ERR_INVALID_ARG, "mrope_section[%d] = %d is negative", k, sec[k]);
    total += sec[k];
  }
  if (total != half)
    return fail(ROPE_ERR_INVALID_ARG, "mrope_section sums to %lld, rotary width / 2 is %lld",
                (long long)total, (long long)half);
  if (layout == 0) {
    int64_t i = 0;
    for (int k = 0; k < 3; ++k)
      for (int32_t c = 0; c < sec[k]; ++c) map[i++] = (uint8_t)k;
    return ROPE_OK;
  }
  if (layout == 1) {
    int64_t used[3] = {0, 0, 0};
    int cur = 0;
    for (int64_t i = 0; i < half; ++i) {
      while (used[cur] >= sec[cur]) cur = (cur + 1) % 3;  // total == half: some stream has room
      map[i] = (uint8_t)cur;
      ++used[cur];
      cur = (cur + 1) % 3;
    }
    return ROPE_OK;
  }
  return fail(ROPE_ERR_INVALID_ARG, "mrope_layout must be 0 or 1 (got %d)", layout);
}

// Shared M-RoPE body for mrope_apply and mrope_apply_stream_map.
rope_status mrope_common(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape, const void* x,
                         void* y, int64_t cache_rows, const void* cos_cache, const void* sin_cache,
                         const int64_t* position_ids, const int32_t* sec, int32_t layout,
                         const uint8_t* explicit_map, float scale, int32_t interleaved,
                         int32_t rde, int32_t num_heads, int32_t* oor_flag, void* scratch,
                         rope_stream_t stream) {
  ROPE_TRY(check_dtype(dtype));
  Geom g;
  ROPE_TRY(x_geometry(x_rank, x_shape, num_heads, &g));
  if (interleaved != 0 && interleaved != 1)
    return fail(ROPE_ERR_INVALID_ARG, "interleaved must be 0 or 1 (got %d)", interleaved);
  ROPE_TRY(rotary_width(rde, /*odd_head_ok=*/true, &g));
  if (g.h > kMaxMRopeHalf)
    return fail(ROPE_ERR_UNSUPPORTED, "M-RoPE rotary width / 2 = %lld exceeds %d", (long long)g.h,
                kMaxMRopeHalf);
  if (cache_rows < 0) return fail(ROPE_ERR_INVALID_ARG, "cache_rows is negative");
  uint8_t map[kMaxMRopeHalf];
  if (explicit_map) {
    for (int64_t i = 0; i < g.h; ++i) {
      if (explicit_map[i] > 2)
        return fail(ROPE_ERR_INVALID_ARG, "stream_map[%lld] = %d is not 0, 1 or 2", (long long)i,
                    explicit_map[i]);
      map[i] = explicit_map[i];
    }
  } else if (g.h > 0) {
    ROPE_TRY(build_stream_map(sec, layout, g.h, map));
  }
  if (g.numel == 0) return ROPE_OK;
  const int es = elem_size(dtype);
  ROPE_TRY(check_elem_ptr(x, "x", es));
  ROPE_TRY(check_elem_ptr(y, "y", es));
  ROPE_TRY(check_elem_ptr(position_ids, "position_ids", 8));
  if (cache_rows > 0) {
    ROPE_TRY(check_elem_ptr(cos_cache, "cos_cache", es));
    ROPE_TRY(check_elem_ptr(sin_cache, "sin_cache", es));
  }
  if (oor_flag && !aligned(oor_flag, 4)) return fail(ROPE_ERR_INVALID_ARG, "oor_flag is misaligned");
  if (scratch && !aligned(scratch, 8)) return fail(ROPE_ERR_INVALID_ARG, "scratch is not aligned to 8 bytes");

  const bool vec = vector_ok(g, es, {x, y, cos_cache, sin_cache});
  KParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.sched = static_cast<unsigned long long*>(scratch);
  kp.x = x;
  kp.y = y;
  kp.cos = cos_cache;
  kp.sin = sin_cache;
  kp.pos = position_ids;
  kp.oor_flag = oor_flag;
  kp.scale = scale;
  kp.scale_is_one = scale == 1.0f;
  kp.cache_rows = cache_rows;
  for (int64_t i = 0; i < g.h; ++i) kp.smap[i >> 4] |= (uint32_t)map[i] << ((i & 15) * 2);
  if (tma_eligible(g, es, vec, true)) {
    const void* tfn = tma_kernel(dtype, interleaved != 0, x_rank == 4, Coef::kMRope);
    TmaLaunch T;
    const rope_status ts = plan_tma(dtype, g, es, x_rank, 3, tfn, x, y, &kp, &T);
    const bool forced = g_variant.load(std::memory_order_relaxed) == ROPE_VARIANT_TMA;
    if (ts == ROPE_OK && (forced || T.tp.x_bytes >= (uint32_t)ROPE_MROPE_TMA_MIN_TILE))
      return launch_tma(tfn, &T, &kp, stream);
    if (ts != ROPE_OK && ts != ROPE_ERR_UNSUPPORTED) return ts;
  }
  const int waves = x_rank == 4 ? ROPE_GRID_WAVES : ROPE_ROWS_WAVES_RANK3;
  Launch L;
  if (vec) {
    // each token's three coefficient rows gathered and merged once per 2 or 4 heads
    const int hpt = g.ntok < ROPE_MROPE_HEADS4_MIN_TOKENS ? 2 : 4;
    const void* fn = rope_kernel_mrope_heads(dtype, interleaved != 0, x_rank == 4, hpt);
    const rope_status ps = plan_heads(g, es, fn, hpt, &kp, &L, waves);
    if (ps == ROPE_OK) return launch(fn, L, &kp, stream, "rope_mrope_heads_kernel");
    if (ps != ROPE_ERR_UNSUPPORTED) return ps;
  }
  const void* fn = rope_kernel_mrope(dtype, vec, interleaved != 0, x_rank == 4);
  ROPE_TRY(plan(g, es, vec, fn, false, &kp, &L, false, waves));
  return launch(fn, L, &kp, stream);
}

}  // namespace

void rope_gb300::set_last_error(const char* msg) { g_last_error = msg; }

extern "C" {

rope_status rope_apply(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape, const void* x,
                       void* y, int32_t cache_rank, const int64_t* cache_shape,
                       const void* cos_cache, const void* sin_cache, const int64_t* position_ids,
                       int32_t interleaved, int32_t rotary_embedding_dim, int32_t num_heads,
                       int32_t* oor_flag, void* scratch, rope_stream_t stream) {
  g_last_error.clear();
  ROPE_TRY(check_dtype(dtype));
  Geom g;
  ROPE_TRY(x_geometry(x_rank, x_shape, num_heads, &g));
  if (interleaved != 0 && interleaved != 1)
    return fail(ROPE_ERR_INVALID_ARG, "interleaved must be 0 or 1 (got %d)", interleaved);
  ROPE_TRY(rotary_width(rotary_embedding_dim, /*odd_head_ok=*/false, &g));
  // The variant is fixed by the cache rank (a NULL position_ids pointer may
  // also be an empty tensor): rank 2 gathers at position_ids, rank 3 is the
  // per-token table and takes no position_ids.
  if (!cache_shape) return fail(ROPE_ERR_INVALID_ARG, "cache_shape is NULL");
  const bool gather = cache_rank == 2;
  int64_t rows = 0;
  if (cache_rank == 2) {
    if (cache_shape[0] < 0) return fail(ROPE_ERR_INVALID_ARG, "cache rows are negative");
    if (cache_shape[1] * 2 != g.rd)
      return fail(ROPE_ERR_INVALID_ARG, "cache width %lld * 2 != rotary width %lld",
                  (long long)cache_shape[1], (long long)g.rd);
    rows = cache_shape[0];
  } else if (cache_rank == 3) {
    if (position_ids)
      return fail(ROPE_ERR_INVALID_ARG, "position_ids given with a 3-D (B, S, rd/2) cache");
    if (cache_shape[0] != g.B || cache_shape[1] != g.S || cache_shape[2] * 2 != g.rd)
      return fail(ROPE_ERR_INVALID_ARG,
                  "3-D cache shape (%lld, %lld, %lld) must be (B, S, rd/2) = (%lld, %lld, %lld)",
                  (long long)cache_shape[0], (long long)cache_shape[1], (long long)cache_shape[2],
                  (long long)g.B, (long long)g.S, (long long)g.h);
  } else {
    return fail(ROPE_ERR_INVALID_ARG, "the cos/sin cache must be rank 2 (with position_ids) or 3, got %d",
                cache_rank);
  }
  if (g.numel == 0) return ROPE_OK;
  const int es = elem_size(dtype);
  ROPE_TRY(check_elem_ptr(x, "x", es));
  ROPE_TRY(check_elem_ptr(y, "y", es));
  if (!gather || rows > 0) {
    ROPE_TRY(check_elem_ptr(cos_cache, "cos_cache", es));
    ROPE_TRY(check_elem_ptr(sin_cache, "sin_cache", es));
  }
  if (gather) ROPE_TRY(check_elem_ptr(position_ids, "position_ids", 8));
  if (oor_flag && !aligned(oor_flag, 4)) return fail(ROPE_ERR_INVALID_ARG, "oor_flag is misaligned");
  if (scratch && !aligned(scratch, 8)) return fail(ROPE_ERR_INVALID_ARG, "scratch is not aligned to 8 bytes");

  const bool vec = vector_ok(g, es, {x, y, cos_cache, sin_cache});
  const Coef mode = gather ? Coef::kCache2D : Coef::kCache3D;
  KParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.x = x;
  kp.y = y;
  kp.cos = cos_cache;
  kp.sin = sin_cache;
  kp.pos = position_ids;
  kp.oor_flag = oor_flag;
  kp.scale = 1.0f;
  kp.scale_is_one = 1;
  kp.cache_rows = rows;
  kp.sched = static_cast<unsigned long long*>(scratch);
  if (tma_eligible(g, es, vec, false)) {
    const void* tfn = tma_kernel(dtype, interleaved != 0, x_rank == 4, mode);
    TmaLaunch T;
    const rope_status ts = plan_tma(dtype, g, es, x_rank, 1, tfn, x, y, &kp, &T);
    if (ts == ROPE_OK) return launch_tma(tfn, &T, &kp, stream);
    if (ts != ROPE_ERR_UNSUPPORTED) return ts;
  }
  const void* fn = rope_kernel_cached(dtype, vec, interleaved != 0, x_rank == 4, mode);
  Launch L;
  ROPE_TRY(plan(g, es, vec, fn, false, &kp, &L, false, x_rank == 4 ? ROPE_GRID_WAVES : ROPE_ROWS_WAVES_RANK3));
  return launch(fn, L, &kp, stream);
}

rope_status mrope_apply(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape, const void* x,
                        void* y, int64_t cache_rows, const void* cos_cache,
                        const void* sin_cache, const int64_t* position_ids,
                        const int32_t* mrope_section, int32_t mrope_layout, float scale,
                        int32_t interleaved, int32_t rotary_embedding_dim, int32_t num_heads,
                        int32_t is_packed_batching, int32_t* oor_flag, void* scratch,
                        rope_stream_t stream) {
  g_last_error.clear();
  if (is_packed_batching == 1)
    return fail(ROPE_ERR_UNSUPPORTED, "is_packed_batching = 1 (packed batching) is not implemented");
  if (is_packed_batching != 0)
    return fail(ROPE_ERR_INVALID_ARG, "is_packed_batching must be 0 or 1 (got %d)", is_packed_batching);
  if (!mrope_section) return fail(ROPE_ERR_INVALID_ARG, "mrope_section is NULL");
  return mrope_common(dtype, x_rank, x_shape, x, y, cache_rows, cos_cache, sin_cache, position_ids,
                      mrope_section, mrope_layout, nullptr, scale, interleaved,
                      rotary_embedding_dim, num_heads, oor_flag, scratch, stream);
}

rope_status mrope_apply_stream_map(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape,
                                   const void* x, void* y, int64_t cache_rows,
                                   const void* cos_cache, const void* sin_cache,
                                   const int64_t* position_ids, const uint8_t* stream_map,
                                   float scale, int32_t interleaved,
                                   int32_t rotary_embedding_dim, int32_t num_heads,
                                   int32_t* oor_flag, void* scratch, rope_stream_t stream) {
  g_last_error.clear();
  if (!stream_map) return fail(ROPE_ERR_INVALID_ARG, "stream_map is NULL");
  return mrope_common(dtype, x_rank, x_shape, x, y, cache_rows, cos_cache, sin_cache, position_ids,
                      nullptr, 0, stream_map, scale, interleaved, rotary_embedding_dim, num_heads,
                      oor_flag, scratch, stream);
}

rope_status mrope_stream_map(const int32_t* mrope_section, int32_t mrope_layout, int32_t half,
                             uint8_t* map_out) {
  g_last_error.clear();
  if (half < 0) return fail(ROPE_ERR_INVALID_ARG, "half is negative");
  if (!map_out && half > 0) return fail(ROPE_ERR_INVALID_ARG, "map_out is NULL");
  return build_stream_map(mrope_section, mrope_layout, half, map_out);
}

rope_status rope_apply_fused(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape,
                             const void* x, void* y, const float* inv_freq,
                             float attention_scaling, const int64_t* position_ids,
                             int32_t interleaved, int32_t rotary_embedding_dim,
                             int32_t num_heads, rope_stream_t stream) {
  g_last_error.clear();
  ROPE_TRY(check_dtype(dtype));
  Geom g;
  ROPE_TRY(x_geometry(x_rank, x_shape, num_heads, &g));
  if (interleaved != 0 && interleaved != 1)
    return fail(ROPE_ERR_INVALID_ARG, "interleaved must be 0 or 1 (got %d)", interleaved);
  ROPE_TRY(rotary_width(rotary_embedding_dim, /*odd_head_ok=*/false, &g));
  if (g.numel == 0) return ROPE_OK;
  const int es = elem_size(dtype);
  ROPE_TRY(check_elem_ptr(x, "x", es));
  ROPE_TRY(check_elem_ptr(y, "y", es));
  ROPE_TRY(check_elem_ptr(inv_freq, "inv_freq", 4));
  ROPE_TRY(check_elem_ptr(position_ids, "position_ids", 8));

  const bool vec = vector_ok(g, es, {x, y});
  const void* fn = fused_kernel(dtype, vec, interleaved != 0, x_rank == 4);
  KParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.x = x;
  kp.y = y;
  kp.pos = position_ids;
  kp.inv_freq = inv_freq;
  kp.scale = attention_scaling;
  Launch L;
  ROPE_TRY(plan(g, es, vec, fn, true, &kp, &L));
  return launch(fn, L, &kp, stream, "rope_fused_kernel");
}

}  // extern "C"

namespace {

// Heads per thread of rope_qkv_heads_kernel: RoPE on 16-bit data, on float32
// data, and RMSNorm + RoPE.
#ifndef ROPE_QKV_HPT_ROPE
#define ROPE_QKV_HPT_ROPE 4
#endif
#ifndef ROPE_QKV_HPT_ROPE32
#define ROPE_QKV_HPT_ROPE32 2
#endif
#ifndef ROPE_QKV_HPT_NORM
#define ROPE_QKV_HPT_NORM 2
#endif
// RoPE on 16-bit data takes ROPE_QKV_HPT_ROPE heads per thread from this many
// tokens on, 2 below (more, smaller CTAs for decode-sized batches).
#ifndef ROPE_QKV_HEADS4_MIN_TOKENS
#define ROPE_QKV_HEADS4_MIN_TOKENS 4096
#endif
// rope_qkv_heads_kernel goes ahead of the pipeline for RoPE without QK-Norm
// over the whole head, except in cache mode with the K/V heads at least half
// the Q heads and [Q|K|V] of at least this many bytes: there the pipeline's
// tiled cache writes (many tokens of one head per store) measured faster.
#ifndef ROPE_QKV_PIPE_CACHE_MIN_BYTES
#define ROPE_QKV_PIPE_CACHE_MIN_BYTES (128ll << 20)
#endif

// rope_qkv_heads_kernel launch (128-bit path, RoPE); ROPE_ERR_UNSUPPORTED (no
// message) when the shape does not fit it, and the caller takes another kernel.
rope_status launch_qkv_heads(int dtype, const Geom& g, int es, bool inter, bool implicit_pos, bool norm,
                             int64_t nq, int64_t nkv, bool cache, KParams* kp, const QKVParams* qa,
                             rope_stream_t stream) {
  const int hpt0 = norm                                     ? ROPE_QKV_HPT_NORM
                   : es == 4                                ? ROPE_QKV_HPT_ROPE32
                   : g.ntok >= ROPE_QKV_HEADS4_MIN_TOKENS ? ROPE_QKV_HPT_ROPE
                                                            : 2;
  // the widest group up to `top` that divides both head counts, else `top` with
  // a short last group per role; wider groups when a token's threads exceed a CTA
  for (int top = hpt0; top <= (norm ? 2 : 4); top *= 2) {
    int hpt = 0;
    for (int w = top; w >= 2 && !hpt; w /= 2)
      if (nq % w == 0 && nkv % w == 0) hpt = w;
    const bool ragged = hpt == 0;
    if (ragged) hpt = top;
    const void* fn = qkv_heads_kernel(dtype, inter, implicit_pos, norm, hpt, ragged);
    if (!fn) continue;
    Launch L;
    const rope_status st = plan_qkv_heads(g, es, fn, hpt, nq, nkv, cache, norm, kp, &L);
    if (st == ROPE_ERR_UNSUPPORTED) continue;
    if (st != ROPE_OK) return st;
    QKVParams a = *qa;
    void* args[] = {kp, &a};
    cudaError_t e = launch_pdl(fn, L.grid, L.block, L.smem, stream, args);
    if (e != cudaSuccess) return cuda_fail(e, "rope_apply_qkv launch (heads per thread)");
    g_last_kernel = "rope_qkv_heads_kernel";
    return ROPE_OK;
  }
  return ROPE_ERR_UNSUPPORTED;
}

// rope_apply_qkv and rope_apply_qkv_rmsnorm (q_weight == NULL: no norm).
rope_status qkv_impl(rope_dtype dtype, int64_t batch, int64_t seq, int32_t num_heads, int32_t kv_num_heads,
                     int64_t head_size, const void* query, const void* key, const void* value,
                     const void* q_weight, const void* k_weight, float epsilon, const void* cos_cache,
                     const void* sin_cache, int64_t cache_rows, const int64_t* position_ids,
                     const int32_t* past_seq_lens, int32_t interleaved, int32_t rotary_embedding_dim,
                     void* q_out, void* k_out, void* k_cache, void* v_cache, int64_t max_cache_len,
                     int32_t* status_flags, void* scratch, rope_stream_t stream,
                     const int32_t* mrope_section = nullptr, int32_t mrope_layout = 0, float mrope_scale = 1.0f) {
  g_last_error.clear();
  ROPE_TRY(check_dtype(dtype));
  const bool norm = q_weight != nullptr || k_weight != nullptr;
  const bool mrope = mrope_section != nullptr;
  if (norm && (!q_weight || !k_weight))
    return fail(ROPE_ERR_INVALID_ARG, "RMSNorm needs both q_norm_weight and k_norm_weight");
  if (norm && !(epsilon >= 0.0f && epsilon < INFINITY))
    return fail(ROPE_ERR_INVALID_ARG, "epsilon must be finite and >= 0");
  if (batch < 0 || seq < 0) return fail(ROPE_ERR_INVALID_ARG, "batch and seq must be >= 0");
  if (num_heads < 1 || kv_num_heads < 1)
    return fail(ROPE_ERR_INVALID_ARG, "num_heads (%d) and kv_num_heads (%d) must be >= 1", num_heads,
                kv_num_heads);
  if (num_heads % kv_num_heads)
    return fail(ROPE_ERR_INVALID_ARG, "kv_num_heads %d does not divide num_heads %d", kv_num_heads,
                num_heads);
  if (head_size < 2) return fail(ROPE_ERR_INVALID_ARG, "head_size must be >= 2");
  if (interleaved != 0 && interleaved != 1)
    return fail(ROPE_ERR_INVALID_ARG, "interleaved must be 0 or 1 (got %d)", interleaved);
  if (cache_rows < 0) return fail(ROPE_ERR_INVALID_ARG, "cache_rows is negative");
  uint8_t smap[kMaxMRopeHalf];
  {
    Geom w;
    w.H = head_size;
    ROPE_TRY(rotary_width(rotary_embedding_dim, /*odd_head_ok=*/false, &w));
    if (mrope) {
      if (w.h > kMaxMRopeHalf)
        return fail(ROPE_ERR_UNSUPPORTED, "M-RoPE rotary width / 2 = %lld exceeds %d", (long long)w.h,
                    kMaxMRopeHalf);
      ROPE_TRY(build_stream_map(mrope_section, mrope_layout, w.h, smap));
    }
  }
  // No tokens: nothing to launch (zero-size tensors may come with NULL pointers).
  if (batch == 0 || seq == 0) return ROPE_OK;
  const bool packed = !key && !value;
  const bool cache = k_cache != nullptr;
  if (!packed && !key) return fail(ROPE_ERR_INVALID_ARG, "value given without key");
  if (cache) {
    if (!v_cache || !past_seq_lens)
      return fail(ROPE_ERR_INVALID_ARG, "k_cache needs v_cache and past_seq_lens");
    if (!packed && !value) return fail(ROPE_ERR_INVALID_ARG, "k_cache needs value (or a packed query)");
    if (k_out) return fail(ROPE_ERR_INVALID_ARG, "k_out must be NULL when k_cache is given");
    if (max_cache_len < 1) return fail(ROPE_ERR_INVALID_ARG, "max_cache_len must be >= 1");
  } else {
    if (v_cache) return fail(ROPE_ERR_INVALID_ARG, "v_cache given without k_cache");
    if (!k_out) return fail(ROPE_ERR_INVALID_ARG, "k_out is NULL (and no k_cache)");
    if (value && !packed) return fail(ROPE_ERR_INVALID_ARG, "value is only read in cache mode");
  }
  // The kernel's view: a rank-3 X of Nq + Nkv (+ Nkv) head rows per token.
  Geom g;
  g.B = batch;
  g.S = seq;
  g.N = (int64_t)num_heads + kv_num_heads + (cache ? kv_num_heads : 0);
  g.H = head_size;
  int64_t t, packed_numel;
  if (!mul_ok(g.B, g.S, &g.ntok) || !mul_ok(g.ntok, g.N, &t) || !mul_ok(t, g.H, &g.numel) ||
      !mul_ok(g.ntok, (int64_t)num_heads + 2 * kv_num_heads, &t) || !mul_ok(t, g.H, &packed_numel))
    return fail(ROPE_ERR_INVALID_ARG, "Q/K/V have more than 2^63 elements");
  if (cache) {
    int64_t c;
    if (!mul_ok(g.B, kv_num_heads, &t) || !mul_ok(t, max_cache_len, &c) || !mul_ok(c, g.H, &t))
      return fail(ROPE_ERR_INVALID_ARG, "the caches have more than 2^63 elements");
  }
  ROPE_TRY(rotary_width(rotary_embedding_dim, /*odd_head_ok=*/false, &g));
  if (g.numel == 0) return ROPE_OK;
  const int es = elem_size(dtype);
  ROPE_TRY(check_elem_ptr(query, "query", es));
  ROPE_TRY(check_elem_ptr(q_out, "q_out", es));
  if (packed && q_out == query)
    return fail(ROPE_ERR_INVALID_ARG, "q_out cannot alias a packed query (different row strides)");
  if (!packed) ROPE_TRY(check_elem_ptr(key, "key", es));
  if (value) ROPE_TRY(check_elem_ptr(value, "value", es));
  if (k_out) ROPE_TRY(check_elem_ptr(k_out, "k_out", es));
  if (cache) {
    ROPE_TRY(check_elem_ptr(k_cache, "k_cache", es));
    ROPE_TRY(check_elem_ptr(v_cache, "v_cache", es));
  }
  if (cache_rows > 0) {
    ROPE_TRY(check_elem_ptr(cos_cache, "cos_cache", es));
    ROPE_TRY(check_elem_ptr(sin_cache, "sin_cache", es));
  }
  if (mrope) ROPE_TRY(check_elem_ptr(position_ids, "position_ids (3, B, S)", 8));
  if (position_ids) ROPE_TRY(check_elem_ptr(position_ids, "position_ids", 8));
  if (past_seq_lens) ROPE_TRY(check_elem_ptr(past_seq_lens, "past_seq_lens", 4));
  if (norm) {
    ROPE_TRY(check_elem_ptr(q_weight, "q_norm_weight", es));
    ROPE_TRY(check_elem_ptr(k_weight, "k_norm_weight", es));
  }
  if (status_flags && !aligned(status_flags, 4)) return fail(ROPE_ERR_INVALID_ARG, "status_flags is misaligned");
  if (scratch && !aligned(scratch, 8)) return fail(ROPE_ERR_INVALID_ARG, "scratch is not aligned to 8 bytes");

  const bool vec = vector_ok(g, es, {query, key, value, q_out, k_out, k_cache, v_cache, cos_cache, sin_cache,
                                     q_weight, k_weight});
  const void* fn = mrope ? mrope_qkv_kernel(dtype, vec, interleaved != 0, norm)
                         : qkv_kernel(dtype, vec, interleaved != 0, position_ids == nullptr, norm);
  KParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.x = query;
  kp.y = q_out;
  kp.cos = cos_cache;
  kp.sin = sin_cache;
  kp.pos = position_ids;
  kp.oor_flag = status_flags;
  kp.cache_rows = cache_rows;
  kp.sched = static_cast<unsigned long long*>(scratch);
  if (mrope) {
    kp.scale = mrope_scale;
    kp.scale_is_one = mrope_scale == 1.0f;
    for (int64_t i = 0; i < g.h; ++i) kp.smap[i >> 4] |= (uint32_t)smap[i] << ((i & 15) * 2);
  }
  QKVParams qa;
  memset(&qa, 0, sizeof(qa));
  qa.k = key;
  qa.v = value;
  qa.k_out = k_out;
  qa.k_cache = k_cache;
  qa.v_cache = v_cache;
  qa.past = past_seq_lens;
  qa.max_len = max_cache_len;
  qa.Nq = num_heads;
  qa.Nkv = kv_num_heads;
  qa.packed = packed;
  qa.cache = cache;
  qa.qw = q_weight;
  qa.kw = k_weight;
  qa.eps = epsilon;
  const int64_t n_all = (int64_t)num_heads + 2 * kv_num_heads;
  const bool pipe_first = cache && num_heads <= 2 * (int64_t)kv_num_heads &&
                          packed_numel * es >= (int64_t)ROPE_QKV_PIPE_CACHE_MIN_BYTES;
  if (vec && !mrope && !norm && g.rd == g.H && !pipe_first &&
      g_variant.load(std::memory_order_relaxed) != ROPE_VARIANT_TMA) {
    const rope_status hs = launch_qkv_heads(dtype, g, es, interleaved != 0, position_ids == nullptr, norm,
                                            num_heads, kv_num_heads, cache, &kp, &qa, stream);
    if (hs != ROPE_ERR_UNSUPPORTED) return hs;
  }
  if (qkv_tma_eligible(g, es, vec, norm, n_all, cache ? max_cache_len : 0, packed_numel * es)) {
    const void* tfn = mrope ? mrope_qkv_tma_kernel(dtype, interleaved != 0, norm)
                            : qkv_tma_kernel(dtype, interleaved != 0, position_ids == nullptr, norm);
    QkvTmaLaunch T;
    KParams tk = kp;
    tk.ntok = g.ntok;  // M-RoPE: stream k of token t is position_ids[k * ntok + t]
    tk.S = g.S;
    tk.H = g.H;
    tk.h = (int32_t)g.h;
    tk.rd = (int32_t)g.rd;
    tk.nP = (int32_t)(g.h / (16 / es));
    const rope_status ts = plan_qkv_tma(dtype, g, es, qa, query, q_out, tfn, mrope, &T);
    if (ts == ROPE_OK) {
      void* targs[] = {&tk, &qa, &T.tp, &T.maps};
      cudaError_t e = launch_pdl(tfn, T.L.grid, T.L.block, T.L.smem, stream, targs);
      if (e != cudaSuccess) return cuda_fail(e, "rope_apply_qkv launch (pipelined)");
      g_last_kernel = "rope_qkv_tma_kernel";
      return ROPE_OK;
    }
    if (ts != ROPE_ERR_UNSUPPORTED) return ts;
  }
  Launch L;
  if (vec && !mrope) {  // below the pipeline: the heads-per-thread kernel where it fits
    const rope_status hs = launch_qkv_heads(dtype, g, es, interleaved != 0, position_ids == nullptr, norm,
                                            num_heads, kv_num_heads, cache, &kp, &qa, stream);
    if (hs != ROPE_ERR_UNSUPPORTED) return hs;
  }
  ROPE_TRY(plan(g, es, vec, fn, false, &kp, &L, /*unit_groups=*/norm));
  void* args[] = {&kp, &qa};
  cudaError_t e = launch_pdl(fn, L.grid, L.block, L.smem, stream, args);
  if (e != cudaSuccess) return cuda_fail(e, "rope_apply_qkv launch");
  g_last_kernel = "rope_qkv_kernel";
  return ROPE_OK;
}

}  // namespace

extern "C" {

rope_status rope_apply_qkv(rope_dtype dtype, int64_t batch, int64_t seq, int32_t num_heads,
                           int32_t kv_num_heads, int64_t head_size, const void* query,
                           const void* key, const void* value, const void* cos_cache,
                           const void* sin_cache, int64_t cache_rows, const int64_t* position_ids,
                           const int32_t* past_seq_lens, int32_t interleaved,
                           int32_t rotary_embedding_dim, void* q_out, void* k_out, void* k_cache,
                           void* v_cache, int64_t max_cache_len, int32_t* status_flags, void* scratch,
                           rope_stream_t stream) {
  return qkv_impl(dtype, batch, seq, num_heads, kv_num_heads, head_size, query, key, value, nullptr, nullptr,
                  0.0f, cos_cache, sin_cache, cache_rows, position_ids, past_seq_lens, interleaved,
                  rotary_embedding_dim, q_out, k_out, k_cache, v_cache, max_cache_len, status_flags, scratch,
                  stream);
}

rope_status rope_apply_qkv_rmsnorm(rope_dtype dtype, int64_t batch, int64_t seq, int32_t num_heads,
                                   int32_t kv_num_heads, int64_t head_size, const void* query,
                                   const void* key, const void* value, const void* q_norm_weight,
                                   const void* k_norm_weight, float epsilon, const void* cos_cache,
                                   const void* sin_cache, int64_t cache_rows,
                                   const int64_t* position_ids, const int32_t* past_seq_lens,
                                   int32_t interleaved, int32_t rotary_embedding_dim, void* q_out,
                                   void* k_out, void* k_cache, void* v_cache, int64_t max_cache_len,
                                   int32_t* status_flags, void* scratch, rope_stream_t stream) {
  if (!q_norm_weight || !k_norm_weight) {
    g_last_error.clear();
    return fail(ROPE_ERR_INVALID_ARG, "q_norm_weight and k_norm_weight are required");
  }
  return qkv_impl(dtype, batch, seq, num_heads, kv_num_heads, head_size, query, key, value, q_norm_weight,
                  k_norm_weight, epsilon, cos_cache, sin_cache, cache_rows, position_ids, past_seq_lens,
                  interleaved, rotary_embedding_dim, q_out, k_out, k_cache, v_cache, max_cache_len,
                  status_flags, scratch, stream);
}

rope_status mrope_apply_qkv(rope_dtype dtype, int64_t batch, int64_t seq, int32_t num_heads,
                            int32_t kv_num_heads, int64_t head_size, const void* query, const void* key,
                            const void* value, const void* q_norm_weight, const void* k_norm_weight,
                            float epsilon, const void* cos_cache, const void* sin_cache, int64_t cache_rows,
                            const int64_t* position_ids, const int32_t* mrope_section, int32_t mrope_layout,
                            float scale, const int32_t* past_seq_lens, int32_t interleaved,
                            int32_t rotary_embedding_dim, void* q_out, void* k_out, void* k_cache,
                            void* v_cache, int64_t max_cache_len, int32_t* status_flags, void* scratch,
                            rope_stream_t stream) {
  g_last_error.clear();
  if (!mrope_section) return fail(ROPE_ERR_INVALID_ARG, "mrope_section is NULL");
  if (batch > 0 && seq > 0 && !position_ids)
    return fail(ROPE_ERR_INVALID_ARG, "position_ids (3, B, S) are required");
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(ROPE_ERR_INVALID_ARG, "scale must be finite");
  return qkv_impl(dtype, batch, seq, num_heads, kv_num_heads, head_size, query, key, value, q_norm_weight,
                  k_norm_weight, epsilon, cos_cache, sin_cache, cache_rows, position_ids, past_seq_lens,
                  interleaved, rotary_embedding_dim, q_out, k_out, k_cache, v_cache, max_cache_len, status_flags,
                  scratch, stream, mrope_section, mrope_layout, scale);
}

rope_status rope_cache_build(rope_dtype dtype, const float* inv_freq, int32_t half, int64_t rows,
                             float attention_scaling, void* cos_out, void* sin_out,
                             rope_stream_t stream) {
  g_last_error.clear();
  ROPE_TRY(check_dtype(dtype));
  if (half < 1) return fail(ROPE_ERR_INVALID_ARG, "half must be >= 1 (got %d)", half);
  if (rows < 0) return fail(ROPE_ERR_INVALID_ARG, "rows is negative");
  int64_t total;
  if (!mul_ok(rows, half, &total)) return fail(ROPE_ERR_INVALID_ARG, "rows * half overflows");
  if (total == 0) return ROPE_OK;
  const int es = elem_size(dtype);
  ROPE_TRY(check_elem_ptr(inv_freq, "inv_freq", 4));
  ROPE_TRY(check_elem_ptr(cos_out, "cos_out", es));
  ROPE_TRY(check_elem_ptr(sin_out, "sin_out", es));
  const void* fn = cache_build_kernel(dtype);
  int sms = 0, per_sm = 0;
  ROPE_TRY(device_facts(fn, 256, 0, &sms, &per_sm));
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * per_sm) blocks = (int64_t)sms * per_sm;
  void* args[] = {&inv_freq, &half, &rows, &attention_scaling, &cos_out, &sin_out};
  cudaError_t e = launch_pdl(fn, dim3((unsigned)blocks), dim3(256), 0, stream, args);
  if (e != cudaSuccess) return cuda_fail(e, "rope_cache_build launch");
  g_last_kernel = "rope_cache_build_kernel";
  return ROPE_OK;
}

rope_status rope_set_variant(rope_variant variant) {
  g_last_error.clear();
  if (variant != ROPE_VARIANT_AUTO && variant != ROPE_VARIANT_SIMT && variant != ROPE_VARIANT_TMA)
    return fail(ROPE_ERR_INVALID_ARG, "unknown variant %d", (int)variant);
  g_variant.store(variant, std::memory_order_relaxed);
  return ROPE_OK;
}

rope_variant rope_get_variant(void) { return (rope_variant)g_variant.load(std::memory_order_relaxed); }

const char* rope_last_kernel(void) { return g_last_kernel; }

const char* rope_status_string(rope_status status) {
  switch (status) {
    case ROPE_OK:
      return "ROPE_OK";
    case ROPE_ERR_INVALID_ARG:
      return "ROPE_ERR_INVALID_ARG";
    case ROPE_ERR_UNSUPPORTED:
      return "ROPE_ERR_UNSUPPORTED";
    case ROPE_ERR_CUDA:
      return "ROPE_ERR_CUDA";
  }
  return "ROPE_ERR_UNKNOWN";
}

const char* rope_last_error(void) { return g_last_error.c_str(); }

rope_status mrope_apply_fused(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape, const void* x,
                              void* y, const float* inv_freq, float attention_scaling,
                              const int64_t* position_ids, const int32_t* mrope_section,
                              int32_t mrope_layout, float scale, int32_t interleaved,
                              int32_t rotary_embedding_dim, int32_t num_heads, rope_stream_t stream) {
  g_last_error.clear();
  ROPE_TRY(check_dtype(dtype));
  if (!mrope_section) return fail(ROPE_ERR_INVALID_ARG, "mrope_section is NULL");
  Geom g;
  ROPE_TRY(x_geometry(x_rank, x_shape, num_heads, &g));
  if (interleaved != 0 && interleaved != 1)
    return fail(ROPE_ERR_INVALID_ARG, "interleaved must be 0 or 1 (got %d)", interleaved);
  ROPE_TRY(rotary_width(rotary_embedding_dim, /*odd_head_ok=*/true, &g));
  if (g.h > kMaxMRopeHalf)
    return fail(ROPE_ERR_UNSUPPORTED, "M-RoPE rotary width / 2 = %lld exceeds %d", (long long)g.h,
                kMaxMRopeHalf);
  uint8_t map[kMaxMRopeHalf];
  if (g.h > 0) ROPE_TRY(build_stream_map(mrope_section, mrope_layout, g.h, map));
  if (g.numel == 0) return ROPE_OK;
  const int es = elem_size(dtype);
  ROPE_TRY(check_elem_ptr(x, "x", es));
  ROPE_TRY(check_elem_ptr(y, "y", es));
  ROPE_TRY(check_elem_ptr(inv_freq, "inv_freq", 4));
  ROPE_TRY(check_elem_ptr(position_ids, "position_ids", 8));

  const bool vec = vector_ok(g, es, {x, y});
  const void* fn = fused_kernel(dtype, vec, interleaved != 0, x_rank == 4, /*mrope=*/true);
  KParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.x = x;
  kp.y = y;
  kp.pos = position_ids;
  kp.inv_freq = inv_freq;
  kp.scale = attention_scaling;
  kp.mscale = scale;
  kp.mscale_is_one = scale == 1.0f;
  for (int64_t i = 0; i < g.h; ++i) kp.smap[i >> 4] |= (uint32_t)map[i] << ((i & 15) * 2);
  Launch L;
  ROPE_TRY(plan(g, es, vec, fn, true, &kp, &L));
  return launch(fn, L, &kp, stream, "rope_fused_kernel");
}

}  // extern "C"
