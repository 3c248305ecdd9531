/*
 * rope.h -- C ABI of the GB300 (sm_103a) rotary position embedding library
 * (librope_gb300.so).
 *
 * Operations (web pages cited by title and section):
 *   rope_apply        ONNX opset-23 RotaryEmbedding: "ai.onnx.RotaryEmbedding"
 *                     WebGPU manifest (manifest.json) -- "inputs", "attributes",
 *                     "attributeDescriptions", "derive" shape contracts.
 *   mrope_apply       com.microsoft.MRotaryEmbedding: its README -- Description,
 *                     Inputs, Attributes, Implementation variants.
 *   rope_apply_fused  the on-the-fly cos/sin form of Qwen3 RoPE: onnxruntime
 *                     pull request "Add RotaryEmbedding fusion for Qwen3
 *                     on-the-fly RoPE patterns" -- Motivation and Context,
 *                     Modeling Code Alignment Check.
 *   rope_cache_build  the cos/sin cache that pull request precomputes from
 *                     inv_freq -- Critical Issues 1, Medium Issues 4.
 *   mrope_apply_stream_map, mrope_apply_fused
 *                     MRotaryEmbedding with an explicit stream per index, and
 *                     with on-the-fly coefficients.
 *   rope_apply_qkv, rope_apply_qkv_rmsnorm, mrope_apply_qkv
 *                     Q and K rotation for grouped-query attention with the
 *                     key/value cache append ("com.microsoft.SparseAttention"
 *                     README), with QK-RMSNorm first (the pull request's
 *                     Qwen3 Architecture), and with M-RoPE.
 *   rope_apply_no_alloc  rope_apply for callers that cannot allocate.
 *
 * Conventions shared by every entry point
 *   - All tensors are dense, contiguous, row-major. Tensor pointers are DEVICE
 *     pointers owned by the caller; the library never allocates, frees or
 *     synchronises, keeps no state between calls and is safe to call from
 *     several host threads. Shape and attribute arrays are HOST pointers read
 *     during the call only.
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream) on the current CUDA device; all device pointers must belong to
 *     that device.
 *   - Element type T is float32 (ROPE_F32), float16 (ROPE_F16) or bfloat16
 *     (ROPE_BF16, beyond the pages); positions are int64. Every pointer must be aligned to its element size. 16-byte
 *     aligned tensors whose head and half-rotary widths are multiples of 16
 *     bytes take the 128-bit vector path; anything else takes the scalar path.
 *     Alignment is never an error.
 *   - y may equal x (in place). Any other overlap between outputs and inputs
 *     is undefined.
 *   - Arithmetic: each pair (x0, x1) with coefficients (c, s) becomes
 *     y0 = x0*c - x1*s, y1 = x1*c + x0*s, computed in float32 and rounded to
 *     nearest-even to T. Elements past the rotary width, and pairs whose
 *     position is out of range, are copied bit-exactly.
 *   - Errors: on ROPE_ERR_INVALID_ARG / ROPE_ERR_UNSUPPORTED nothing is
 *     launched and no output is written. ROPE_ERR_CUDA means a CUDA call
 *     failed while launching. rope_last_error() returns a message for the
 *     last failure on the calling thread.
 *   - An empty X (any dimension 0) is valid and launches nothing.
 *   - Status word (the optional oor_flag / status_flags): a device int32 the
 *     kernels OR bits into and never clear. Bit 0: some position was outside
 *     the table (those elements were copied through). Bit 1: a pipelined
 *     kernel gave up on one of its waits (each is bounded by 2 s of device
 *     time) and returned early, so the output is incomplete; not expected in
 *     normal operation. Bit 2 (Q/K entry points): some cache row was outside
 *     the cache and was not stored.
 */
#ifndef ROPE_GB300_H
#define ROPE_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rope_status {
  ROPE_OK = 0,
  ROPE_ERR_INVALID_ARG = 1, /* shape / attribute contract violated */
  ROPE_ERR_UNSUPPORTED = 2, /* valid ONNX, not implemented (other dtypes, packed batching) */
  ROPE_ERR_CUDA = 3         /* a CUDA runtime call failed */
} rope_status;

/* ROPE_BF16: bfloat16 storage. The pages list float32 and float16 only (and
   mark bfloat16 unimplemented); it is offered here with the same float32
   arithmetic and one final rounding to nearest-even bfloat16. */
typedef enum rope_dtype { ROPE_F32 = 0, ROPE_F16 = 1, ROPE_BF16 = 2 } rope_dtype;

/*
 * Scratch for the dynamic tile schedule (optional `scratch` argument of
 * rope_apply, mrope_apply, mrope_apply_stream_map, rope_apply_qkv and
 * rope_apply_qkv_rmsnorm): ROPE_SCRATCH_BYTES of
 * caller-owned device memory, 8-byte aligned, set to zero once before its first
 * use. With it, the pipelined kernel hands tiles to whichever CTA asks next, so
 * CTAs that run faster take more tiles and the launch ends sooner; every launch
 * leaves the scratch zeroed again when it completes. Launches that may run on
 * the GPU at the same time (other streams, other threads) must use different
 * scratch buffers; launches in one stream can share one. NULL keeps the static
 * schedule (tiles dealt round robin). The result is the same either way.
 */
#define ROPE_SCRATCH_BYTES 64

/* A cudaStream_t (the two types are the same pointer type). */
typedef struct CUstream_st* rope_stream_t;

/*
 * rope_apply -- RotaryEmbedding.
 *
 * x, y          X and Y, same shape: rank 3 (B, S, num_heads*H) or rank 4
 *               (B, N, S, H). H must be even. ([RotaryEmbedding manifest,
 *               inputs/X and outputs/Y])
 * x_shape       x_rank (3 or 4) host int64 values.
 * cos_cache,    cache_rank 2: (max_sequence_length, rd/2), gathered at
 * sin_cache     position_ids; row p is the coefficient row of position p.
 *               cache_rank 3: (B, S, rd/2), row (b, s) belongs to token (b, s),
 *               and no position_ids are taken. cache_shape holds cache_rank
 *               host int64 values; both tables have this shape. ([manifest,
 *               inputs/cos_cache, sin_cache])
 * position_ids  device int64 (B, S), required with a rank-2 cache (it may be
 *               NULL only when X is empty); must be NULL with a rank-3 cache.
 *               ([manifest, inputs/position_ids])
 *               A position outside [0, max_sequence_length) never reads the
 *               cache: every element of that token is copied through and, if
 *               oor_flag is not NULL, bit 0 of the device int32 *oor_flag is
 *               set (the status word above; never cleared by the library).
 * interleaved   0: pair i is (i, i + rd/2); 1: pair i is (2i, 2i+1).
 * rotary_embedding_dim  0 = H; otherwise an even rd with 0 < rd <= H. Elements
 *               [rd, H) of every head are copied through.
 * num_heads     required (>= 1, dividing the last dimension) for rank 3; for
 *               rank 4 it must be 0 or equal to N.
 * scratch       NULL or ROPE_SCRATCH_BYTES of device scratch (see above).
 * The shape contract is the manifest's "derive" rank3Contract, rank4Contract,
 * rank3PosContract, rank4PosContract: cache width * 2 == rd, 3-D cache
 * leading dims == (B, S), position_ids present iff the cache is 2-D.
 */
rope_status rope_apply(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape, const void* x,
                       void* y, int32_t cache_rank, const int64_t* cache_shape,
                       const void* cos_cache, const void* sin_cache, const int64_t* position_ids,
                       int32_t interleaved, int32_t rotary_embedding_dim, int32_t num_heads,
                       int32_t* oor_flag, void* scratch, rope_stream_t stream);

/*
 * mrope_apply -- MRotaryEmbedding (multimodal RoPE).
 *
 * x, y, x_shape, interleaved, rotary_embedding_dim, num_heads: as rope_apply,
 *               except that H may be odd when rd is a smaller even number
 *               ([MRotaryEmbedding README, Description, Attributes/
 *               rotary_embedding_dim]). rd/2 must not exceed 1024.
 * cos_cache, sin_cache  device (cache_rows, rd/2), shared by the three
 *               streams ([README, Inputs/cos]).
 * position_ids  device int64 (3, B, S): temporal, height and width streams
 *               ([README, Inputs/positionIds]). A pair whose stream position
 *               is negative or >= cache_rows is copied through unchanged and
 *               bit 0 of *oor_flag (if not NULL) is set.
 * mrope_section host int32[3], non-negative, summing to rd/2: how many
 *               half-rotary indices each stream drives ([README, Attributes/
 *               mrope_section]).
 * mrope_layout  0: chunked -- indices [0, t) use t, the next h use h, the rest
 *               w. 1: interleaved -- the streams are dealt round by round in
 *               the order t, h, w, each for as many rounds as its section
 *               count. ([README, Attributes/mrope_layout]; the page names the
 *               interleaved layout without printing its order, this is the
 *               reading that keeps each stream's count equal to its section.)
 * scale         multiplies the gathered cos and sin; each scaled coefficient
 *               is rounded to T before the rotation ([README, Attributes/
 *               scale; Implementation variants/pairs4]). The product is
 *               rounded once from its exact value.
 * is_packed_batching  must be 0; 1 returns ROPE_ERR_UNSUPPORTED ([README,
 *               Attributes/is_packed_batching]).
 * scratch       NULL or ROPE_SCRATCH_BYTES of device scratch (see above).
 */
rope_status mrope_apply(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape, const void* x,
                        void* y, int64_t cache_rows, const void* cos_cache,
                        const void* sin_cache, const int64_t* position_ids,
                        const int32_t* mrope_section, int32_t mrope_layout, float scale,
                        int32_t interleaved, int32_t rotary_embedding_dim, int32_t num_heads,
                        int32_t is_packed_batching, int32_t* oor_flag, void* scratch,
                        rope_stream_t stream);

/*
 * mrope_apply_stream_map -- MRotaryEmbedding with an explicit stream per
 * half-rotary index instead of (mrope_section, mrope_layout).
 *
 * stream_map    host uint8[rd/2], each 0 (t), 1 (h) or 2 (w). Lets a caller
 *               use another interleaving convention than mrope_apply's layout 1
 *               (for example fixed stride-3 slots). Everything else as
 *               mrope_apply.
 */
rope_status mrope_apply_stream_map(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape,
                                   const void* x, void* y, int64_t cache_rows,
                                   const void* cos_cache, const void* sin_cache,
                                   const int64_t* position_ids, const uint8_t* stream_map,
                                   float scale, int32_t interleaved,
                                   int32_t rotary_embedding_dim, int32_t num_heads,
                                   int32_t* oor_flag, void* scratch, rope_stream_t stream);

/*
 * mrope_stream_map -- host-only helper: the stream of each of the `half`
 * half-rotary indices for (mrope_section, mrope_layout), as mrope_apply uses
 * it. map_out is a host uint8[half]. ROPE_ERR_INVALID_ARG if the sections are
 * negative or do not sum to half, or the layout is not 0 or 1. No CUDA call.
 */
rope_status mrope_stream_map(const int32_t* mrope_section, int32_t mrope_layout, int32_t half,
                             uint8_t* map_out);

/*
 * rope_apply_fused -- RotaryEmbedding with cos/sin computed on the fly.
 *
 * For token (b, s) at position p = position_ids[b, s] and index i < rd/2
 * ([Qwen3 fusion pull request, Motivation and Context; Modeling Code
 * Alignment Check]):
 *   theta = float32(float32(p) * inv_freq[i]),
 *   c = T(float32(float32(cos(theta)) * attention_scaling)), s likewise,
 * where cos/sin of the float32 angle are evaluated in double precision and
 * rounded to float32; then the rotation of rope_apply. Any int64 position is
 * valid (there is no cache to overrun).
 *
 * inv_freq      device float32[rd/2].
 * position_ids  device int64 (B, S), required.
 * Other arguments as rope_apply. The result equals rope_apply with tables from
 * rope_cache_build(inv_freq, attention_scaling) gathered at the same positions.
 */
rope_status rope_apply_fused(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape,
                             const void* x, void* y, const float* inv_freq,
                             float attention_scaling, const int64_t* position_ids,
                             int32_t interleaved, int32_t rotary_embedding_dim,
                             int32_t num_heads, rope_stream_t stream);

/*
 * rope_apply_qkv -- Q and K rotation for grouped-query attention in one
 * launch, optionally appending the rotated K and the V of the new tokens to a
 * key/value cache ([SparseAttention README, Description: grouped-query heads,
 * separate or packed [Q|K|V] input, rotary embedding in NeoX or interleaved
 * layout, past key/value updated in place; Inputs: query, key, value,
 * past_key, past_value; Attributes: do_rotary rotates Q and K before K enters
 * the cache, kv_num_heads divides num_heads] and [Qwen3 fusion pull request,
 * Verification and Qwen3 Architecture: RoPE on both the Q and the K path,
 * fewer K/V heads than Q heads]).
 *
 * Every Q and K head is rotated exactly as rope_apply rotates one head of a
 * rank-3 X: tables (cache_rows, rd/2) gathered at the token's position,
 * pairing `interleaved`, rotary width `rotary_embedding_dim` (0 = head_size)
 * with the tail copied, and a position outside [0, cache_rows) copies the
 * token's Q and K heads through (status bit 0). V heads are copied bit for
 * bit.
 *
 * query     device T (B, S, num_heads*H), or packed (B, S, (num_heads +
 *           2*kv_num_heads)*H) = [Q|K|V] per token when key and value are
 *           both NULL.
 * key       device T (B, S, kv_num_heads*H), or NULL (packed).
 * value     device T (B, S, kv_num_heads*H): required in cache mode unless
 *           packed; must be NULL without a cache (V is not touched then).
 * position_ids  device int64 (B, S), or NULL: token s of batch b then takes
 *           position past_seq_lens[b] + s (s when past_seq_lens is NULL).
 * past_seq_lens device int32 (B): rows each batch's cache already holds;
 *           required in cache mode, optional otherwise (positions only).
 * q_out     device T (B, S, num_heads*H); may equal query unless packed.
 * Without a cache (k_cache NULL): k_out is device T (B, S, kv_num_heads*H)
 *           (may equal key) and v_cache must be NULL.
 * Cache mode (k_cache non-NULL): k_out must be NULL; k_cache and v_cache are
 *           device T (B, kv_num_heads, max_cache_len, H), updated in place:
 *           token s of batch b goes to row past_seq_lens[b] + s of both
 *           (rotated K, V as given); no other row is written. A token whose
 *           row falls outside [0, max_cache_len) is not stored (status bit 2).
 * status_flags  NULL or a device int32 the kernel ORs bits into (never
 *           clears): bit 0 a position out of range, bit 1 a pipelined wait
 *           that gave up, bit 2 a cache row out of range.
 * scratch   NULL or ROPE_SCRATCH_BYTES of device scratch for the dynamic tile
 *           schedule of the pipelined kernel, with the rules of rope_apply's
 *           scratch (zero before first use, one per concurrently running
 *           stream); the result is the same either way.
 * All buffers are caller-owned; nothing is allocated. Buffers other than the
 * aliases named above must not overlap. ROPE_ERR_INVALID_ARG (before any
 * launch) for: num_heads or kv_num_heads < 1, kv_num_heads not dividing
 * num_heads, an odd or < 2 head_size, a bad rotary width, interleaved not 0/1,
 * an inconsistent set of key/value/k_out/k_cache/v_cache/past_seq_lens,
 * max_cache_len < 1 in cache mode, negative cache_rows, NULL or misaligned
 * pointers, or element counts beyond 2^63. B*S == 0 launches nothing.
 */
rope_status rope_apply_qkv(rope_dtype dtype, int64_t batch, int64_t seq, int32_t num_heads,
                           int32_t kv_num_heads, int64_t head_size, const void* query,
                           const void* key, const void* value, const void* cos_cache,
                           const void* sin_cache, int64_t cache_rows, const int64_t* position_ids,
                           const int32_t* past_seq_lens, int32_t interleaved,
                           int32_t rotary_embedding_dim, void* q_out, void* k_out, void* k_cache,
                           void* v_cache, int64_t max_cache_len, int32_t* status_flags, void* scratch,
                           rope_stream_t stream);

/*
 * rope_apply_qkv_rmsnorm -- rope_apply_qkv with each Q and K head
 * RMS-normalised first, in the same launch ([Qwen3 fusion pull request, Qwen3
 * Architecture: QK-Norm applies RMSNorm to Q and K after the projection and
 * reshape, before RoPE; Verification: SimplifiedLayerNormalization, i.e.
 * RMSNorm, nodes]). For every Q (resp. K) head x of H elements:
 *   r = 1 / sqrt(mean_j(x_j^2) + epsilon),  z_j = T(w_j * T(x_j * r)),
 * with w = q_norm_weight (resp. k_norm_weight), each product rounded once to T
 * and the mean and r in float32; z is then rotated exactly as rope_apply_qkv
 * rotates a head (an out-of-range position copies z through; the tail past
 * the rotary width is z). V heads are not normalised.
 *
 * q_norm_weight, k_norm_weight  device T[head_size], both required.
 * epsilon       finite, >= 0 (Qwen3 uses 1e-6). With epsilon 0 an all-zero
 *               head divides by zero (inf/NaN), as the definition does.
 * Every other argument, layout, ownership and status bit as rope_apply_qkv.
 * The mean is computed by one group of at most 32 threads per head:
 * ROPE_ERR_UNSUPPORTED when a head has more than 32 units (16-byte vectors
 * on the aligned path: head_size <= 256 float16 or 128 float32 at full
 * rotation; single elements otherwise). ROPE_ERR_INVALID_ARG as
 * rope_apply_qkv, and for a missing weight, a misaligned weight or a bad
 * epsilon.
 */
rope_status rope_apply_qkv_rmsnorm(rope_dtype dtype, int64_t batch, int64_t seq, int32_t num_heads,
                                   int32_t kv_num_heads, int64_t head_size, const void* query,
                                   const void* key, const void* value, const void* q_norm_weight,
                                   const void* k_norm_weight, float epsilon, const void* cos_cache,
                                   const void* sin_cache, int64_t cache_rows,
                                   const int64_t* position_ids, const int32_t* past_seq_lens,
                                   int32_t interleaved, int32_t rotary_embedding_dim, void* q_out,
                                   void* k_out, void* k_cache, void* v_cache, int64_t max_cache_len,
                                   int32_t* status_flags, void* scratch, rope_stream_t stream);

/*
 * mrope_apply_fused -- MRotaryEmbedding with cos/sin computed on the fly
 * ([MRotaryEmbedding README, Description, Inputs, Attributes] for the three
 * position streams, mrope_section / mrope_layout and scale; [Qwen3 fusion
 * pull request, Motivation and Context] for the on-the-fly coefficients).
 *
 * Coefficient index i of token (b, s) follows stream m(i) (the map of
 * mrope_apply) at position p = position_ids[m(i), b, s]; its cos/sin are the
 * values rope_cache_build(inv_freq, attention_scaling) stores at row p, then
 * multiplied by `scale` and rounded to T as mrope_apply does. With no table
 * no position is out of range. Wherever the positions lie inside a table
 * built by rope_cache_build, the result equals mrope_apply over that table,
 * bit for bit.
 *
 * inv_freq      device float32[rd/2].
 * position_ids  device int64 (3, B, S), required.
 * Other arguments, layouts, ownership and errors as mrope_apply (no cache,
 * no status word, no scratch; packed batching is not offered).
 */
rope_status mrope_apply_fused(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape, const void* x,
                              void* y, const float* inv_freq, float attention_scaling,
                              const int64_t* position_ids, const int32_t* mrope_section,
                              int32_t mrope_layout, float scale, int32_t interleaved,
                              int32_t rotary_embedding_dim, int32_t num_heads, rope_stream_t stream);

/*
 * rope_cache_build -- the (rows, half) cos and sin tables of rope_apply's
 * 2-D cache: row p holds the coefficients rope_apply_fused computes for
 * position p ([Qwen3 fusion pull request, Medium Issues 4: cos(freqs) *
 * scaling with freqs[p, i] = p * inv_freq[i]]).
 *
 * inv_freq      device float32[half]; cos_out, sin_out device T[rows * half].
 * half >= 1, rows >= 0.
 */
rope_status rope_cache_build(rope_dtype dtype, const float* inv_freq, int32_t half, int64_t rows,
                             float attention_scaling, void* cos_out, void* sin_out,
                             rope_stream_t stream);

/*
 * Kernel variant selection (process-wide; default ROPE_VARIANT_AUTO).
 *   ROPE_VARIANT_AUTO  M-RoPE and partial rotation (rotary_embedding_dim <
 *                      head size) on the 128-bit vector path with X of at
 *                      least 8 MiB go through the TMA pipeline (shared-memory
 *                      stage ring); everything else, full-rotation RoPE
 *                      included, through the SIMT kernels (faster there).
 *   ROPE_VARIANT_SIMT  always the SIMT kernels.
 *   ROPE_VARIANT_TMA   the TMA pipeline whenever the shape allows it (vector
 *                      path, head size <= 256 elements), whatever its size.
 * All variants compute the same result. ([MRotaryEmbedding README,
 * Implementation variants]: one implementation is selected per call from the
 * device, the shapes and the dtypes.) Returns ROPE_ERR_INVALID_ARG for an
 * unknown value. No CUDA call.
 */
typedef enum rope_variant {
  ROPE_VARIANT_AUTO = 0,
  ROPE_VARIANT_SIMT = 1,
  ROPE_VARIANT_TMA = 2
} rope_variant;
rope_status rope_set_variant(rope_variant variant);
rope_variant rope_get_variant(void);

/*
 * mrope_apply_qkv -- rope_apply_qkv with multimodal RoPE: every Q and K head is
 * rotated exactly as mrope_apply rotates one head of a rank-3 X
 * ([MRotaryEmbedding README, Description: the three position streams t, h, w;
 * Inputs/positionIds; Attributes: mrope_section, mrope_layout, scale]), with
 * the grouped-query heads, packed or separate inputs and the key/value cache
 * append of rope_apply_qkv ([SparseAttention README, Description, Inputs]) and,
 * when q_norm_weight and k_norm_weight are given, the RMS normalisation of
 * rope_apply_qkv_rmsnorm first ([Qwen3 fusion pull request, Qwen3
 * Architecture: QK-Norm before the rotary step]). The pages describe these
 * pieces separately; their composition here follows each one unchanged.
 *
 * position_ids  device int64 (3, B, S), required: the t, h, w positions of
 *               every token. A pair whose stream position is outside
 *               [0, cache_rows) is copied through (the normalised value with
 *               the norm) and bit 0 of status_flags is set.
 * mrope_section, mrope_layout, scale  as mrope_apply (rd/2 <= 1024).
 * q_norm_weight, k_norm_weight  both NULL (no norm) or both device T[head_size];
 *               epsilon as rope_apply_qkv_rmsnorm.
 * Every other argument, layout, ownership, status bit and error as
 * rope_apply_qkv (head_size even; past_seq_lens only says where cache rows go,
 * positions always come from position_ids). ROPE_ERR_INVALID_ARG also for a
 * missing section or position_ids, sections that do not sum to rd/2, a layout
 * other than 0 or 1, or a non-finite scale.
 */
rope_status mrope_apply_qkv(rope_dtype dtype, int64_t batch, int64_t seq, int32_t num_heads,
                            int32_t kv_num_heads, int64_t head_size, const void* query, const void* key,
                            const void* value, const void* q_norm_weight, const void* k_norm_weight,
                            float epsilon, const void* cos_cache, const void* sin_cache, int64_t cache_rows,
                            const int64_t* position_ids, const int32_t* mrope_section, int32_t mrope_layout,
                            float scale, const int32_t* past_seq_lens, int32_t interleaved,
                            int32_t rotary_embedding_dim, void* q_out, void* k_out, void* k_cache,
                            void* v_cache, int64_t max_cache_len, int32_t* status_flags, void* scratch,
                            rope_stream_t stream);

/*
 * rope_apply_no_alloc -- rope_apply for callers that cannot allocate device
 * memory. The operator pages have no counterpart: this is a library-level
 * variant. rope_apply's dynamic tile schedule needs ROPE_SCRATCH_BYTES of
 * caller-owned device scratch; some callers cannot provide even that -- code
 * running inside CUDA stream capture (where allocating is not allowed),
 * plugins or runtimes that are handed only their input and output buffers,
 * callers without a device allocator. This entry point takes the scratch from
 * a fixed 256-byte array in the library's own device memory (every GPU that
 * loads the library holds it until the process exits; the schedule uses 16
 * bytes of it and no input size needs more). It allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library call.
 *
 * Arguments, results and errors are those of rope_apply without `scratch`
 * (shapes the pipelined kernel cannot take run the SIMT kernels, which use no
 * scratch). The first call on a device (and again after the device was reset,
 * or from another context on it) sets the array up: it looks up the array's
 * device address for the current context. Make that first call before any
 * stream capture that includes this entry point. The array is zero when the
 * library's device code is loaded, every call on a device shares it, and each
 * completed launch leaves it zero for the next: calls that overlap on the GPU
 * (different streams, different threads) race on it and must not be issued;
 * calls in one stream are fine.
 */
rope_status rope_apply_no_alloc(rope_dtype dtype, int32_t x_rank, const int64_t* x_shape,
                                const void* x, void* y, int32_t cache_rank,
                                const int64_t* cache_shape, const void* cos_cache,
                                const void* sin_cache, const int64_t* position_ids,
                                int32_t interleaved, int32_t rotary_embedding_dim,
                                int32_t num_heads, int32_t* oor_flag, rope_stream_t stream);

/* Static name of a status code. */
const char* rope_status_string(rope_status status);

/* Message describing the last failed call on the calling thread ("" if none).
   Valid until the next call into the library on this thread. */
const char* rope_last_error(void);

/* Kernel family that the last call on the calling thread which launched work
   used: "rope_rows_kernel" (SIMT), "rope_mrope_heads_kernel" (SIMT M-RoPE, several heads
   per thread), "rope_tma_kernel" (TMA pipeline),
   "rope_fused_kernel", "rope_qkv_kernel" (SIMT, one head per thread),
   "rope_qkv_heads_kernel" (SIMT Q/K, several heads of one role per thread),
   "rope_qkv_tma_kernel" (TMA pipeline) or "rope_cache_build_kernel"; "" before the first
   launch. Calls that fail or launch nothing (empty X) leave it unchanged.
   A diagnostic for profilers and benchmarks: the pages have no counterpart.
   The string is static; never free it. */
const char* rope_last_kernel(void);

#ifdef __cplusplus
}
#endif

#endif /* ROPE_GB300_H */
