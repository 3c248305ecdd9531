// TMA-pipelined rotary kernels for sm_103a.
//
// The operation streams X once and writes Y once; the bandwidth a streaming
// kernel reaches is set by how many bytes it keeps in flight. Here the bytes
// in flight live in shared memory, not registers. Each CTA runs a K-stage ring
// of tiles (TS tokens x NG heads x H) with three warp roles:
//   copy warp     (lane 0) starts each tile's TMA tensor copy into a free
//                 stage and writes rotated tiles back with TMA tensor stores;
//                 a stage is refilled the moment its store has read it;
//   gather warp   loads the tile's positions (one tile ahead) and gathers each
//                 token's cos/sin rows next to the tile with 16-byte
//                 asynchronous copies;
//   consumers     rotate the tile in place (ROPE_TMA_CONSUMER_WARPS warps).
// Pass-through elements (the tail past the rotary width, tokens or pairs whose
// position is out of range) are never touched: the store writes back the
// bytes the load brought in.
//
// Pipeline protocol (per stage s, round r = tile index / K):
//   issued[s]   count 1: the copy warp, after writing the stage's tile index
//               (its header) and starting the copy.
//   landed[b]   count 1, a ring of 2K (tile jj uses landed[jj mod 2K]): the
//               copy warp's arrive.expect_tx(tile bytes), whose TMA copy
//               completes the transaction bytes (a plain arrive for the
//               sentinel). Only the copy hardware completes it, so the copy
//               warp can always wait for its own loads. With 2K of them, the
//               barrier of tile jj is reused by tile jj + 2K, which cannot be
//               started before every warp has finished tile jj + K: a parity
//               wait on tile jj's phase never sees a later one.
//   full[s]     count 32: one asynchronous arrive per gather lane, triggered
//               when that lane's cp.async copies of the tile's cos/sin rows
//               have landed.
//   computed[s] count = consumer warps: each consumer warp arrives after it
//               has rotated its rows of the stage (and fenced them for TMA).
// Consumers wait on tile j's landed barrier and full[s].
// Tiles go to CTAs round robin, or -- when the caller gives a scratch counter --
// to whichever CTA's copy warp asks next (dynamic schedule); an index past the
// last tile (the sentinel) ends the pipeline.
// Every wait is bounded (kWaitLimitNs of global time); a wait that runs out
// sets bit 1 of the caller's status word (if given) and the kernel leaves
// uniformly (each warp agrees through a warp vote). No copy into shared
// memory is left in flight when a CTA leaves: the gather warp waits for its
// cp.async copies, and the copy warp waits, again bounded, on landed[] for
// every tile load it started that no consumer has seen complete.
//
// Definitions followed: "ai.onnx.RotaryEmbedding" WebGPU manifest (inputs,
// attributeDescriptions) and "com.microsoft.MRotaryEmbedding" README (Inputs,
// Attributes, Implementation variants/pairs4) -- the same arithmetic as
// rope_kernels.cuh, which this file shares.
#pragma once

#include <cuda.h>

#include "rope_kernels.cuh"
#include "rope_packed.cuh"

namespace rope_gb300 {


#ifndef ROPE_TMA_CONSUMER_WARPS
#define ROPE_TMA_CONSUMER_WARPS 8
#endif
#ifndef ROPE_TMA_MIN_CTAS
#define ROPE_TMA_MIN_CTAS 2
#endif
constexpr int kTmaConsumerWarps = ROPE_TMA_CONSUMER_WARPS;
constexpr int kTmaConsumers = kTmaConsumerWarps * 32;
constexpr int kTmaRoleWarps = 2;  // the copy warp and the gather warp
constexpr int kTmaThreads = kTmaConsumers + 32 * kTmaRoleWarps;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kMaxGather = 8;  // 16-byte cos/sin pieces per gather lane per tile
constexpr int kMaxHeads = 4;   // heads one consumer thread rotates per tile column

struct TParams {
  int32_t TS, NG, K;    // tokens per tile, heads per tile, pipeline stages
  int32_t slots;        // coefficient rows gathered per token: 1 (RoPE) or 3 (M-RoPE)
  int64_t ntiles;
  int32_t head_groups;  // ceil(N / NG)
  int32_t s_tiles;      // rank 4: ceil(S / TS)
  uint32_t x_bytes;     // bytes of one X box
  uint32_t coef_off;    // stage offsets: coefficient rows, per-token flags
  uint32_t flag_off;
  uint32_t pos_off;     // the tile's positions (gather warp scratch inside the stage)
  uint32_t hdr_off;     // the stage's tile index (8 bytes)
  uint32_t stage_bytes;
  uint32_t bar_bytes;   // barrier block in front of stage 0
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// A waiting thread is suspended (it issues nothing) until the phase completes
// or kSuspendHintNs elapse, so waiting warps leave the issue slots to the
// warps that have work.
constexpr uint32_t kSuspendHintNs = 1000000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Whether the phase of `bar` with parity `parity` has completed (no waiting).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete; false after
// kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

template <bool RANK4>
__device__ __forceinline__ void tma_load_x(uint32_t dst, const CUtensorMap* map, const int* c,
                                           uint32_t bar, uint64_t pol) {
  if (RANK4) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(bar),
        "l"(pol)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(bar), "l"(pol)
        : "memory");
  }
}

template <bool RANK4>
__device__ __forceinline__ void tma_store_y(const CUtensorMap* map, const int* c, uint32_t src,
                                            uint64_t pol) {
  if (RANK4) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group.L2::cache_hint"
        " [%0, {%1, %2, %3, %4}], [%5], %6;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(src), "l"(pol)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint"
        " [%0, {%1, %2, %3}], [%4], %5;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(src), "l"(pol)
        : "memory");
  }
}

// 16-byte asynchronous copy global -> shared (LSU path, not the TMA unit).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (counts as one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_read_0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Tile geometry
// ---------------------------------------------------------------------------
struct Tile {
  int64_t tok0;  // first token of the tile
  int ntok;      // tokens of the tile inside X (the box may run past the end)
  int64_t n0;    // first head
  int c[4];      // TMA box coordinates, innermost first
};

template <bool RANK4>
__device__ __forceinline__ Tile tile_of(const KParams& p, const TParams& tp, int64_t t64) {
  Tile tl;
  const uint32_t t = (uint32_t)t64;  // tile counts stay below 2^31
  if (!RANK4) {
    // X viewed as (ntok, N, H); box (TS, NG, H)
    const uint32_t hg = tp.head_groups == 1 ? 0u : t % (uint32_t)tp.head_groups;
    const uint32_t tt = tp.head_groups == 1 ? t : t / (uint32_t)tp.head_groups;
    tl.tok0 = (int64_t)tt * tp.TS;
    const int64_t left = p.ntok - tl.tok0;
    tl.ntok = (int)(left < tp.TS ? left : tp.TS);
    tl.n0 = (int64_t)hg * tp.NG;
    tl.c[0] = 0;
    tl.c[1] = (int)tl.n0;
    tl.c[2] = (int)tl.tok0;
    tl.c[3] = 0;
  } else {
    // X is (B, N, S, H); box (1, NG, TS, H)
    const uint32_t st = t % (uint32_t)tp.s_tiles;
    const uint32_t rest = t / (uint32_t)tp.s_tiles;
    const uint32_t hg = tp.head_groups == 1 ? 0u : rest % (uint32_t)tp.head_groups;
    const uint32_t b = tp.head_groups == 1 ? rest : rest / (uint32_t)tp.head_groups;
    const int64_t s0 = (int64_t)st * tp.TS;
    tl.tok0 = (int64_t)b * p.S + s0;
    const int64_t left = p.S - s0;
    tl.ntok = (int)(left < tp.TS ? left : tp.TS);
    tl.n0 = (int64_t)hg * tp.NG;
    tl.c[0] = 0;
    tl.c[1] = (int)s0;
    tl.c[2] = (int)tl.n0;
    tl.c[3] = (int)b;
  }
  return tl;
}

// Positions of token `lane` of a tile (gather lanes), prefetched one tile ahead.
template <Coef MODE>
struct TilePos {
  int64_t v[MODE == Coef::kMRope ? 3 : 1];
};

template <Coef MODE>
__device__ __forceinline__ TilePos<MODE> load_tile_pos(const KParams& p, const Tile& tl, int lane) {
  TilePos<MODE> tp;
#pragma unroll
  for (int k = 0; k < (MODE == Coef::kMRope ? 3 : 1); ++k) tp.v[k] = -1;
  if (MODE == Coef::kCache3D || lane >= tl.ntok) return tp;
  const int64_t tok = tl.tok0 + lane;
  if (MODE == Coef::kCache2D) {
    tp.v[0] = __ldg(p.pos + tok);
  } else if (MODE == Coef::kMRope) {
#pragma unroll
    for (int k = 0; k < 3; ++k) tp.v[k] = __ldg(p.pos + k * p.ntok + tok);
  }
  return tp;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <class T, bool INTER, bool RANK4, Coef MODE>
__global__ void __launch_bounds__(kTmaThreads, ROPE_TMA_MIN_CTAS)
    rope_tma_kernel(const KParams p, const TParams tp, const __grid_constant__ CUtensorMap tmx,
                    const __grid_constant__ CUtensorMap tmy) {
  using E = Elem<T>;
  using bits = typename E::bits;
  constexpr int V = 16 / sizeof(bits);
  using VT = VecT<T, V>;
  constexpr int SLOTS = MODE == Coef::kMRope ? 3 : 1;

  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase;                  // full[s]      at 8*s
  const uint32_t done0 = sbase + 8 * tp.K;       // computed[s]  at 8*(K+s)
  const uint32_t issued0 = sbase + 16 * tp.K;    // issued[s]    at 8*(2K+s)
  const uint32_t landed0 = sbase + 24 * tp.K;    // landed[b]    at 8*(3K+b), b < 2K
  // tile jj's landed barrier and the parity of its phase there
  auto landed_bar = [&](int64_t jj) -> uint32_t { return landed0 + 8 * (uint32_t)(jj % (2 * tp.K)); };
  auto landed_par = [&](int64_t jj) -> uint32_t { return (uint32_t)((jj / (2 * tp.K)) & 1); };
  unsigned char* stage0 = smem + tp.bar_bytes;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t row_bytes = (uint32_t)p.h * sizeof(bits);  // one cos (or sin) row

  if (threadIdx.x == 0) {
    for (int s = 0; s < tp.K; ++s) {
      mbar_init(full0 + 8 * s, 32);  // every gather lane
      mbar_init(done0 + 8 * s, kTmaConsumerWarps);  // one arrive per consumer warp
      mbar_init(issued0 + 8 * s, 1);  // the copy warp, once the stage header is written
      mbar_init(landed0 + 8 * s, 1);  // the X copy's arrive.expect_tx (two per stage)
      mbar_init(landed0 + 8 * (tp.K + s), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmy)) : "memory");
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // everything above overlaps the previous kernel's tail

  // Each stage starts with the index of the tile it holds (written by the
  // copy warp before the stage's full barrier can complete); an index >= ntiles
  // is the sentinel that ends the gather warp, the consumers and the copy warp.
  auto stage_tile = [&](int s) -> int64_t* {
    return reinterpret_cast<int64_t*>(stage0 + (size_t)s * tp.stage_bytes + tp.hdr_off);
  };

  if (warp == 0) {
    // --------------------------------------------------- copy warp (lane 0)
    // Starts the X copies and writes the rotated tiles back. The first K
    // tiles' copies leave at once; after that, the moment the TMA store of
    // tile j has finished reading its stage, the same lane refills the stage
    // with tile j+K. Tile indices are blockIdx.x + j*gridDim.x, or -- dynamic
    // schedule -- the next value of the shared counter, so CTAs that run
    // faster take more tiles. Each index is recorded in the stage header and
    // published to the gather warp through issued[s].
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      bool timed_out = false;
      auto pick = [&](int64_t jj) -> int64_t {  // the index of this CTA's tile jj
        return p.sched ? (int64_t)atomicAdd(p.sched, 1ull) : (int64_t)blockIdx.x + jj * (int64_t)gridDim.x;
      };
      // stage and landed slot of the next tile issued (jx % K, jx % 2K),
      // stepped per issue: this lane's serial path between a store and the
      // refill it allows is the pipeline's critical path when K is 2
      int is_s = 0, is_l = 0;
      auto issue = [&](int64_t t, const Tile& tl) {
        const int s = is_s;
        const uint32_t lb = landed0 + 8 * (uint32_t)is_l;
        *stage_tile(s) = t;
        if (t < tp.ntiles) {
          mbar_arrive_expect_tx(lb, tp.x_bytes);
          tma_load_x<RANK4>(smem_addr(stage0 + (size_t)s * tp.stage_bytes), &tmx, tl.c, lb, pol);
        } else {
          mbar_arrive(lb);  // the sentinel carries no bytes
        }
        mbar_arrive(issued0 + 8 * s);  // publishes the header to the gather warp
        if (++is_s == tp.K) is_s = 0;
        if (++is_l == 2 * tp.K) is_l = 0;
      };
      bool ended = false;
      int64_t jx = 0;  // tiles issued (the sentinel included)
      for (; jx < tp.K && !ended; ++jx) {
        const int64_t t = pick(jx);
        Tile tl{};
        if (t < tp.ntiles) tl = tile_of<RANK4>(p, tp, t);
        issue(t, tl);
        ended = t >= tp.ntiles;
      }
      // The next store's tile and the next refill's tile are worked out while
      // the previous store is still reading its stage, so nothing but the
      // copies' issue sits between one store and the next.
      int64_t t_st = *stage_tile(0);
      Tile tl_st{};
      if (t_st < tp.ntiles) tl_st = tile_of<RANK4>(p, tp, t_st);
      int64_t j = 0;  // the tile whose store comes next
      int s = 0;      // its stage (j % K) and the parity of its phase there
      uint32_t ph = 0;
      for (;; ++j) {
        if (!mbar_wait(done0 + 8 * s, ph)) {
          timed_out = true;
          break;
        }
        if (t_st >= tp.ntiles) break;  // sentinel
        tma_store_y<RANK4>(&tmy, tl_st.c, smem_addr(stage0 + (size_t)s * tp.stage_bytes), pol);
        bulk_commit();
        int64_t t_new = 0;
        Tile tl_new{};
        if (!ended) {
          t_new = pick(jx);
          if (t_new < tp.ntiles) tl_new = tile_of<RANK4>(p, tp, t_new);
        }
        if (++s == tp.K) {
          s = 0;
          ph ^= 1u;
        }
        // tile j+1 is already issued (K >= 2), so its header is in place
        t_st = *stage_tile(s);
        if (t_st < tp.ntiles) tl_st = tile_of<RANK4>(p, tp, t_st);
        if (!ended) {
          bulk_wait_read_0();  // the stage may be refilled once the store has read it
          issue(t_new, tl_new);  // jx == j + K: the tile that goes into tile j's stage next
          ended = t_new >= tp.ntiles;
          ++jx;
        }
      }
      bulk_wait_all();
      if (timed_out) {
        // Tiles j .. jx-1 were started and never stored: their loads must
        // land before the CTA's shared memory goes away. Each one's landed
        // phase is completed by the copy hardware alone (the sentinel's by its
        // plain arrive), and nothing later was started, so no wait aliases.
        for (int64_t jj = j; jj < jx; ++jj) (void)mbar_wait(landed_bar(jj), landed_par(jj));
        if (p.oor_flag) atomicOr(p.oor_flag, 2);
      }
      if (p.sched) {
        // The last CTA to stop drawing resets the counter pair for the next launch.
        __threadfence();
        if (atomicAdd(p.sched + 1, 1ull) == (unsigned long long)gridDim.x - 1) {
          p.sched[0] = 0;
          p.sched[1] = 0;
          __threadfence();
        }
      }
    }
    return;
  }

  if (warp == 1) {
    // ------------------------------------------------------------ gather warp
    // For each tile, once its stage holds the header: the tokens' flags and
    // positions, then the cos/sin rows (layout [token][slot][cos|sin][rd/2])
    // gathered 16 bytes per copy from the L2-resident tables by asynchronous
    // copies that arrive on full[s] when they land, so this warp never waits
    // on the gather. The next tile's positions are loaded one tile ahead.
    const bits* cosb = static_cast<const bits*>(p.cos);
    const bits* sinb = static_cast<const bits*>(p.sin);
    bool timed_out = false;
    // Piece c of a full tile's coefficient block (16 bytes at byte 16*c) goes
    // to lane c % 32; each lane's pieces are the same for every tile, so they
    // are decoded once.
    const int ch = (int)(row_bytes / 16);
    const int per_tok = SLOTS * 2 * ch;
    const int pieces = tp.TS * per_tok;
    const int n_gather = (pieces - lane + 31) / 32;
    int g_lt[kMaxGather], g_k[kMaxGather], g_piece[kMaxGather];
    bool g_sin[kMaxGather];
    uint32_t g_dst[kMaxGather];
#pragma unroll
    for (int g = 0; g < kMaxGather; ++g) {
      const int c = lane + 32 * g;
      const int lt = c / per_tok;
      const int rem = c - lt * per_tok;
      const int k = rem / (2 * ch);
      const int rem2 = rem - k * 2 * ch;
      g_lt[g] = lt;
      g_k[g] = k;
      g_sin[g] = rem2 >= ch;
      g_piece[g] = rem2 % ch;
      g_dst[g] = 16u * (uint32_t)c;
    }
    // Static schedule: tile indices are known in advance, so positions are
    // prefetched before the stage is even free. Dynamic schedule: the next
    // index is read from its stage header when that is already published.
    TilePos<MODE> cur{};
    bool have_cur = false;
    if (!p.sched) {
      if ((int64_t)blockIdx.x < tp.ntiles) cur = load_tile_pos<MODE>(p, tile_of<RANK4>(p, tp, blockIdx.x), lane);
      have_cur = true;
    }
    // tile j's stage and phase parity (j % K, (j / K) & 1) and landed slot
    // (j % 2K, (j / 2K) & 1); the same for tile j-1, which rank 4 waits on
    int s = 0, lsl = 0, s_prev = 0, lsl_prev = 0;
    uint32_t ph = 0, lph = 0, ph_prev = 0, lph_prev = 0;
    for (int64_t j = 0;; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(issued0 + 8 * s, ph))) {
        timed_out = true;
        break;
      }
      const int64_t t = *stage_tile(s);
      if (t >= tp.ntiles) {  // sentinel: complete its full barrier and stop
        cp_async_arrive(full0 + 8 * s);
        break;
      }
      const Tile tl = tile_of<RANK4>(p, tp, t);
      if (!have_cur) cur = load_tile_pos<MODE>(p, tl, lane);
      // Rank 4: a tile is NG strided blocks of TS*H elements, and those loads
      // run best with the least in flight, so the gather of tile j waits until
      // tile j-1 is complete: its data and this warp's own row copies for it
      // (measured: waiting for the data alone lets the row copies run ahead,
      // rank-4 partial rotation 84.0 -> 90.7 us). Neither parity can alias:
      // the landed barrier's next use, tile j-1+2K, and full[s]'s next phase,
      // tile j-1+K, both need this warp's arrival for tile j-1+K first.
      if (RANK4 && j > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(landed0 + 8 * (uint32_t)lsl_prev, lph_prev) &&
                                       mbar_wait(full0 + 8 * s_prev, ph_prev))) {
        timed_out = true;
        break;
      }
      // the stage and parity of tile j+1
      const int sn = s + 1 == tp.K ? 0 : s + 1;
      const uint32_t phn = s + 1 == tp.K ? ph ^ 1u : ph;
      TilePos<MODE> nxt{};
      bool have_nxt = false;
      if (!p.sched) {
        const int64_t tn = (int64_t)blockIdx.x + (j + 1) * (int64_t)gridDim.x;
        if (tn < tp.ntiles) nxt = load_tile_pos<MODE>(p, tile_of<RANK4>(p, tp, tn), lane);
        have_nxt = true;
      } else {
        // the copy warp publishes headers in tile order, and tile j+1-K's
        // phase of that barrier is already complete, so the parity test
        // cannot alias
        if (__all_sync(0xffffffffu, mbar_test(issued0 + 8 * sn, phn))) {
          const int64_t tn = *stage_tile(sn);
          if (tn < tp.ntiles) nxt = load_tile_pos<MODE>(p, tile_of<RANK4>(p, tp, tn), lane);
          have_nxt = true;
        }
      }
      unsigned char* st = stage0 + (size_t)s * tp.stage_bytes;
      uint32_t flags = 0;
      if (lane < tl.ntok) {
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
          bool ok;
          if (MODE == Coef::kCache3D)
            ok = true;
          else
            ok = (uint64_t)cur.v[k] < (uint64_t)p.cache_rows;
          if (ok) flags |= 1u << k;
        }
        if (MODE != Coef::kCache3D && flags != (1u << SLOTS) - 1 && p.oor_flag) atomicOr(p.oor_flag, 1);
      }
      if (lane < tp.TS) {
        reinterpret_cast<uint32_t*>(st + tp.flag_off)[lane] = flags;
        if (MODE != Coef::kCache3D) {
#pragma unroll
          for (int k = 0; k < SLOTS; ++k) reinterpret_cast<int64_t*>(st + tp.pos_off)[lane * SLOTS + k] = cur.v[k];
        }
      }
      __syncwarp();  // the flags and positions precede the gather and the lanes' (releasing) arrivals
      const uint32_t coef_addr = smem_addr(st) + tp.coef_off;
#pragma unroll
      for (int g = 0; g < kMaxGather; ++g) {
        if (g >= n_gather) break;
        const int lt = g_lt[g];
        if (lt >= tl.ntok) continue;
        int64_t row;
        uint32_t fl;
        if (MODE == Coef::kCache3D) {
          row = tl.tok0 + lt;
          fl = 1u;
        } else {
          // token lt's position(s) and flags were published by lane lt above
          fl = reinterpret_cast<const uint32_t*>(st + tp.flag_off)[lt];
          row = reinterpret_cast<const int64_t*>(st + tp.pos_off)[lt * SLOTS + g_k[g]];
        }
        if ((fl >> g_k[g]) & 1u)
          cp_async16(coef_addr + g_dst[g], reinterpret_cast<const uint4*>(
                                               (g_sin[g] ? sinb : cosb) + row * p.h) + g_piece[g]);
      }
      cp_async_arrive(full0 + 8 * s);
      cur = nxt;
      have_cur = have_nxt;
      s_prev = s;
      ph_prev = ph;
      lsl_prev = lsl;
      lph_prev = lph;
      s = sn;
      ph = phn;
      if (++lsl == 2 * tp.K) {
        lsl = 0;
        lph ^= 1u;
      }
    }
    // every copy this warp issued has landed before it leaves
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (timed_out && lane == 0 && p.oor_flag) atomicOr(p.oor_flag, 2);
    return;
  }
  // -------------------------------------------------------------- consumers
  // Thread q owns column (token ts, pair unit k) of the tile for up to
  // kMaxHeads heads ng = hq, hq + tpc, ... The column's cos/sin (for M-RoPE:
  // the three streams merged) are read once and reused for every head.
  const int q = threadIdx.x - 32 * kTmaRoleWarps;
  const int nP = p.nP;
  const int cols = tp.TS * nP;
  const int tpc = kTmaConsumers / cols;  // threads per column (the host keeps cols <= consumers)
  const int col = q % cols;
  const int hq = q / cols;
  const bool has_col = hq < tpc;
  const int ts = col / nP;
  const int k = col - ts * nP;
  int oa, ob;
  unit_offsets<V, INTER>(k, p.h, oa, ob);
  const int oc = k * V;
  uint32_t um = 0, present = 0;  // M-RoPE: stream of each of the unit's V indices
  uint32_t m0[4] = {0, 0, 0, 0}, m1[4] = {0, 0, 0, 0};
  if (MODE == Coef::kMRope) {
    const uint32_t word = p.smap[oc >> 4];
    um = (word >> ((oc & 15) * 2)) & (uint32_t)((1ull << (2 * V)) - 1);
#pragma unroll
    for (int jj = 0; jj < V; ++jj) present |= 1u << ((um >> (2 * jj)) & 3);
    stream_masks<V>(um, m0, m1);
  }
  bool timed_out = false;
  // tile j's stage s and full parity, landed slot and parity (j % K,
  // (j / K) & 1, j % 2K, (j / 2K) & 1), stepped once per tile
  int s = 0, lsl = 0;
  uint32_t ph = 0, lph = 0;
  for (;;) {
    // the lanes of a warp agree, so a timeout never splits a warp
    const bool ok = __all_sync(0xffffffffu, mbar_wait(landed0 + 8 * (uint32_t)lsl, lph) &&
                                                mbar_wait(full0 + 8 * s, ph));
    const int64_t t = ok ? *stage_tile(s) : 0;
    if (ok && t >= tp.ntiles) {  // sentinel: hand it to the copy warp and stop
      __syncwarp();
      if (lane == 0) mbar_arrive(done0 + 8 * s);
      break;
    }
    const Tile tl = tile_of<RANK4>(p, tp, t);
    unsigned char* st = stage0 + (size_t)s * tp.stage_bytes;
    if (ok && has_col && ts < tl.ntok) {
      const uint32_t fl = reinterpret_cast<const uint32_t*>(st + tp.flag_off)[ts];
      const bits* scoef = reinterpret_cast<const bits*>(st + tp.coef_off);
      bits* sx = reinterpret_cast<bits*>(st);
      // the column's rows (element offsets into the stage)
      bool act[kMaxHeads];
      uint32_t rowo[kMaxHeads];
#pragma unroll
      for (int u = 0; u < kMaxHeads; ++u) {
        const int ng = hq + u * tpc;
        act[u] = ng < tp.NG && tl.n0 + ng < p.N;
        const int r = RANK4 ? ng * tp.TS + ts : ts * tp.NG + ng;
        rowo[u] = (uint32_t)r * (uint32_t)p.H;
      }
      bool fast = true;
      bool blend_on = false;
      uint32_t ma[4], mb[4];
      VT c, sn;
      if (MODE != Coef::kMRope) {
        fast = fl & 1u;  // otherwise the position is out of range: the rows stay as loaded
        if (fast) {
          const bits* cr = scoef + (size_t)ts * 2 * p.h;
          c = *reinterpret_cast<const VT*>(cr + oc);
          sn = *reinterpret_cast<const VT*>(cr + p.h + oc);
        }
      } else {
        const bits* cr = scoef + (size_t)ts * 3 * 2 * p.h;
        const uint32_t valid = fl & present;
        VT cs[3], ss[3];
#pragma unroll
        for (int st3 = 0; st3 < 3; ++st3) {
          cs[st3] = VT{};
          ss[st3] = VT{};
          if ((valid >> st3) & 1u) {
            cs[st3] = *reinterpret_cast<const VT*>(cr + (size_t)st3 * 2 * p.h + oc);
            ss[st3] = *reinterpret_cast<const VT*>(cr + (size_t)st3 * 2 * p.h + p.h + oc);
          }
        }
        c = merge3(cs[0], cs[1], cs[2], m0, m1);
        sn = merge3(ss[0], ss[1], ss[2], m0, m1);
        if (!p.scale_is_one) {
          scale_round<T, V>(c, p.scale);
          scale_round<T, V>(sn, p.scale);
        }
        // pairs whose stream is out of range are put back from X after the rotation
        blend_on = valid != present;
        if (blend_on) pair_masks<V, INTER>(um, valid, ma, mb);
      }
      // 16-bit storage: the column's coefficients unpacked to float32 pairs
      // once, every head rotated with float32x2 operations (the same bits as
      // the scalar form; measured on M-RoPE 39.1 -> 38.4 us per launch from a
      // graph and 44.6 -> 42.6 us alone, rank-4 partial rotation unchanged)
      constexpr bool PACKED = sizeof(bits) == 2 && V == 8;
      float2 cf[4], sf[4];
      if constexpr (PACKED) {
        if (fast) {
          unpack_coef8<T>(reinterpret_cast<const VecT<T, 8>&>(c), cf);
          unpack_coef8<T>(reinterpret_cast<const VecT<T, 8>&>(sn), sf);
        }
      }
      if (fast) {
        // X loads of HOIST heads are issued together, then rotated and stored
        constexpr int HOIST = MODE == Coef::kMRope ? 2 : kMaxHeads;
#pragma unroll
        for (int u0 = 0; u0 < kMaxHeads; u0 += HOIST) {
          VT a[HOIST], bv[HOIST];
#pragma unroll
          for (int u = 0; u < HOIST; ++u) {
            if (act[u0 + u]) {
              a[u] = *reinterpret_cast<const VT*>(sx + rowo[u0 + u] + oa);
              bv[u] = *reinterpret_cast<const VT*>(sx + rowo[u0 + u] + ob);
            }
          }
#pragma unroll
          for (int u = 0; u < HOIST; ++u) {
            if (!act[u0 + u]) continue;
            VT ya, yb;
            if constexpr (PACKED) {
              Unit8<T> ua, ub, ra, rb;
              __builtin_memcpy(&ua, &a[u], 16);
              __builtin_memcpy(&ub, &bv[u], 16);
              rotate8p<T, INTER>(ua, ub, cf, sf, ra, rb);
              __builtin_memcpy(&ya, &ra, 16);
              __builtin_memcpy(&yb, &rb, 16);
            } else {
              rotate_unit<T, V, INTER>(a[u], bv[u], c, sn, ya, yb);
            }
            if (MODE == Coef::kMRope && blend_on) {
              blend(ya, a[u], ma);
              blend(yb, bv[u], mb);
            }
            *reinterpret_cast<VT*>(sx + rowo[u0 + u] + oa) = ya;
            *reinterpret_cast<VT*>(sx + rowo[u0 + u] + ob) = yb;
          }
        }
      }
    }
    if (!ok) {  // the copy and gather warps and the other consumer warps also give up
      timed_out = true;
      break;
    }
    fence_async_smem();  // this thread's smem writes, before the TMA store reads them
    __syncwarp();
    if (lane == 0) mbar_arrive(done0 + 8 * s);
    if (++s == tp.K) {
      s = 0;
      ph ^= 1u;
    }
    if (++lsl == 2 * tp.K) {
      lsl = 0;
      lph ^= 1u;
    }
  }
  if (timed_out && lane == 0 && p.oor_flag) atomicOr(p.oor_flag, 2);
}

}  // namespace rope_gb300
