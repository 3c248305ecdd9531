// TMA-pipelined rotary kernels for sm_103a.
//
// The operation streams X once and writes Y once; the bandwidth a streaming
// kernel reaches is set by how many bytes it keeps in flight. Here the bytes
// in flight live in shared memory, not registers: a producer warp moves whole
// tiles of X (TS tokens x NG heads x H) into a K-stage ring with TMA tensor
// copies, and gathers each token's cos/sin rows next to the tile with 16-byte
// asynchronous copies; eight consumer warps rotate the tile in place; one consumer thread
// writes the tile back with a TMA tensor store. Pass-through elements (the
// tail past the rotary width, tokens or pairs whose position is out of range)
// are never touched: the store writes back the bytes the load brought in.
//
// Pipeline protocol (per stage s, round r = tile index / K):
//   full[s]   count 33: producer lane 0's arrive.expect_tx(tile bytes), whose
//             TMA copy completes the transaction bytes, and one asynchronous
//             arrive per producer lane, triggered when that lane's cp.async
//             copies of the tile's cos/sin rows have landed.
// Tiles go to CTAs round robin, or -- when the caller gives a scratch counter --
// to whichever CTA's producer asks next (dynamic schedule); each stage records
// its tile index, and an index past the last tile ends the pipeline.
//   computed[s] count = consumer warps: each consumer warp arrives after it
//             has rotated its rows of the stage (and fenced them for TMA).
//   empty[s]  count 1: the store warp arrives once the TMA store of the stage
//             has finished reading shared memory, so the producer may refill it.
// Every wait is bounded (kWaitLimitNs of global time); a wait that runs out
// sets bit 1 of the caller's status word (if given) and the kernel leaves
// uniformly (consumers agree through a barrier reduction), after the
// producer has waited, again bounded, for the loads it issued.
//
// Definitions followed: "ai.onnx.RotaryEmbedding" WebGPU manifest (inputs,
// attributeDescriptions) and "com.microsoft.MRotaryEmbedding" README (Inputs,
// Attributes, Implementation variants/pairs4) -- the same arithmetic as
// rope_kernels.cuh, which this file shares.
#pragma once

#include <cuda.h>

#include "rope_kernels.cuh"

namespace rope_gb300 {

#ifndef ROPE_TMA_CONSUMER_WARPS
#define ROPE_TMA_CONSUMER_WARPS 8
#endif
#ifndef ROPE_TMA_MIN_CTAS
#define ROPE_TMA_MIN_CTAS 2
#endif
constexpr int kTmaConsumerWarps = ROPE_TMA_CONSUMER_WARPS;
constexpr int kTmaConsumers = kTmaConsumerWarps * 32;
constexpr int kTmaThreads = kTmaConsumers + 64;  // + producer warp + store warp
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kMaxGather = 8;  // 16-byte cos/sin pieces per producer lane per tile
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
  uint32_t pos_off;     // the tile's positions (producer scratch inside the stage)
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

// Positions of token `lane` of a tile (producer lanes), prefetched one tile ahead.
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
  const uint32_t empty0 = sbase + 8 * tp.K;      // empty[s]     at 8*(K+s)
  const uint32_t done0 = sbase + 16 * tp.K;      // computed[s]  at 8*(2K+s)
  unsigned char* stage0 = smem + tp.bar_bytes;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t row_bytes = (uint32_t)p.h * sizeof(bits);  // one cos (or sin) row

  if (threadIdx.x == 0) {
    for (int s = 0; s < tp.K; ++s) {
      mbar_init(full0 + 8 * s, 33);  // producer lane 0's arrive.expect_tx + every producer lane
      mbar_init(empty0 + 8 * s, 1);  // the store warp, once the stage's store has read it
      mbar_init(done0 + 8 * s, kTmaConsumerWarps);  // one arrive per consumer warp
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
  // producer before the stage's full barrier can complete); an index >= ntiles
  // is the sentinel that ends the consumers and the store warp.
  auto stage_tile = [&](int s) -> int64_t* {
    return reinterpret_cast<int64_t*>(stage0 + (size_t)s * tp.stage_bytes + tp.hdr_off);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    const bits* cosb = static_cast<const bits*>(p.cos);
    const bits* sinb = static_cast<const bits*>(p.sin);
    bool timed_out = false;
    // Gather roles: piece c of a full tile's coefficient block (16 bytes at
    // byte 16*c, layout [token][slot][cos|sin][rd/2]) goes to lane c % 32;
    // each lane's pieces are the same for every tile, so they are decoded once.
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
    // Tile j of this CTA: blockIdx.x + j*gridDim.x (static schedule), or the
    // next index drawn from the shared counter (dynamic schedule: CTAs that
    // run faster take more tiles, so all of them finish together).
    // X copies run D = K-1 tiles ahead of the cos/sin work: they need only the
    // tile index and a free stage, so the first copies leave at once and the
    // positions' latency never delays a tile copy.
    const int64_t D = tp.K - 1;
    // issue_x: lane 0 picks tile jj's index, records it in the stage and starts
    // its X copy; returns (on every lane) whether that was the sentinel.
    auto issue_x = [&](int64_t jj) -> bool {
      int64_t t = 0;
      if (lane == 0) {
        const int s = (int)(jj % tp.K);
        t = p.sched ? (int64_t)atomicAdd(p.sched, 1ull) : (int64_t)blockIdx.x + jj * (int64_t)gridDim.x;
        *stage_tile(s) = t;
        if (t < tp.ntiles) {
          const Tile tl = tile_of<RANK4>(p, tp, t);
          mbar_arrive_expect_tx(full0 + 8 * s, tp.x_bytes);
          tma_load_x<RANK4>(smem_addr(stage0 + (size_t)s * tp.stage_bytes), &tmx, tl.c, full0 + 8 * s, pol);
        } else {
          mbar_arrive(full0 + 8 * s);  // the sentinel carries no bytes
        }
      }
      t = __shfl_sync(0xffffffffu, t, 0);
      return t >= tp.ntiles;
    };
    bool ended = false;
    int64_t jx = 0;  // tiles whose X copy (or the sentinel) is issued
    for (; jx < D && !ended; ++jx) ended = issue_x(jx);
    __syncwarp();
    int64_t j = 0;
    TilePos<MODE> cur{};
    {
      const int64_t t0 = *stage_tile(0);
      if (t0 < tp.ntiles) cur = load_tile_pos<MODE>(p, tile_of<RANK4>(p, tp, t0), lane);
    }
    // Invariant: tile j's copy (or the sentinel) is out (j < jx) at the top of
    // every iteration, since the prologue issues D >= 1 of them and each
    // iteration issues one more until the sentinel.
    for (;; ++j) {
      const int s = (int)(j % tp.K);
      const int64_t t = *stage_tile(s);
      if (t >= tp.ntiles) {  // sentinel: complete its full barrier and stop
        cp_async_arrive(full0 + 8 * s);
        ++j;
        break;
      }
      // prefetch the next tile's positions (when its copy is already out)
      TilePos<MODE> nxt{};
      const bool have_nxt = j + 1 < jx;
      if (have_nxt) {
        const int64_t tn = *stage_tile((int)((j + 1) % tp.K));
        if (tn < tp.ntiles) nxt = load_tile_pos<MODE>(p, tile_of<RANK4>(p, tp, tn), lane);
      }
      const Tile tl = tile_of<RANK4>(p, tp, t);
      unsigned char* st = stage0 + (size_t)s * tp.stage_bytes;
      const uint32_t st_addr = smem_addr(st);
      uint32_t flags = 0;
      const bool mine = lane < tl.ntok;
      if (mine) {
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
      // The tile's cos/sin rows (layout [token][slot][cos|sin][rd/2]) are
      // gathered 16 bytes per copy from the L2-resident tables with
      // asynchronous copies that arrive on full[s] when they land, so the
      // producer never waits on the gather. Piece c sits at byte 16*c.
      const uint32_t coef_addr = st_addr + tp.coef_off;
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
      if (!ended && jx == j + D) {  // the next copy goes into the stage tile j-1 used
        const int64_t rx = jx / tp.K;
        if (rx > 0 && !__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * (jx % tp.K), (uint32_t)((rx - 1) & 1)))) {
          ++j;  // tile j's arrivals are complete
          timed_out = true;
          break;
        }
        ended = issue_x(jx);
        ++jx;
        __syncwarp();
      }
      if (!have_nxt && j + 1 < jx) {  // D = 1: the next copy only just went out
        const int64_t tn = *stage_tile((int)((j + 1) % tp.K));
        if (tn < tp.ntiles) nxt = load_tile_pos<MODE>(p, tile_of<RANK4>(p, tp, tn), lane);
      }
      cur = nxt;
    }
    // Leave only after every copy this warp issued has landed: the full
    // barriers of the stages it completed (the last K of them).
    for (int64_t q = j - tp.K > 0 ? j - tp.K : 0; q < j; ++q) {
      const int s = (int)(q % tp.K);
      if (!mbar_wait(full0 + 8 * s, (uint32_t)((q / tp.K) & 1))) timed_out = true;
    }
    if (timed_out) {
      // X copies issued ahead of cos/sin work that never happened: give them
      // time to land before the CTA's shared memory goes away (bounded).
      const uint64_t t0 = global_ns();
      while (global_ns() - t0 < 1000000ull) {
      }
      if (lane == 0 && p.oor_flag) atomicOr(p.oor_flag, 2);
    }
    if (p.sched && lane == 0) {
      // The last CTA to stop drawing resets the counter pair for the next launch.
      __threadfence();
      if (atomicAdd(p.sched + 1, 1ull) == (unsigned long long)gridDim.x - 1) {
        p.sched[0] = 0;
        p.sched[1] = 0;
        __threadfence();
      }
    }
    return;
  }

  if (warp == 1) {
    // ---------------------------------------------------------- store warp
    const uint64_t pol = policy_evict_first();
    bool timed_out = false;
    int64_t j = 0;
    for (;; ++j) {
      const int s = (int)(j % tp.K);
      if (!__all_sync(0xffffffffu, mbar_wait(done0 + 8 * s, (uint32_t)((j / tp.K) & 1)))) {
        timed_out = true;
        break;
      }
      const int64_t t = *stage_tile(s);
      if (t >= tp.ntiles) break;  // sentinel
      if (lane == 0) {
        const Tile tl = tile_of<RANK4>(p, tp, t);
        tma_store_y<RANK4>(&tmy, tl.c, smem_addr(stage0 + (size_t)s * tp.stage_bytes), pol);
        bulk_commit();
        bulk_wait_read_0();  // the stage may be refilled once the store has read it
        mbar_arrive(empty0 + 8 * s);
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
    if (timed_out && lane == 0 && p.oor_flag) atomicOr(p.oor_flag, 2);
    return;
  }

  // -------------------------------------------------------------- consumers
  // Thread q owns column (token ts, pair unit k) of the tile for up to
  // kMaxHeads heads ng = hq, hq + tpc, ... The column's cos/sin (for M-RoPE:
  // the three streams merged) are read once and reused for every head.
  const int q = threadIdx.x - 64;
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
  int64_t j = 0;
  for (;; ++j) {
    const int s = (int)(j % tp.K);
    // the lanes of a warp agree, so a timeout never splits a warp
    const bool ok = __all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (uint32_t)((j / tp.K) & 1)));
    const int64_t t = ok ? *stage_tile(s) : 0;
    if (ok && t >= tp.ntiles) {  // sentinel: hand it to the store warp and stop
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
            rotate_unit<T, V, INTER>(a[u], bv[u], c, sn, ya, yb);
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
    if (!ok) {  // the producer, the store warp and the other consumer warps also give up
      timed_out = true;
      break;
    }
    fence_async_smem();  // this thread's smem writes, before the TMA store reads them
    __syncwarp();
    if (lane == 0) mbar_arrive(done0 + 8 * s);
  }
  if (timed_out && lane == 0 && p.oor_flag) atomicOr(p.oor_flag, 2);
}

}  // namespace rope_gb300
