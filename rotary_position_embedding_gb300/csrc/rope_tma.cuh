// TMA-pipelined rotary kernels for sm_103a.
//
// The operation streams X once and writes Y once; the bandwidth a streaming
// kernel reaches is set by how many bytes it keeps in flight. Here the bytes
// in flight live in shared memory, not registers: a producer warp moves whole
// tiles of X (TS tokens x NG heads x H) into a K-stage ring with TMA tensor
// copies, and gathers each token's cos/sin rows next to the tile with
// coalesced loads; eight consumer warps rotate the tile in place; one consumer thread
// writes the tile back with a TMA tensor store. Pass-through elements (the
// tail past the rotary width, tokens or pairs whose position is out of range)
// are never touched: the store writes back the bytes the load brought in.
//
// Pipeline protocol (per stage s, round r = tile index / K):
//   full[s]   count 33: producer lane 0's arrive.expect_tx(tile bytes), whose
//             TMA copy completes the transaction bytes, and one arrive per
//             producer lane after it has stored its share of the tile's
//             cos/sin rows into the stage.
//   empty[s]  count 1: consumer thread 0 arrives once the TMA store of the
//             stage has finished reading shared memory.
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

constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaConsumers = kTmaConsumerWarps * 32;
constexpr int kTmaThreads = kTmaConsumers + 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

struct TParams {
  int32_t TS, NG, K;    // tokens per tile, heads per tile, pipeline stages
  int32_t slots;        // coefficient rows gathered per token: 1 (RoPE) or 3 (M-RoPE)
  int64_t ntiles;
  int32_t head_groups;  // ceil(N / NG)
  int32_t s_tiles;      // rank 4: ceil(S / TS)
  uint32_t x_bytes;     // bytes of one X box
  uint32_t coef_off;    // stage offsets: coefficient rows, per-token flags
  uint32_t flag_off;
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

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
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

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumers) : "memory");
}

// Barrier among the consumer warps that also ORs a predicate across them.
__device__ __forceinline__ bool consumer_any(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 2, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)pred), "n"(kTmaConsumers)
      : "memory");
  return out != 0;
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
__global__ void __launch_bounds__(kTmaThreads, 2)
    rope_tma_kernel(const KParams p, const TParams tp, const __grid_constant__ CUtensorMap tmx,
                    const __grid_constant__ CUtensorMap tmy) {
  using E = Elem<T>;
  using bits = typename E::bits;
  constexpr int V = 16 / sizeof(bits);
  using VT = VecT<T, V>;
  constexpr int SLOTS = MODE == Coef::kMRope ? 3 : 1;

  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase;                 // full[s]  at  8*s
  const uint32_t empty0 = sbase + 8 * tp.K;     // empty[s] at  8*(K+s)
  unsigned char* stage0 = smem + tp.bar_bytes;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t row_bytes = (uint32_t)p.h * sizeof(bits);  // one cos (or sin) row

  if (threadIdx.x == 0) {
    for (int s = 0; s < tp.K; ++s) {
      mbar_init(full0 + 8 * s, 33);  // producer lane 0's arrive.expect_tx + every producer lane
      mbar_init(empty0 + 8 * s, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    const bits* cosb = static_cast<const bits*>(p.cos);
    const bits* sinb = static_cast<const bits*>(p.sin);
    bool timed_out = false;
    int64_t j = 0;
    int64_t t = blockIdx.x;
    TilePos<MODE> cur{};
    if (t < tp.ntiles) cur = load_tile_pos<MODE>(p, tile_of<RANK4>(p, tp, t), lane);
    for (; t < tp.ntiles; t += gridDim.x, ++j) {
      const int s = (int)(j % tp.K);
      const int64_t r = j / tp.K;
      TilePos<MODE> nxt{};
      if (t + gridDim.x < tp.ntiles)
        nxt = load_tile_pos<MODE>(p, tile_of<RANK4>(p, tp, t + gridDim.x), lane);
      if (r > 0 && !mbar_wait(empty0 + 8 * s, (uint32_t)((r - 1) & 1))) {
        timed_out = true;
        break;
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
      if (lane < tp.TS) reinterpret_cast<uint32_t*>(st + tp.flag_off)[lane] = flags;
      if (lane == 0) {
        mbar_arrive_expect_tx(full0 + 8 * s, tp.x_bytes);
        tma_load_x<RANK4>(st_addr, &tmx, tl.c, full0 + 8 * s, pol);
      }
      // The tile's cos/sin rows (layout [token][slot][cos|sin][rd/2]) are
      // gathered with coalesced 16-byte loads from the L2-resident tables:
      // many small bulk copies would queue behind the tile copies in the
      // SM's TMA unit. Piece c of the block is 16 bytes at byte offset 16*c.
      const int ch = (int)(row_bytes / 16);
      const int per_tok = SLOTS * 2 * ch;
      const int pieces = tl.ntok * per_tok;
      for (int base = 0; base < pieces; base += 32 * 8) {
        uint4 v[8];
        bool okv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = base + u * 32 + lane;
          const int cl = c < pieces ? c : 0;
          const int lt = cl / per_tok;
          const int rem = cl - lt * per_tok;
          const int k = rem / (2 * ch);
          const int rem2 = rem - k * 2 * ch;
          const int cs = rem2 / ch;
          const int piece = rem2 - cs * ch;
          const uint32_t fl = __shfl_sync(0xffffffffu, flags, lt);
          int64_t row;
          if (MODE == Coef::kCache3D) {
            row = tl.tok0 + lt;
          } else {
            const int64_t p0 = __shfl_sync(0xffffffffu, cur.v[0], lt);
            row = p0;
            if (MODE == Coef::kMRope) {
              const int64_t p1 = __shfl_sync(0xffffffffu, cur.v[SLOTS > 1 ? 1 : 0], lt);
              const int64_t p2 = __shfl_sync(0xffffffffu, cur.v[SLOTS > 2 ? 2 : 0], lt);
              row = k == 0 ? p0 : (k == 1 ? p1 : p2);
            }
          }
          okv[u] = c < pieces && ((fl >> k) & 1u);
          if (okv[u]) v[u] = __ldg(reinterpret_cast<const uint4*>((cs ? sinb : cosb) + row * p.h) + piece);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (okv[u]) reinterpret_cast<uint4*>(st + tp.coef_off)[base + u * 32 + lane] = v[u];
      }
      mbar_arrive(full0 + 8 * s);  // each lane releases its own stores
      cur = nxt;
    }
    // Leave only after every load this warp issued has landed.
    const int64_t issued = j;
    for (int64_t q = issued - tp.K > 0 ? issued - tp.K : 0; q < issued; ++q) {
      const int s = (int)(q % tp.K);
      if (!mbar_wait(full0 + 8 * s, (uint32_t)((q / tp.K) & 1))) timed_out = true;
    }
    if (timed_out && lane == 0 && p.oor_flag) atomicOr(p.oor_flag, 2);
    return;
  }

  // -------------------------------------------------------------- consumers
  // Thread q owns pair unit k of rows r0, r0 + rpp, ... (at most RU rows of a
  // tile; the host sizes tiles so). The rows' (token, head) coordinates are
  // the same for every tile, so they are worked out once.
  constexpr int RU = MODE == Coef::kMRope ? 2 : 4;
  const int q = threadIdx.x - 32;
  const int nP = p.nP;
  const int k = q % nP;
  const int r0 = q / nP;
  const int rpp = kTmaConsumers / nP;
  const int nrows = tp.TS * tp.NG;
  int row_ts[RU], row_ng[RU];
  bool row_in[RU];
#pragma unroll
  for (int u = 0; u < RU; ++u) {
    const int r = r0 + u * rpp;
    row_in[u] = r0 < rpp && r < nrows;
    row_ts[u] = RANK4 ? r % tp.TS : r / tp.NG;
    row_ng[u] = RANK4 ? r / tp.TS : r % tp.NG;
  }
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
  const uint64_t pol = policy_evict_first();
  bool timed_out = false;
  int64_t j = 0;
  for (int64_t t = blockIdx.x; t < tp.ntiles; t += gridDim.x, ++j) {
    const int s = (int)(j % tp.K);
    const bool ok = mbar_wait(full0 + 8 * s, (uint32_t)((j / tp.K) & 1));
    if (consumer_any(!ok)) {
      timed_out = true;
      break;
    }
    const Tile tl = tile_of<RANK4>(p, tp, t);
    unsigned char* st = stage0 + (size_t)s * tp.stage_bytes;
    const uint32_t* sflags = reinterpret_cast<const uint32_t*>(st + tp.flag_off);
    const bits* scoef = reinterpret_cast<const bits*>(st + tp.coef_off);
    bits* sx = reinterpret_cast<bits*>(st);
    bool act[RU];
    uint32_t fl[RU];
    VT a[RU], bv[RU];
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      act[u] = row_in[u] && row_ts[u] < tl.ntok && tl.n0 + row_ng[u] < p.N;
      fl[u] = act[u] ? sflags[row_ts[u]] : 0u;
      if (MODE != Coef::kMRope) act[u] = act[u] && (fl[u] & 1u);  // out of range: row stays as loaded
      if (act[u]) {
        const bits* row = sx + (size_t)(r0 + u * rpp) * p.H;
        a[u] = *reinterpret_cast<const VT*>(row + oa);
        bv[u] = *reinterpret_cast<const VT*>(row + ob);
      }
    }
    if (MODE != Coef::kMRope) {
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        if (act[u]) {
          const bits* cr = scoef + (size_t)row_ts[u] * 2 * p.h;
          const VT c = *reinterpret_cast<const VT*>(cr + oc);
          const VT sn = *reinterpret_cast<const VT*>(cr + p.h + oc);
          VT ya, yb;
          rotate_unit<T, V, INTER>(a[u], bv[u], c, sn, ya, yb);
          bits* row = sx + (size_t)(r0 + u * rpp) * p.H;
          *reinterpret_cast<VT*>(row + oa) = ya;
          *reinterpret_cast<VT*>(row + ob) = yb;
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        if (!act[u]) continue;
        const bits* cr = scoef + (size_t)row_ts[u] * 3 * 2 * p.h;
        const uint32_t valid = fl[u] & present;
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
        VT ya, yb;
        if (valid == present) {
          VT c = merge3(cs[0], cs[1], cs[2], m0, m1);
          VT sn = merge3(ss[0], ss[1], ss[2], m0, m1);
          if (!p.scale_is_one) {
            scale_round<T, V>(c, p.scale);
            scale_round<T, V>(sn, p.scale);
          }
          rotate_unit<T, V, INTER>(a[u], bv[u], c, sn, ya, yb);
        } else {
          mrope_unit_general<T, V, INTER>(a[u], bv[u], cs, ss, um, valid, !p.scale_is_one, p.scale, ya, yb);
        }
        bits* row = sx + (size_t)(r0 + u * rpp) * p.H;
        *reinterpret_cast<VT*>(row + oa) = ya;
        *reinterpret_cast<VT*>(row + ob) = yb;
      }
    }
    fence_async_smem();
    consumer_sync();
    if (q == 0) {
      tma_store_y<RANK4>(&tmy, tl.c, smem_addr(st), pol);
      bulk_commit();
      bulk_wait_read_1();  // the previous tile's store has read its stage
      if (j > 0) mbar_arrive(empty0 + 8 * ((j - 1) % tp.K));
    }
  }
  if (q == 0) bulk_wait_all();
  if (timed_out && q == 0 && p.oor_flag) atomicOr(p.oor_flag, 2);
}

}  // namespace rope_gb300
