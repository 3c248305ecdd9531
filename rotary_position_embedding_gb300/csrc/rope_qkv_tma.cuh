// TMA-pipelined Q/K rotation with the key/value cache append (and the
// optional QK-RMSNorm) for sm_103a.
//
// The same operation as rope_qkv_kernel (rope_qkv.cuh) -- every Q and K head
// rotated as RotaryEmbedding (or, in the MROPE instances, MRotaryEmbedding)
// rotates one head of a rank-3 X, V copied, K and V appended to the caches at
// rows past[b] + s -- with the bytes in flight held in shared memory instead
// of registers, as in rope_tma_kernel. A tile is NG heads of one role (Q, K or
// V) times TS consecutive tokens of one batch; RoPE gives every role the same
// TS x NG, M-RoPE gives each role its own (host-planned, QRole). A Q
// tile (and a K tile without caches) is one tensor box of TS x NG x H, laid
// out in the stage as in the tensor and stored to q_out (k_out) as one box; a
// cache tile is NG per-head boxes of TS x H, which are exactly TS consecutive
// rows of one head of a (B, Nkv, max_len, H) cache.
//   copy warp  (lane 0) starts a tile's tensor copies into a free stage and
//              writes the finished tile back with tensor stores;
//   gather warp loads the tile's positions (a tile ahead) and gathers its
//              cos/sin rows (Q and K tiles): one bulk copy per row for RoPE,
//              16-byte asynchronous copies for M-RoPE's three rows per token;
//   consumers  normalise (RMSNorm) and rotate Q and K tiles in place; V tiles
//              pass through untouched.
// A cache tile that is ragged (the batch's last, partial token tile) or whose
// rows leave [0, max_len) is not given to the tensor store -- a store must
// neither write rows past the batch's new tokens nor start at a negative row
// -- but stored row by row by the consumers, which skip rows outside the cache
// (status bit 2). Barrier protocol, bounded waits and the exit on a timeout
// are those of rope_tma_kernel (rope_tma.cuh): a ring of 2K landed barriers
// for the tile copies, full[s] for the gather lanes. Here the gather's RoPE
// rows are bulk copies that complete on full[s], so a gather warp that gives
// up also waits (bounded) for the full phases of the tiles it has served.
//
// Definitions followed (web pages, by title and section):
//  - "com.microsoft.SparseAttention" README: Description, Inputs (query or
//    packed [Q|K|V], key, value, past_key / past_value updated in place),
//    Attributes (do_rotary, kv_num_heads, rotary_interleaved).
//  - onnxruntime pull request "Add RotaryEmbedding fusion for Qwen3 on-the-fly
//    RoPE patterns": Verification and Qwen3 Architecture (RoPE on Q and K; GQA;
//    QK-Norm: RMSNorm on Q and K before RoPE).
//  - "com.microsoft.MRotaryEmbedding" README: Description, Inputs/positionIds
//    (t, h, w streams), Attributes (mrope_section, mrope_layout, scale).
#pragma once

#include "rope_packed.cuh"
#include "rope_qkv.cuh"
#include "rope_tma.cuh"

namespace rope_gb300 {

// Bulk copy global -> shared on the TMA unit (no tensor map): `bytes` (a
// multiple of 16, both addresses 16-byte aligned) completing as transaction
// bytes on the mbarrier `bar`. The gather warp copies each cos/sin row of a
// tile this way: one instruction per row instead of one per 16 bytes (the
// RoPE pipeline keeps 16-byte copies, whose small rows would otherwise queue
// behind its tile copies on the TMA unit; measured slower there).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed,
// counted as a pending arrival of its own: the barrier's phase waits for it
// without it taking one of the expected arrivals.
__device__ __forceinline__ void cp_async_arrive_pending(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Pipelines per CTA. With two, a CTA holds two independent copies of the
// pipeline (copy warp, gather warp, 8 consumers, K stages) whose warps
// interleave (even warps pipeline 0, odd warps pipeline 1), in place of two
// CTAs per SM. Two resident CTAs do not progress alike: the one launched first
// refills its stages faster, and the other finishes last. For M-RoPE the
// single two-pipeline CTA measured faster (44.6 against 46.0 us on the
// M-RoPE QK-Norm prefill), for RoPE slower (37.7 against 36.1 us with the norm).
#ifndef ROPE_QKV_TMA_PIPES
#define ROPE_QKV_TMA_PIPES 1
#endif
#ifndef ROPE_QKV_TMA_MROPE_PIPES
#define ROPE_QKV_TMA_MROPE_PIPES 2
#endif
__host__ __device__ constexpr int qkv_pipes(bool mrope) { return mrope ? ROPE_QKV_TMA_MROPE_PIPES : ROPE_QKV_TMA_PIPES; }

// Heads a consumer thread loads and reduces together.
#ifndef ROPE_QKV_TMA_HEAD_BATCH
#define ROPE_QKV_TMA_HEAD_BATCH 2
#endif

// Division of x < 2^31 by a divisor d fixed at planning time, as a multiply
// and a shift: with l = ceil(log2 d) and m = ceil(2^(31+l) / d) (m < 2^32),
// floor(x * m / 2^(31+l)) = floor(x / d) because the error x*(m*d - 2^(31+l))
// / (d * 2^(31+l)) stays below 1/d (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994).
struct Div {
  uint32_t m;
  int32_t shift;  // 31 + l
};
__device__ __forceinline__ uint32_t div_by(uint32_t x, Div d) {
  return (uint32_t)(((uint64_t)x * d.m) >> d.shift);
}

// Tile geometry of one role (Q, K or V): TS tokens x NG heads (host-planned).
struct QRole {
  int32_t TS, NG;         // tokens and heads per tile
  int32_t G;              // head groups of the role: its heads / NG
  int32_t s_tiles;        // ceil(S / TS)
  int32_t nt_tiles;       // token tiles: B * s_tiles
  int32_t head_off;       // source head of the role's head 0 (packed: 0, Nq, Nq + Nkv)
  uint32_t blk_bytes;     // cache tiles: one head's TS x H block in a stage (a multiple of 128 bytes)
  uint32_t x_bytes;       // transaction bytes of a tile
  uint32_t coef_off;      // stage offset of the tile's cos/sin rows (after its NG blocks)
  int64_t first;          // index of the role's first tile (ntiles: the role has none)
  Div by_nt, by_s;        // division by nt_tiles and by s_tiles
  // consumer columns (token, pair unit): TS * nP of them, tpc threads each
  // (cols <= consumers), hpt heads per thread
  int32_t cols, tpc, hpt;
  Div by_cols;
};

// Tile geometry and stage layout of the pipelined Q/K kernel (host-planned).
struct QTParams {
  int32_t K;              // stages
  int32_t nT;             // tail units (H - rd) / V
  int64_t ntiles;
  uint32_t flag_off;      // stage offsets: per-token flags, positions, header
  uint32_t pos_off;       // M-RoPE: the tile's t/h/w positions (gather warp scratch)
  uint32_t hdr_off;
  uint32_t stage_bytes;
  uint32_t bar_bytes;
  Div by_nP;              // division by the pair units per row
  QRole r[3];
};

// Tensor maps: the source of each role (Q, K, V) and its destination (q_out;
// k_out or k_cache; v_cache). Q and K-without-caches boxes are TS x NG heads;
// cache-mode K and V boxes are one head's TS rows.
struct QKVMaps {
  CUtensorMap src[3];
  CUtensorMap dst[3];
};

struct QTile {
  int role;       // 0 Q, 1 K, 2 V
  int n;          // tokens of the tile inside the sequence (the box may run past S)
  int32_t head0;  // first head of the tile within its role
  int32_t s0;     // first token (sequence index)
  int32_t b;
  QRole R;        // the role's geometry
};

__device__ __forceinline__ QRole qrole(const QTParams& tp, int role) {
  return role == 0 ? tp.r[0] : (role == 1 ? tp.r[1] : tp.r[2]);
}

// Tiles are numbered head group by head group (all token tiles of Q group 0,
// then Q group 1, ..., the K groups, the V groups), so the round-robin
// schedule deals every CTA the same mix of Q, K and V tiles -- which differ in
// cost: V tiles gather and compute nothing -- and the tiles left over after
// the last full round are the cheap V tiles.
// UNIFORM: every role has the same TS and NG (the RoPE path), so those come
// from role 0 and only the role's first tile and head offset differ.
template <bool UNIFORM>
__device__ __forceinline__ QTile qtile_of(const KParams& p, const QTParams& tp, int64_t t64) {
  QTile q;
  q.role = t64 < tp.r[1].first ? 0 : (t64 < tp.r[2].first ? 1 : 2);
  if (UNIFORM) {
    q.R = tp.r[0];
    q.R.first = q.role == 0 ? 0 : (q.role == 1 ? tp.r[1].first : tp.r[2].first);
    q.R.head_off = q.role == 0 ? tp.r[0].head_off : (q.role == 1 ? tp.r[1].head_off : tp.r[2].head_off);
  } else {
    q.R = qrole(tp, q.role);
  }
  const uint32_t t = (uint32_t)(t64 - q.R.first);  // tile counts stay below 2^31
  const uint32_t g = div_by(t, q.R.by_nt);
  const uint32_t tt = t - g * (uint32_t)q.R.nt_tiles;
  const uint32_t bb = div_by(tt, q.R.by_s);
  const uint32_t st = tt - bb * (uint32_t)q.R.s_tiles;
  q.b = (int32_t)bb;
  q.s0 = (int32_t)(st * (uint32_t)q.R.TS);
  const int64_t left = p.S - q.s0;
  q.n = (int)(left < q.R.TS ? left : q.R.TS);
  q.head0 = (int32_t)g * q.R.NG;
  return q;
}

// Q tiles and (without caches) K tiles are one NG-head box in the stage,
// laid out [TS][NG][H] like the tensor; cache tiles are NG per-head blocks of
// TS x H, the rows of the cache.
__device__ __forceinline__ bool qtile_wide(const QKVParams& a, const QTile& q) {
  return q.role == 0 || !a.cache;
}

// Whether a cache tile goes out row by row from the consumers instead of by
// tensor store: ragged, or not entirely inside [0, max_len).
__device__ __forceinline__ bool qtile_direct(const QKVParams& a, const QTile& q, int64_t row0) {
  return q.role != 0 && a.cache && (q.n < q.R.TS || row0 < 0 || row0 + q.R.TS > a.max_len);
}

template <class T, bool INTER, bool IMPLICIT, bool NORM, bool MROPE = false>
__global__ void __launch_bounds__(kTmaThreads * qkv_pipes(MROPE), ROPE_TMA_MIN_CTAS / qkv_pipes(MROPE))
    rope_qkv_tma_kernel(const KParams p, const QKVParams a, const QTParams tp,
                        const __grid_constant__ QKVMaps maps) {
  using E = Elem<T>;
  using bits = typename E::bits;
  constexpr int V = 16 / sizeof(bits);
  using VT = VecT<T, V>;

  constexpr int kQkvPipes = qkv_pipes(MROPE);
  extern __shared__ __align__(1024) unsigned char smem_all[];
  // this thread's pipeline: its shared memory, and its index among all
  // pipelines (vb of vg), which the schedule uses as a CTA index
  const int pipe = (int)(threadIdx.x >> 5) % kQkvPipes;
  const int warp = (int)(threadIdx.x >> 5) / kQkvPipes;
  const int lane = threadIdx.x & 31;
  unsigned char* smem = smem_all + (size_t)pipe * (tp.bar_bytes + (size_t)tp.K * tp.stage_bytes);
  const int64_t vb = (int64_t)blockIdx.x * kQkvPipes + pipe;
  const int64_t vg = (int64_t)gridDim.x * kQkvPipes;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase;                // full[s]      at 8*s
  const uint32_t done0 = sbase + 8 * tp.K;     // computed[s]  at 8*(K+s)
  const uint32_t issued0 = sbase + 16 * tp.K;  // issued[s]    at 8*(2K+s)
  const uint32_t landed0 = sbase + 24 * tp.K;  // landed[b]    at 8*(3K+b), b < 2K
  // tile jj's landed barrier and the parity of its phase there (see rope_tma.cuh)
  auto landed_bar = [&](int64_t jj) -> uint32_t { return landed0 + 8 * (uint32_t)(jj % (2 * tp.K)); };
  auto landed_par = [&](int64_t jj) -> uint32_t { return (uint32_t)((jj / (2 * tp.K)) & 1); };
  unsigned char* stage0 = smem + tp.bar_bytes;
  const int H = (int)p.H;
  const int h = p.h;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < tp.K; ++s) {
      mbar_init(full0 + 8 * s, 32);  // every gather lane
      mbar_init(done0 + 8 * s, kTmaConsumerWarps);
      mbar_init(issued0 + 8 * s, 1);
      mbar_init(landed0 + 8 * s, 1);  // the tile copies' arrive.expect_tx (two per stage)
      mbar_init(landed0 + 8 * (tp.K + s), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.src[r])) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.dst[r])) : "memory");
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  // stage header: [0] the tile index (copy warp), [1] a cache tile's first row (gather warp)
  auto stage_hdr = [&](int s) -> int64_t* {
    return reinterpret_cast<int64_t*>(stage0 + (size_t)s * tp.stage_bytes + tp.hdr_off);
  };

  if (warp == 0) {
    // --------------------------------------------------- copy warp (lane 0)
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      bool timed_out = false;
      // Tile indices: vb + jj*vg (static schedule), or -- with
      // a caller scratch counter -- the next value of the counter, so CTAs
      // that run faster take more tiles. Each index is recorded in its stage
      // header; the first index past the last tile (the sentinel) ends the
      // pipeline.
      auto pick = [&](int64_t jj) -> int64_t {
        return p.sched ? (int64_t)atomicAdd(p.sched, 1ull) : vb + jj * vg;
      };
      // stage and landed slot of the next tile issued (jx % K, jx % 2K),
      // stepped per issue (see rope_tma.cuh)
      int is_s = 0, is_l = 0;
      auto issue = [&](int64_t t) {
        const int s = is_s;
        const uint32_t lb = landed0 + 8 * (uint32_t)is_l;
        *stage_hdr(s) = t;
        if (t < tp.ntiles) {
          const QTile q = qtile_of<!MROPE>(p, tp, t);
          const uint32_t dst = smem_addr(stage0 + (size_t)s * tp.stage_bytes);
          mbar_arrive_expect_tx(lb, q.R.x_bytes);
          // one NG-head box, or (cache tiles) one box per head
          const int nbox = qtile_wide(a, q) ? 1 : q.R.NG;
          for (int u = 0; u < nbox; ++u) {
            const int c[4] = {0, q.R.head_off + q.head0 + u, q.s0, q.b};
            tma_load_x<true>(dst + (uint32_t)u * q.R.blk_bytes, &maps.src[q.role], c, lb, pol);
          }
        } else {
          mbar_arrive(lb);  // the sentinel carries no bytes
        }
        mbar_arrive(issued0 + 8 * s);
        if (++is_s == tp.K) is_s = 0;
        if (++is_l == 2 * tp.K) is_l = 0;
      };
      bool ended = false;
      int64_t jx = 0;  // tiles issued (the sentinel included)
      for (; jx < tp.K && !ended; ++jx) {
        const int64_t t = pick(jx);
        issue(t);
        ended = t >= tp.ntiles;
      }
      // the next store's tile and cache row are worked out while the previous
      // store is still reading its stage
      int64_t t_st = *stage_hdr(0);
      QTile q_st{};
      int64_t past_st = 0;  // raw past[b]: the load is consumed only at the store
      auto prep = [&](int64_t t) {
        if (t < tp.ntiles) {
          q_st = qtile_of<!MROPE>(p, tp, t);
          past_st = (q_st.role != 0 && a.cache && a.past) ? (int64_t)__ldg(a.past + q_st.b) : 0;
        }
      };
      prep(t_st);
      int64_t j = 0;  // the tile whose store comes next
      int s = 0;      // its stage (j % K) and the parity of its phase there
      uint32_t ph = 0;
      for (;; ++j) {
        if (!mbar_wait(done0 + 8 * s, ph)) {
          timed_out = true;
          break;
        }
        if (t_st >= tp.ntiles) break;  // sentinel
        const int64_t row_st = past_st + q_st.s0;
        if (!qtile_direct(a, q_st, row_st)) {
          const uint32_t src = smem_addr(stage0 + (size_t)s * tp.stage_bytes);
          const bool to_cache = !qtile_wide(a, q_st);
          for (int u = 0; u < (to_cache ? q_st.R.NG : 1); ++u) {
            int c[4];
            if (to_cache) {
              c[0] = 0, c[1] = (int)row_st, c[2] = q_st.head0 + u, c[3] = q_st.b;
            } else {
              c[0] = 0, c[1] = q_st.head0 + u, c[2] = q_st.s0, c[3] = q_st.b;
            }
            tma_store_y<true>(&maps.dst[q_st.role], c, src + (uint32_t)u * q_st.R.blk_bytes, pol);
          }
          bulk_commit();
        }
        const int64_t t_new = ended ? 0 : pick(jx);
        if (++s == tp.K) {
          s = 0;
          ph ^= 1u;
        }
        // tile j+1 is already issued (K >= 2), so its header is in place
        t_st = *stage_hdr(s);
        prep(t_st);
        if (!ended) {
          bulk_wait_read_0();  // the stage may be refilled once the store has read it
          issue(t_new);        // jx == j + K: the tile that goes into tile j's stage next
          ended = t_new >= tp.ntiles;
          ++jx;
        }
      }
      bulk_wait_all();
      if (timed_out) {
        // tiles j .. jx-1 were started and never stored: their loads land
        // before the CTA's shared memory goes away (see rope_tma.cuh)
        for (int64_t jj = j; jj < jx; ++jj) (void)mbar_wait(landed_bar(jj), landed_par(jj));
        if (p.oor_flag) atomicOr(p.oor_flag, 2);
      }
      if (p.sched) {
        // The last CTA to stop drawing resets the counter pair for the next launch.
        __threadfence();
        if (atomicAdd(p.sched + 1, 1ull) == (unsigned long long)vg - 1) {
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
    // Per Q or K tile: the tokens' positions (explicit, or past[b] + s; M-RoPE:
    // t, h, w) and range flags, then the cos/sin rows ([token][stream][cos|sin]
    // [rd/2]); the copies arrive on full[s] when they land. V tiles gather
    // nothing. Cache tiles also get their first row in the header.
    const bits* cosb = static_cast<const bits*>(p.cos);
    const bits* sinb = static_cast<const bits*>(p.sin);
    bool timed_out = false;
    // RoPE: row r of a tile's coefficient block (the cos or sin row of token
    // r / 2, row_bytes at byte r*row_bytes) goes to lane r % 32 as one bulk
    // copy. M-RoPE: 16-byte pieces, piece c by lane c % 32 (below).
    const uint32_t row_bytes = (uint32_t)h * (uint32_t)sizeof(bits);
    constexpr int SLOTS = MROPE ? 3 : 1;  // coefficient rows per token: one per position stream
    // M-RoPE: the streams some coefficient index uses (an unused stream's
    // position never matters, nor does it flag anything)
    uint32_t used = 1u;
    if (MROPE) {
      used = 0u;
      for (int i = 0; i < h; ++i) used |= 1u << ((p.smap[i >> 4] >> ((i & 15) * 2)) & 3u);
    }
    // M-RoPE: 16-byte pieces per row, and this lane's first piece and stride
    const int ch = (int)(row_bytes / 16);
    const int r_first = lane / ch, pc_first = lane % ch;
    const int r_step = 32 / ch, pc_step = 32 % ch;
    // What a tile needs from global memory -- its positions, or the past
    // length its positions and cache rows start from -- is loaded one tile
    // ahead: under a saturated memory system even these L2 hits take
    // microseconds, and the gather of the tile waits on none.
    struct Pre {
      int64_t pos[SLOTS];  // explicit position(s) of token `lane` (M-RoPE: t, h, w)
      int64_t past;        // past[b]
    };
    auto prefetch = [&](int64_t t) -> Pre {
      Pre r{};
      if (t < tp.ntiles) {
        const QTile q = qtile_of<!MROPE>(p, tp, t);
        if (a.past && (IMPLICIT || (q.role != 0 && a.cache))) r.past = (int64_t)__ldg(a.past + q.b);
        if (!IMPLICIT && q.role != 2 && lane < q.n) {
          const int64_t tok = (int64_t)q.b * p.S + q.s0 + lane;
#pragma unroll
          for (int k = 0; k < SLOTS; ++k) r.pos[k] = __ldg(p.pos + k * p.ntok + tok);
        }
      }
      return r;
    };
    // Dynamic schedule: the next index is read from its stage header when the
    // copy warp has already published it; otherwise the tile's own values are
    // loaded when it comes up.
    Pre cur{};
    bool have_cur = false;
    if (!p.sched) {
      cur = prefetch(vb);
      have_cur = true;
    }
    int64_t j = 0;  // the tile served next
    int s = 0;      // its stage (j % K) and the parity of its phase there
    uint32_t ph = 0;
    for (;; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(issued0 + 8 * s, ph))) {
        timed_out = true;
        break;
      }
      const int64_t t = *stage_hdr(s);
      if (t >= tp.ntiles) {
        cp_async_arrive(full0 + 8 * s);
        break;
      }
      if (!have_cur) cur = prefetch(t);
      // the stage and parity of tile j+1
      const int sn = s + 1 == tp.K ? 0 : s + 1;
      const uint32_t phn = s + 1 == tp.K ? ph ^ 1u : ph;
      Pre nxt{};
      bool have_nxt = false;
      if (!p.sched) {
        nxt = prefetch(t + vg);  // this pipeline's next tile
        have_nxt = true;
      } else {
        // headers are published in tile order and tile j+1-K's phase of this
        // barrier is already complete, so the parity test cannot alias
        if (__all_sync(0xffffffffu, mbar_test(issued0 + 8 * sn, phn))) {
          nxt = prefetch(*stage_hdr(sn));
          have_nxt = true;
        }
      }
      const QTile q = qtile_of<!MROPE>(p, tp, t);
      unsigned char* st = stage0 + (size_t)s * tp.stage_bytes;
      if (q.role != 0 && a.cache && lane == 0) stage_hdr(s)[1] = cur.past + q.s0;
      if (q.role != 2) {
        int64_t pp[SLOTS];
        uint32_t flag = 0;  // bit k: stream k's position is inside the table
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) pp[k] = -1;
        if (lane < q.n) {
#pragma unroll
          for (int k = 0; k < SLOTS; ++k) {
            pp[k] = MROPE ? cur.pos[k] : (IMPLICIT ? cur.past + q.s0 + lane : cur.pos[0]);
            if ((uint64_t)pp[k] < (uint64_t)p.cache_rows) flag |= 1u << k;
          }
          if ((flag & used) != used && q.role == 0 && q.head0 == 0 && p.oor_flag) atomicOr(p.oor_flag, 1);
        }
        if (lane < q.R.TS) reinterpret_cast<uint32_t*>(st + tp.flag_off)[lane] = flag;
        const uint32_t coef_addr = smem_addr(st) + q.R.coef_off;
        if (MROPE) {
          // Three rows per token: one bulk copy per row would queue 6 TS
          // requests on the SM's copy engine behind the tile loads, so the
          // rows go as 16-byte asynchronous copies through the load path,
          // piece c of the block (row c / ch, piece c % ch) by lane c % 32.
          // Positions go through the stage so that any lane can read any
          // token's.
          if (lane < q.R.TS) {
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) reinterpret_cast<int64_t*>(st + tp.pos_off)[lane * SLOTS + k] = pp[k];
          }
          __syncwarp();  // positions and flags, before the lanes read them
          const int64_t* pv = reinterpret_cast<const int64_t*>(st + tp.pos_off);
          const uint32_t* fv = reinterpret_cast<const uint32_t*>(st + tp.flag_off);
          const int lim = q.n * (2 * SLOTS);  // rows of the tile's tokens
          int r = r_first, pc = pc_first;
          while (r < lim) {
            const int lt = r / (2 * SLOTS);
            const int k = (r >> 1) % SLOTS;
            if ((fv[lt] >> k) & 1u)
              cp_async16(coef_addr + 16u * (uint32_t)(r * ch + pc),
                         reinterpret_cast<const uint4*>(((r & 1) ? sinb : cosb) + pv[lt * SLOTS + k] * h) + pc);
            r += r_step;
            pc += pc_step;
            if (pc >= ch) {
              pc -= ch;
              ++r;
            }
          }
          // the copies' arrival is pending on full[s] until they land; the
          // plain arrival releases the flags, positions and header
          cp_async_arrive_pending(full0 + 8 * s);
          mbar_arrive(full0 + 8 * s);
        } else {
          const int rows = q.R.TS * SLOTS * 2;
          const int rounds = (rows + 31) / 32;  // the same for every lane: the shuffles below are warp-wide
          const bits* src[kMaxGather];
          uint32_t bytes = 0, go = 0;
#pragma unroll
          for (int g = 0; g < kMaxGather; ++g) {
            if (g >= rounds) break;
            // row r: token r / (2*SLOTS), stream (r / 2) % SLOTS, cos or sin (r % 2)
            const int r = lane + 32 * g;
            const int lt = r < rows ? r / (2 * SLOTS) : 0;
            const int k = (r >> 1) % SLOTS;
            // token lt's positions live in lane lt
            int64_t row = __shfl_sync(0xffffffffu, pp[0], lt);
#pragma unroll
            for (int kk = 1; kk < SLOTS; ++kk) {
              const int64_t other = __shfl_sync(0xffffffffu, pp[kk], lt);
              if (k == kk) row = other;
            }
            const uint32_t ok = (__shfl_sync(0xffffffffu, flag, lt) >> k) & 1u;
            src[g] = ((r & 1) ? sinb : cosb) + row * h;
            if (r < rows && ok) {
              bytes += row_bytes;
              go |= 1u << g;
            }
          }
          __syncwarp();  // flags and the header precede the lanes' (releasing) arrivals
          // this lane's arrival carries the bytes its copies will complete
          mbar_arrive_expect_tx(full0 + 8 * s, bytes);
#pragma unroll
          for (int g = 0; g < kMaxGather; ++g)
            if ((go >> g) & 1u) bulk_g2s(coef_addr + row_bytes * (uint32_t)(lane + 32 * g), src[g], row_bytes,
                                         full0 + 8 * s);
        }
      } else {
        __syncwarp();  // the header precedes the lanes' (releasing) arrivals
        mbar_arrive(full0 + 8 * s);
      }
      cur = nxt;
      have_cur = have_nxt;
      s = sn;
      ph = phn;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (timed_out) {
      // The bulk copies of the last K tiles served may still be landing; each
      // such tile's full phase has every lane's arrival, so it completes when
      // they land (its next phase needs this warp's arrival for tile jj + K,
      // never made: the parity wait cannot alias).
      for (int64_t jj = j > tp.K ? j - tp.K : 0; jj < j; ++jj)
        (void)mbar_wait(full0 + 8 * (int)(jj % tp.K), (uint32_t)((jj / tp.K) & 1));
      if (lane == 0 && p.oor_flag) atomicOr(p.oor_flag, 2);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Thread q owns column (token ts, pair unit k) of the tile for heads
  // hq, hq + tpc, ...; with RMSNorm the nP threads of one (token, head) row
  // are an aligned lane group that adds up the row's squares with shuffles.
  // A role's TS x nP columns are a multiple of nP, so the unit k is the same
  // in every role's layout; ts and hq follow the tile's role.
  const int qi = (warp - kTmaRoleWarps) * 32 + lane;
  const int nP = p.nP;
  const int k = qi - nP * (int)div_by((uint32_t)qi, tp.by_nP);
  int oa, ob;
  unit_offsets<V, INTER>(k, h, oa, ob);
  const int oc = k * V;
  // the column of role r's tiles (once for all roles when they share a shape)
  int cols = 0, tpc = 0, hpt = 0, hq = 0, ts = 0;
  bool has_col = false;
  uint32_t blk_elems = 0;
  auto columns = [&](const QRole& R) {
    cols = R.cols;
    tpc = R.tpc;
    hpt = R.hpt;  // the same for every thread
    hq = (int)div_by((uint32_t)qi, R.by_cols);
    has_col = hq < tpc;
    ts = (int)div_by((uint32_t)(qi - hq * cols), tp.by_nP);
    blk_elems = R.blk_bytes / (uint32_t)sizeof(bits);
  };
  if (!MROPE) columns(tp.r[0]);
  // M-RoPE: the stream of each of the unit's V coefficient indices, and the
  // masks that merge the three gathered rows word by word
  uint32_t um = 0, present = 0;
  uint32_t m0[4] = {0, 0, 0, 0}, m1[4] = {0, 0, 0, 0};
  if (MROPE) {
    const uint32_t word = p.smap[oc >> 4];
    um = (word >> ((oc & 15) * 2)) & (uint32_t)((1ull << (2 * V)) - 1);
#pragma unroll
    for (int jj = 0; jj < V; ++jj) present |= 1u << ((um >> (2 * jj)) & 3);
    stream_masks<V>(um, m0, m1);
  }
  // mean of a head's squares: for a power-of-two H the product with 1/H is the
  // same correctly rounded value as the quotient, without the division
  const bool h_pow2 = (H & (H - 1)) == 0;
  const float inv_h = 1.0f / (float)H;
  auto mean_sq = [&](float ss) -> float { return h_pow2 ? ss * inv_h : ss / (float)H; };
  bool timed_out = false;
  // tile j's stage s and full parity, landed slot and parity (j % K,
  // (j / K) & 1, j % 2K, (j / 2K) & 1), stepped once per tile
  int s = 0, lsl = 0;
  uint32_t ph = 0, lph = 0;
  for (;;) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(landed0 + 8 * (uint32_t)lsl, lph) &&
                                                mbar_wait(full0 + 8 * s, ph));
    const int64_t t = ok ? *stage_hdr(s) : 0;
    if (ok && t >= tp.ntiles) {
      __syncwarp();
      if (lane == 0) mbar_arrive(done0 + 8 * s);
      break;
    }
    if (!ok) {
      timed_out = true;
      break;
    }
    const QTile q = qtile_of<!MROPE>(p, tp, t);
    if (MROPE) columns(q.R);
    unsigned char* st = stage0 + (size_t)s * tp.stage_bytes;
    bits* sx = reinterpret_cast<bits*>(st);
    const bool tok_in = ts < q.n;
    const bool wide = qtile_wide(a, q);
    if (q.role != 2) {
      const uint32_t fl = reinterpret_cast<const uint32_t*>(st + tp.flag_off)[ts];
      // M-RoPE rotates every token and puts back the pairs of out-of-range streams
      const bool valid = tok_in && (MROPE || (fl & 1u));
      VT c{}, sn{};
      bool blend_on = false;
      uint32_t ma[4] = {0, 0, 0, 0}, mb[4] = {0, 0, 0, 0};
      if (valid) {
        if (MROPE) {
          const bits* cr = reinterpret_cast<const bits*>(st + q.R.coef_off) + (size_t)ts * 3 * 2 * h;
          const uint32_t vmask = fl & present;
          VT cs[3], ss[3];
#pragma unroll
          for (int k3 = 0; k3 < 3; ++k3) {
            cs[k3] = VT{};
            ss[k3] = VT{};
            if ((vmask >> k3) & 1u) {
              cs[k3] = *reinterpret_cast<const VT*>(cr + (size_t)k3 * 2 * h + oc);
              ss[k3] = *reinterpret_cast<const VT*>(cr + (size_t)k3 * 2 * h + h + oc);
            }
          }
          c = merge3(cs[0], cs[1], cs[2], m0, m1);
          sn = merge3(ss[0], ss[1], ss[2], m0, m1);
          if (!p.scale_is_one) {
            scale_round<T, V>(c, p.scale);
            scale_round<T, V>(sn, p.scale);
          }
          blend_on = vmask != present;
          if (blend_on) pair_masks<V, INTER>(um, vmask, ma, mb);
        } else {
          const bits* cr = reinterpret_cast<const bits*>(st + q.R.coef_off) + (size_t)ts * 2 * h;
          c = *reinterpret_cast<const VT*>(cr + oc);
          sn = *reinterpret_cast<const VT*>(cr + h + oc);
        }
      }
      constexpr bool PACKED = sizeof(bits) == 2;  // float16 / bfloat16: packed arithmetic
      VT wa{}, wb{};
      if (NORM && has_col) {  // rd == H with the norm: the nP units cover the whole head
        const bits* w = static_cast<const bits*>(q.role == 0 ? a.qw : a.kw);
        wa = ld_shared_ro(reinterpret_cast<const VT*>(w + oa));
        wb = ld_shared_ro(reinterpret_cast<const VT*>(w + ob));
      }
      float2 cf[4], sf[4];  // the column's coefficients, unpacked once per tile (packed path)
      if constexpr (PACKED) {
        Unit8<T> cu, su;
        __builtin_memcpy(&cu, &c, 16);
        __builtin_memcpy(&su, &sn, 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          cf[k] = P2<T>::tof(cu.w[k]);
          sf[k] = P2<T>::tof(su.w[k]);
        }
      }
      // A thread's heads go through in batches of HB: a batch's rows are
      // loaded together and reduced together, so their latencies overlap.
      constexpr int HB = ROPE_QKV_TMA_HEAD_BATCH;
      for (int u0 = 0; u0 < hpt; u0 += HB) {  // hpt is the same for every lane
        bool act[HB];
        uint32_t ro[HB];
        VT xa[HB], xb[HB];
#pragma unroll
        for (int u = 0; u < HB; ++u) {
          const int hh = hq + (u0 + u) * tpc;
          act[u] = u0 + u < hpt && has_col && tok_in && hh < q.R.NG && (NORM || valid);
          ro[u] = wide ? ((uint32_t)ts * (uint32_t)q.R.NG + (uint32_t)hh) * (uint32_t)H
                       : (uint32_t)hh * blk_elems + (uint32_t)ts * (uint32_t)H;
          xa[u] = VT{};
          xb[u] = VT{};
          if (act[u]) {
            xa[u] = *reinterpret_cast<const VT*>(sx + ro[u] + oa);
            xb[u] = *reinterpret_cast<const VT*>(sx + ro[u] + ob);
          }
        }
        if constexpr (PACKED) {
          Unit8<T> ua[HB], ub[HB];
          float2 fa[HB][4], fb[HB][4];
#pragma unroll
          for (int u = 0; u < HB; ++u) {
            __builtin_memcpy(&ua[u], &xa[u], 16);
            __builtin_memcpy(&ub[u], &xb[u], 16);
          }
          float r[HB];
          if (NORM) {
            float ss[HB];
#pragma unroll
            for (int u = 0; u < HB; ++u) {
              // the squares in sum_squares' order: a's eight values, then b's
              float sa = 0.f, sb = 0.f;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                fa[u][k] = P2<T>::tof(ua[u].w[k]);
                fb[u][k] = P2<T>::tof(ub[u].w[k]);
                sa = __fmaf_rn(fa[u][k].x, fa[u][k].x, sa);
                sa = __fmaf_rn(fa[u][k].y, fa[u][k].y, sa);
                sb = __fmaf_rn(fb[u][k].x, fb[u][k].x, sb);
                sb = __fmaf_rn(fb[u][k].y, fb[u][k].y, sb);
              }
              ss[u] = sa + sb;
            }
            for (int o = nP >> 1; o > 0; o >>= 1) {
#pragma unroll
              for (int u = 0; u < HB; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
            }
#pragma unroll
            for (int u = 0; u < HB; ++u) r[u] = 1.0f / sqrtf(mean_sq(ss[u]) + a.eps);
          }
#pragma unroll
          for (int u = 0; u < HB; ++u) {
            if (!act[u]) continue;
            Unit8<T> za = ua[u], zb = ub[u], ya, yb;
            if (NORM) {
              Unit8<T> wua, wub;
              __builtin_memcpy(&wua, &wa, 16);
              __builtin_memcpy(&wub, &wb, 16);
              za = norm8p<T>(fa[u], r[u], wua);
              zb = norm8p<T>(fb[u], r[u], wub);
            }
            if (valid) {
              rotate8p<T, INTER>(za, zb, cf, sf, ya, yb);
              if (MROPE && blend_on) {  // pairs of out-of-range streams keep their input
                VT t0, t1, z0, z1;
                __builtin_memcpy(&t0, &ya, 16);
                __builtin_memcpy(&t1, &yb, 16);
                __builtin_memcpy(&z0, &za, 16);
                __builtin_memcpy(&z1, &zb, 16);
                blend(t0, z0, ma);
                blend(t1, z1, mb);
                __builtin_memcpy(&ya, &t0, 16);
                __builtin_memcpy(&yb, &t1, 16);
              }
            } else {
              ya = za;
              yb = zb;
            }
            *reinterpret_cast<Unit8<T>*>(sx + ro[u] + oa) = ya;
            *reinterpret_cast<Unit8<T>*>(sx + ro[u] + ob) = yb;
          }
        } else {
          float r[HB];
          if (NORM) {
            float ss[HB];
#pragma unroll
            for (int u = 0; u < HB; ++u) ss[u] = sum_squares<T, V>(xa[u]) + sum_squares<T, V>(xb[u]);
            for (int o = nP >> 1; o > 0; o >>= 1) {
#pragma unroll
              for (int u = 0; u < HB; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
            }
#pragma unroll
            for (int u = 0; u < HB; ++u) r[u] = 1.0f / sqrtf(mean_sq(ss[u]) + a.eps);
          }
#pragma unroll
          for (int u = 0; u < HB; ++u) {
            if (!act[u]) continue;
            VT ya, yb;
            VT za = xa[u], zb = xb[u];
            if (NORM) {
              za = norm_weight<T, V>(xa[u], r[u], wa);
              zb = norm_weight<T, V>(xb[u], r[u], wb);
            }
            if (valid) {
              rotate_unit<T, V, INTER>(za, zb, c, sn, ya, yb);
              if (MROPE && blend_on) {  // pairs of out-of-range streams keep their input
                blend(ya, za, ma);
                blend(yb, zb, mb);
              }
            } else {
              ya = za;
              yb = zb;
            }
            *reinterpret_cast<VT*>(sx + ro[u] + oa) = ya;
            *reinterpret_cast<VT*>(sx + ro[u] + ob) = yb;
          }
        }
      }
    }
    if (q.role != 0 && a.cache) {
      const int64_t row0 = stage_hdr(s)[1];
      if (qtile_direct(a, q, row0)) {
        // rows inside the cache, stored by the threads that own them
        if (q.role == 1 && q.head0 == 0 && qi == 0 && (row0 < 0 || row0 + q.n > a.max_len))
          flag_cache_row(p.oor_flag);
        const int64_t r = row0 + ts;
        if (has_col && tok_in && r >= 0 && r < a.max_len) {
          bits* cbase = static_cast<bits*>(q.role == 1 ? a.k_cache : a.v_cache);
          for (int u = 0; u < hpt; ++u) {
            const int hh = hq + u * tpc;
            if (hh >= q.R.NG) break;
            const uint32_t ro = (uint32_t)hh * blk_elems + (uint32_t)ts * (uint32_t)H;
            bits* dr = cbase + (((int64_t)q.b * a.Nkv + q.head0 + hh) * a.max_len + r) * H;
            *reinterpret_cast<VT*>(dr + oa) = *reinterpret_cast<const VT*>(sx + ro + oa);
            *reinterpret_cast<VT*>(dr + ob) = *reinterpret_cast<const VT*>(sx + ro + ob);
            for (int tu = k; tu < tp.nT; tu += nP) {
              const int off = p.rd + tu * V;
              *reinterpret_cast<VT*>(dr + off) = *reinterpret_cast<const VT*>(sx + ro + off);
            }
          }
        }
      }
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
