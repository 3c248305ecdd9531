"""Seeded synthetic inputs for the RoPE / M-RoPE workloads.

This module draws inputs only: activations X, position ids and the inv_freq
parameter vector. It holds none of the operator's arithmetic; the cos/sin
tables are produced by whichever side is under test (the library's
``rope_cache_build`` on the GPU, the oracle's cache build on the CPU). Both
the test suite and ``bench.py`` take their inputs from here, so both sides of
every parity check see identical bytes.

Recipes (one seed per tensor: X seed 0, positions seed 1, out-of-range mask
seed 2):
  X            N(0, 1) drawn in float32, rounded to the storage type.
  RoPE ids     ``pos[b, s] = s + off_b`` with ``off_b ~ U[0, 4096)`` (gather
               workload), or uniform over the cache rows.
  Q/K/V        packed [Q|K|V] activations like X; past lengths
               ``past[b] ~ U[0, max_past]`` (seed 1), positions past[b] + s;
               QK-Norm weights ``U[0.5, 1.5)`` per channel (seed 3).
  M-RoPE ids   per batch: 1024 text tokens (t = h = w), 4 frames of a 32x32
               image grid (t = st + f, h = st + r, w = st + c), 1024 text
               tokens starting at the previous maximum + 1, 2 frames of a
               32x32 grid; a per-batch offset ~ U[0, 16384) on all three
               streams; then 1 % of the 3*B*S ids set past the cache.
  inv_freq     ``base ** (-2 i / d)`` in binary64, rounded to float32 (a model
               parameter, built identically for both sides).
"""

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "rope" | "mrope" | "fused"
    rank: int
    shape: tuple              # X shape
    dtype: str                # "float16" | "float32"
    num_heads: int            # heads N (explicit for rank 4 too)
    interleaved: int = 0
    rotary_embedding_dim: int = 0
    positions: str = "none"   # "none" | "offset" | "uniform" | "mrope"
    cache_rows: int = 0       # rows of the 2-D cache (or S for the 3-D cache)
    rope_base: float = 10000.0
    rope_dim: int = 0         # d in base ** (-2i/d); 0 = rotary dim
    mrope_section: tuple = ()
    mrope_layout: int = 0
    scale: float = 1.0
    attention_scaling: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def head_size(self):
        if self.kind == "qkv":  # packed [Q|K|V] rows: num_heads + 2 * kv_num_heads per token
            return self.shape[2] // (self.num_heads + 2 * self.extra["kv_num_heads"])
        return self.shape[2] // self.num_heads if self.rank == 3 else self.shape[3]

    @property
    def batch(self):
        return self.shape[0]

    @property
    def seq(self):
        return self.shape[1] if self.rank == 3 else self.shape[2]

    @property
    def rotary_dim(self):
        return self.rotary_embedding_dim or self.head_size

    @property
    def half(self):
        return self.rotary_dim // 2

    @property
    def tokens(self):
        return self.batch * self.seq

    @property
    def numel(self):
        return int(np.prod(self.shape))

    def with_shape(self, **kw):
        """Same recipe at another size: keys B, S, N (and H for rank 4)."""
        B = kw.get("B", self.batch)
        S = kw.get("S", self.seq)
        N = kw.get("N", self.num_heads)
        H = kw.get("H", self.head_size)
        shape = (B, S, N * H) if self.rank == 3 else (B, N, S, H)
        d = dict(self.__dict__)
        d.update(shape=shape, num_heads=N, name=self.name + f"@{shape}")
        for k in ("cache_rows", "rotary_embedding_dim", "mrope_section", "scale", "mrope_layout",
                  "interleaved", "dtype", "positions", "attention_scaling"):
            if k in kw:
                d[k] = kw[k]
        return Workload(**d)


# The five workloads. Sizes follow the operator's published configurations;
# the largest of them, the rank-4 interleaved partial rotation (541 MB a
# pass), is the headline benchmark.
WORKLOADS = {
    "rope_r4_f32_cache3d": Workload(
        name="rope_r4_f32_cache3d", kind="rope", rank=4, shape=(1, 2, 8, 16), dtype="float32",
        num_heads=2, interleaved=0, positions="none", cache_rows=8, rope_base=10000.0, rope_dim=16),
    "rope_r3_f16_gather": Workload(
        name="rope_r3_f16_gather", kind="rope", rank=3, shape=(4, 2048, 32 * 128), dtype="float16",
        num_heads=32, interleaved=0, positions="offset", cache_rows=8192, rope_base=10000.0,
        rope_dim=128),
    # the headline shape in bfloat16 (storage beyond the pages' float32/float16)
    "rope_r3_bf16_gather": Workload(
        name="rope_r3_bf16_gather", kind="rope", rank=3, shape=(4, 2048, 32 * 128), dtype="bfloat16",
        num_heads=32, interleaved=0, positions="offset", cache_rows=8192, rope_base=10000.0,
        rope_dim=128),
    "rope_r4_f16_interleaved_partial": Workload(
        name="rope_r4_f16_interleaved_partial", kind="rope", rank=4, shape=(8, 32, 4096, 128),
        dtype="float16", num_heads=32, interleaved=1, rotary_embedding_dim=64, positions="uniform",
        cache_rows=16384, rope_base=10000.0, rope_dim=64),
    "mrope_r3_f16_layout0": Workload(
        name="mrope_r3_f16_layout0", kind="mrope", rank=3, shape=(2, 8192, 28 * 128), dtype="float16",
        num_heads=28, positions="mrope", cache_rows=32768, rope_base=10000.0, rope_dim=128,
        mrope_section=(16, 24, 24), mrope_layout=0, scale=1.0),
    "mrope_r3_f16_layout1": Workload(
        name="mrope_r3_f16_layout1", kind="mrope", rank=3, shape=(2, 8192, 28 * 128), dtype="float16",
        num_heads=28, positions="mrope", cache_rows=32768, rope_base=10000.0, rope_dim=128,
        mrope_section=(16, 24, 24), mrope_layout=1, scale=1.0),
    # Q/K rotation with the key/value cache append, Qwen3-8B attention shape
    # (32 query heads, 8 key/value heads, head size 128), packed [Q|K|V] input,
    # positions past[b] + s: a chunked prefill and a decode step.
    "qkv_prefill_r3_f16": Workload(
        name="qkv_prefill_r3_f16", kind="qkv", rank=3, shape=(4, 2048, (32 + 2 * 8) * 128), dtype="float16",
        num_heads=32, positions="past", cache_rows=8192, rope_base=1.0e6, rope_dim=128,
        extra={"kv_num_heads": 8, "max_len": 4096, "max_past": 2048}),
    # the same prefill with Qwen3's QK-Norm (RMSNorm of every Q and K head) first
    "qkv_norm_prefill_r3_f16": Workload(
        name="qkv_norm_prefill_r3_f16", kind="qkv", rank=3, shape=(4, 2048, (32 + 2 * 8) * 128),
        dtype="float16", num_heads=32, positions="past", cache_rows=8192, rope_base=1.0e6, rope_dim=128,
        extra={"kv_num_heads": 8, "max_len": 4096, "max_past": 2048, "rms_norm": True, "epsilon": 1e-6}),
    "qkv_decode_r3_f16": Workload(
        name="qkv_decode_r3_f16", kind="qkv", rank=3, shape=(256, 1, (32 + 2 * 8) * 128), dtype="float16",
        num_heads=32, positions="past", cache_rows=8192, rope_base=1.0e6, rope_dim=128,
        extra={"kv_num_heads": 8, "max_len": 4096, "max_past": 4095}),
    # M-RoPE decode with the coefficients computed on the fly (Qwen-VL
    # attention shape: 28 heads of 128, sections [16, 24, 24], interleaved
    # layout), against the same step over a (32768, 64) table
    "mrope_fused_decode_r3_f16": Workload(
        name="mrope_fused_decode_r3_f16", kind="mrope_fused", rank=3, shape=(256, 1, 28 * 128), dtype="float16",
        num_heads=28, positions="mrope", cache_rows=32768, rope_base=1.0e6, rope_dim=128,
        mrope_section=(16, 24, 24), mrope_layout=1, scale=1.0),
    "mrope_r3_bf16_layout1": Workload(
        name="mrope_r3_bf16_layout1", kind="mrope", rank=3, shape=(2, 8192, 28 * 128), dtype="bfloat16",
        num_heads=28, positions="mrope", cache_rows=32768, rope_base=10000.0, rope_dim=128,
        mrope_section=(16, 24, 24), mrope_layout=1, scale=1.0),
    # M-RoPE Q/K rotation with QK-Norm and the cache append: a Qwen3-VL-8B-like
    # attention prefill (32 query heads, 8 key/value heads, head size 128,
    # interleaved sections [24, 20, 20]), t/h/w ids from the M-RoPE recipe
    "mrope_qkv_norm_prefill_r3_f16": Workload(
        name="mrope_qkv_norm_prefill_r3_f16", kind="qkv", rank=3, shape=(2, 4096, (32 + 2 * 8) * 128),
        dtype="float16", num_heads=32, positions="mrope", cache_rows=32768, rope_base=5.0e6, rope_dim=128,
        mrope_section=(24, 20, 20), mrope_layout=1, scale=1.0,
        extra={"kv_num_heads": 8, "max_len": 8192, "max_past": 4096, "rms_norm": True, "epsilon": 1e-6}),
    # the same model's decode step: one token per sequence, 256 sequences, the
    # rest of the K/V history already in the caches (SIMT Q/K kernel: 3 MB)
    "mrope_qkv_norm_decode_r3_f16": Workload(
        name="mrope_qkv_norm_decode_r3_f16", kind="qkv", rank=3, shape=(256, 1, (32 + 2 * 8) * 128),
        dtype="float16", num_heads=32, positions="mrope", cache_rows=32768, rope_base=5.0e6, rope_dim=128,
        mrope_section=(24, 20, 20), mrope_layout=1, scale=1.0,
        extra={"kv_num_heads": 8, "max_len": 8192, "max_past": 8191, "rms_norm": True, "epsilon": 1e-6}),
    "fused_decode_r3_f16": Workload(
        name="fused_decode_r3_f16", kind="fused", rank=3, shape=(256, 1, 40 * 128), dtype="float16",
        num_heads=40, positions="uniform", cache_rows=32768, rope_base=1.0e6, rope_dim=128,
        attention_scaling=1.0),
}

HEADLINE = "rope_r4_f16_interleaved_partial"

# The published configurations in order (the rank-4 float32 parity case, the
# rank-3 gather, the rank-4 partial rotation, M-RoPE in both layouts, the
# decode step with on-the-fly coefficients).
CONFIGS = ["rope_r4_f32_cache3d", "rope_r3_f16_gather", "rope_r4_f16_interleaved_partial",
           "mrope_r3_f16_layout0", "mrope_r3_f16_layout1", "fused_decode_r3_f16"]


# numpy has no bfloat16: bfloat16 data is carried as its uint16 bit patterns.
BF16_BITS = np.uint16


def storage_dtype(name):
    """numpy dtype carrying storage type ``name`` ("float32", "float16", "bfloat16")."""
    return np.dtype(BF16_BITS) if name == "bfloat16" else np.dtype(name)


def itemsize(name):
    return 2 if name == "bfloat16" else np.dtype(name).itemsize


def to_bf16_bits(a):
    """float32 values rounded to nearest-even bfloat16, as bit patterns (finite inputs)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def to_storage(a, dtype):
    """Float data rounded to the storage type carried by numpy dtype ``dtype``."""
    if np.dtype(dtype) == BF16_BITS:
        return to_bf16_bits(a)
    return np.asarray(a).astype(dtype)


def x_normal(shape, dtype, seed=0):
    """N(0, 1) drawn in float32 and rounded to ``dtype`` (nearest-even)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return to_storage(x, dtype)


def inv_freq(base, d, half):
    """``base ** (-2 i / d)`` for i < half: binary64 power, rounded to float32."""
    i = np.arange(half, dtype=np.float64)
    return np.power(np.float64(base), -(2.0 * i) / np.float64(d)).astype(np.float32)


def positions_offset(B, S, seed=1, max_offset=4096):
    rng = np.random.default_rng(seed)
    off = rng.integers(0, max_offset, size=(B, 1), dtype=np.int64)
    return np.arange(S, dtype=np.int64)[None, :] + off


def positions_uniform(B, S, rows, seed=1):
    rng = np.random.default_rng(seed)
    return rng.integers(0, rows, size=(B, S), dtype=np.int64)


def mrope_ids(B, S, rows, seed=1, oor_seed=2, oor_fraction=0.01, grid=32, max_offset=16384):
    """(3, B, S) t/h/w ids: text and image spans, a per-batch offset, 1 % past the cache."""
    rng = np.random.default_rng(seed)
    ids = np.empty((3, B, S), dtype=np.int64)
    spans = [("text", 1024), ("image", 4), ("text", 1024), ("image", 2)]
    for b in range(B):
        t, h, w = [], [], []
        nxt = 0
        for kind, n in spans:
            if kind == "text":
                q = np.arange(nxt, nxt + n, dtype=np.int64)
                t.append(q), h.append(q), w.append(q)
                nxt = nxt + n
            else:
                f, r, c = np.meshgrid(np.arange(n), np.arange(grid), np.arange(grid), indexing="ij")
                t.append(nxt + f.ravel()), h.append(nxt + r.ravel()), w.append(nxt + c.ravel())
                nxt = int(max(t[-1].max(), h[-1].max(), w[-1].max())) + 1
        row = np.stack([np.concatenate(t), np.concatenate(h), np.concatenate(w)])
        # tile or truncate the span pattern to S tokens
        reps = -(-S // row.shape[1])
        if reps > 1:
            width = int(row.max()) + 1
            row = np.concatenate([row + k * width for k in range(reps)], axis=1)
        ids[:, b, :] = row[:, :S] + rng.integers(0, max_offset, dtype=np.int64)
    ids = np.minimum(ids, rows - 1) if rows > 0 else ids
    orng = np.random.default_rng(oor_seed)
    flat = ids.reshape(-1)
    n_oor = int(round(oor_fraction * flat.size))
    if n_oor:
        where = orng.choice(flat.size, size=n_oor, replace=False)
        flat[where] = rows + orng.integers(0, 1 << 20, size=n_oor, dtype=np.int64)
    return ids


def make_inputs(w: Workload, shard=0):
    """Host arrays for workload ``w``: x, position_ids (or None), inv_freq.

    ``shard`` selects an independent batch of the same recipe (one per rank
    when several GPUs each process their own batch); shard 0 is the default.
    """
    base = 1000 * int(shard)
    x = x_normal(w.shape, storage_dtype(w.dtype), seed=base + 0)
    B, S = w.batch, w.seq
    if w.positions == "none":
        pos = None
    elif w.positions == "offset":
        pos = positions_offset(B, S, seed=base + 1)
    elif w.positions == "uniform":
        pos = positions_uniform(B, S, w.cache_rows, seed=base + 1)
    elif w.positions == "mrope":
        pos = mrope_ids(B, S, w.cache_rows, seed=base + 1, oor_seed=base + 2)
    elif w.positions == "past":  # implicit positions past[b] + s; past drawn here
        pos = None
    else:
        raise ValueError(w.positions)
    inv = inv_freq(w.rope_base, w.rope_dim or w.rotary_dim, w.half)
    out = {"x": x, "position_ids": pos, "inv_freq": inv}
    if w.kind == "qkv":
        rng = np.random.default_rng(base + 1)
        out["past_seq_lens"] = rng.integers(0, w.extra["max_past"] + 1, size=B).astype(np.int32)
        if w.extra.get("rms_norm"):
            wrng = np.random.default_rng(base + 3)
            out["q_norm_weight"] = to_storage(wrng.uniform(0.5, 1.5, w.head_size), storage_dtype(w.dtype))
            out["k_norm_weight"] = to_storage(wrng.uniform(0.5, 1.5, w.head_size), storage_dtype(w.dtype))
    return out


def algorithmic_bytes(w: Workload, cached=True):
    """Bytes one pass must move: X + Y + cos/sin touched + positions (+ inv_freq).

    cos/sin "touched" counts rd/2 cosines and rd/2 sines per token (a
    per-token gather, not unique rows); the on-the-fly variant reads inv_freq
    once instead.
    """
    esz = itemsize(w.dtype)
    xy = 2 * w.numel * esz
    if w.kind == "qkv":
        # Q, K, V read once; Q out, K and V into the caches; rd/2 cosines and
        # rd/2 sines per token; the int32 past lengths; with M-RoPE the three
        # int64 position streams (otherwise positions are implicit).
        norm_w = 2 * w.head_size * esz if w.extra.get("rms_norm") else 0
        pos = 3 * 8 * w.tokens if w.positions == "mrope" else 0
        return xy + 2 * w.tokens * w.half * esz + 4 * w.batch + norm_w + pos
    npos = 3 if w.kind in ("mrope", "mrope_fused") else (0 if w.positions == "none" else 1)
    pos = npos * w.tokens * 8
    if w.kind in ("fused", "mrope_fused") and not cached:
        coef = w.half * 4
    else:
        coef = 2 * w.tokens * w.half * esz
    return xy + pos + coef
