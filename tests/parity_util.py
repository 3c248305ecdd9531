"""Comparison helpers for GPU-vs-oracle parity.

Tolerances (the operator's published acceptance bar):
  - pass-through elements (the tail past the rotary width, pairs or tokens
    whose position is out of range) and gathers: bit-exact;
  - float32 outputs: max |gpu - oracle| <= 1e-5;
  - float16 outputs: within 1 float16 ulp of the oracle (which computes the
    exact rotation and rounds once), i.e. adjacent or equal encodings.
"""

import numpy as np

TOL_F32_ABS = 1e-5
TOL_F16_ULP = 1

# numpy has no bfloat16: bfloat16 data travels as its uint16 bit patterns (as
# the oracle takes it). Its tolerance is the float16 one: one ulp of the type.
BF16 = np.uint16


def cast(a, dtype):
    """Float data rounded to the storage type: float16 / float32 by numpy,
    bfloat16 by nearest-even on the float32 bit pattern (finite inputs)."""
    from rotary_position_embedding_gb300.workloads import to_storage

    return to_storage(a, dtype)


def to_float64(a):
    """Values of storage-typed data as float64 (bfloat16 bit patterns decoded)."""
    a = np.asarray(a)
    if a.dtype == BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def is_half_width(dtype):
    return np.dtype(dtype) in (np.dtype(np.float16), np.dtype(BF16))


def f16_ordinal(a):
    u = a.view(np.uint16).astype(np.int32)
    return np.where(u & 0x8000, -(u & 0x7FFF), u)


def head_view(a, rank, N):
    """(B, S, N, H) view of X-shaped data (rank 4 is transposed to token-major)."""
    if rank == 3:
        B, S, HN = a.shape
        return a.reshape(B, S, N, HN // N)
    return a.transpose(0, 2, 1, 3)


def rope_passthrough_mask(shape, rank, N, rd, pos, rows):
    """(B, S, N, H) mask of RotaryEmbedding elements that must be copied bit-exactly."""
    if rank == 3:
        B, S, HN = shape
        H = HN // N
    else:
        B, N, S, H = shape
    rd = rd or H
    m = np.zeros((B, S, N, H), dtype=bool)
    m[..., rd:] = True
    if pos is not None:
        bad = (pos < 0) | (pos >= rows)
        m[bad] = True
    return m


def mrope_passthrough_mask(shape, rank, N, rd, pos3, rows, stream_map, interleaved):
    if rank == 3:
        B, S, HN = shape
        H = HN // N
    else:
        B, N, S, H = shape
    rd = rd or H
    h = rd // 2
    m = np.zeros((B, S, N, H), dtype=bool)
    m[..., rd:] = True
    bad = (pos3 < 0) | (pos3 >= rows)          # (3, B, S)
    for i in range(h):
        st = int(stream_map[i])
        j0, j1 = (2 * i, 2 * i + 1) if interleaved else (i, i + h)
        m[:, :, :, j0] |= bad[st][:, :, None]
        m[:, :, :, j1] |= bad[st][:, :, None]
    return m


def compare(y_gpu, y_ref, x, rank, N, exact_mask=None):
    """Assert parity; returns a dict of statistics (bit-exact fraction, max error)."""
    assert y_gpu.shape == y_ref.shape and y_gpu.dtype == y_ref.dtype
    g = head_view(y_gpu, rank, N)
    r = head_view(y_ref, rank, N)
    xv = head_view(x, rank, N)
    stats = {}
    if exact_mask is not None and exact_mask.any():
        bits = np.uint16 if is_half_width(y_gpu.dtype) else np.uint32
        gb, xb, rb = g.view(bits), xv.view(bits), r.view(bits)
        assert np.array_equal(rb[exact_mask], xb[exact_mask]), "oracle pass-through is not a copy"
        bad = gb[exact_mask] != xb[exact_mask]
        assert not bad.any(), f"{int(bad.sum())} pass-through elements differ from X"
        stats["passthrough"] = int(exact_mask.sum())
    rot = ~exact_mask if exact_mask is not None else np.ones(g.shape, dtype=bool)
    if is_half_width(y_gpu.dtype):
        # sign-magnitude ordinals: float16 and bfloat16 alike
        d = np.abs(f16_ordinal(np.ascontiguousarray(g)) - f16_ordinal(np.ascontiguousarray(r)))
        d = d[rot]
        worst = int(d.max()) if d.size else 0
        assert worst <= TOL_F16_ULP, f"16-bit error {worst} ulp > {TOL_F16_ULP} ({int((d > 1).sum())} elements)"
        stats["max_ulp"] = worst
        stats["bit_exact_frac"] = float((d == 0).mean()) if d.size else 1.0
    else:
        d = np.abs(g.astype(np.float64) - r.astype(np.float64))[rot]
        worst = float(d.max()) if d.size else 0.0
        assert worst <= TOL_F32_ABS, f"float32 max abs error {worst} > {TOL_F32_ABS}"
        stats["max_abs"] = worst
        stats["bit_exact_frac"] = float((d == 0).mean()) if d.size else 1.0
    return stats
