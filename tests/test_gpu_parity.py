"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, element by element.

Small cases span several CTA tiles with ragged tails, every variant (rank 3/4,
2-D/3-D cache, half-split/interleaved, full/partial rotation, float32/float16,
128-bit vector and scalar paths), out-of-range positions, in-place calls and
edge sizes. The full-size workloads run in the launch configuration the
benchmark times and are compared in full.
"""

import itertools
import zlib

import numpy as np
import pytest

from parity_util import BF16, cast, compare, mrope_passthrough_mask, rope_passthrough_mask
from rotary_position_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DT = {"f16": np.float16, "f32": np.float32, "bf16": BF16}


def _tdt(torch, dt):
    return {"f16": torch.float16, "f32": torch.float32, "bf16": torch.bfloat16}[dt]


def _bits(torch, dt):
    return torch.int32 if dt == "f32" else torch.int16


def _dev(a, torch, cuda, offset=0):
    """Device copy of a host array; offset > 0 places it that many elements past a
    16-byte boundary (contiguous but misaligned for the vector path)."""
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == BF16 else torch.from_numpy(a)
    if offset == 0:
        return t.to(cuda)
    big = torch.empty(t.numel() + offset, dtype=t.dtype, device=cuda)
    v = big[offset:offset + t.numel()].view(t.shape)
    v.copy_(t.to(cuda))
    return v


def _seed(*params):
    return zlib.crc32(repr(params).encode())


def _host(t):
    import torch

    if t.dtype == torch.bfloat16:
        return t.detach().view(torch.int16).cpu().numpy().view(BF16)
    return t.detach().cpu().numpy()


def _x_shape(rank, B, S, N, H):
    return (B, S, N * H) if rank == 3 else (B, N, S, H)


@pytest.fixture(scope="module")
def torch_mod():
    import torch

    return torch


# ---------------------------------------------------------------------------
# RotaryEmbedding: small exhaustive grid
# ---------------------------------------------------------------------------

ROPE_GRID = [c + (v,) for c in itertools.product(
    ["f16", "f32", "bf16"], [3, 4], ["pos", "cache3d"], [0, 1], ["full", "partial"],
    ["vector", "scalar_shape", "scalar_misaligned"]) for v in (["simt", "tma"] if c[-1] == "vector" else ["simt"])]


@pytest.mark.parametrize("dt,rank,cache,inter,rot,path,variant", ROPE_GRID)
def test_rope_grid(lib, orc, cuda, torch_mod, dt, rank, cache, inter, rot, path, variant):
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(_seed(dt, rank, cache, inter, rot, path))
    B, S, N = 3, 37, 5
    H = 6 if path == "scalar_shape" else 32
    rd = 0 if rot == "full" else (4 if H == 6 else 16)
    h = (rd or H) // 2
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    inv = wl.inv_freq(10000.0, rd or H, h)
    if cache == "pos":
        R = 97
        cos, sin = orc.cache_build(inv, R, dtype)
        pos = rng.integers(0, R, (B, S))
        pos[0, 3], pos[1, 0], pos[2, S - 1], pos[2, 5] = -1, R, 1 << 40, R - 1
    else:
        R = 0
        cos3, sin3 = orc.cache_build(inv, B * S, dtype)
        cos, sin = cos3.reshape(B, S, h), sin3.reshape(B, S, h)
        pos = None
    nh = N if rank == 3 else 0
    y_ref, n_oor = orc.rope(x, cos, sin, pos, inter, rd, nh)
    off = 1 if path == "scalar_misaligned" else 0
    xd = _dev(x, torch, cuda, off)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    with lib.variant(variant):
        yd = lib.rope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda),
                            None if pos is None else _dev(pos, torch, cuda), interleaved=inter,
                            rotary_embedding_dim=rd, num_heads=nh, oor_flag=flag)
    torch.cuda.synchronize()
    mask = rope_passthrough_mask(shape, rank, N, rd, pos, R)
    compare(_host(yd), y_ref, x, rank, N, mask)
    assert int(flag.item()) == (1 if n_oor else 0)


@pytest.mark.parametrize("dt,rank,inter", list(itertools.product(["f16", "f32", "bf16"], [3, 4], [0, 1])))
def test_rope_in_place(lib, orc, cuda, torch_mod, dt, rank, inter):
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(21)
    B, S, N, H = 2, 19, 4, 64
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    inv = wl.inv_freq(10000.0, H, H // 2)
    cos, sin = orc.cache_build(inv, 50, dtype)
    pos = rng.integers(0, 50, (B, S))
    nh = N if rank == 3 else 0
    y_ref, _ = orc.rope(x, cos, sin, pos, inter, 0, nh)
    xd = _dev(x, torch, cuda)
    out = lib.rope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos, torch, cuda),
                         interleaved=inter, num_heads=nh, out=xd)
    torch.cuda.synchronize()
    assert out.data_ptr() == xd.data_ptr()
    compare(_host(xd), y_ref, x, rank, N, rope_passthrough_mask(shape, rank, N, 0, pos, 50))


@pytest.mark.parametrize("case", ["B1S1N1H2", "N1_long_S", "many_heads", "H8_f32_rank4", "all_oor",
                                  "zero_rows", "big_positions"])
def test_rope_edges(lib, orc, cuda, torch_mod, case):
    torch = torch_mod
    rng = np.random.default_rng(22)
    rank, dtype, inter, rd = 3, np.float16, 0, 0
    if case == "B1S1N1H2":
        B, S, N, H, R = 1, 1, 1, 2, 4
    elif case == "N1_long_S":
        B, S, N, H, R = 2, 3001, 1, 16, 4000
    elif case == "many_heads":
        B, S, N, H, R = 1, 5, 160, 128, 16    # N*U > 1024 threads: heads split across CTAs
    elif case == "H8_f32_rank4":
        B, S, N, H, R, rank, dtype, inter = 3, 33, 2, 8, 40, 4, np.float32, 1
    elif case == "all_oor":
        B, S, N, H, R = 2, 7, 3, 16, 5
    elif case == "zero_rows":
        B, S, N, H, R = 2, 7, 3, 16, 0
    else:
        B, S, N, H, R = 2, 9, 2, 32, 1 << 20
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    h = (rd or H) // 2
    inv = wl.inv_freq(10000.0, H, h)
    Rb = min(R, 4096) if case != "big_positions" else 4096
    cos, sin = orc.cache_build(inv, max(Rb, 0), dtype)
    if case == "big_positions":
        # a (2^20)-row table is only partly materialised: gather rows < 4096 or >= 2^20
        cos_full = np.zeros((R, h), dtype=dtype)
        sin_full = np.zeros((R, h), dtype=dtype)
        cos_full[:Rb], sin_full[:Rb] = cos, sin
        cos, sin = cos_full, sin_full
        pos = rng.integers(0, Rb, (B, S))
        pos[0, 0], pos[1, 1] = R, (1 << 62)
    elif case == "all_oor":
        pos = rng.integers(R, 100, (B, S))
    elif case == "zero_rows":
        pos = rng.integers(0, 3, (B, S))
    else:
        pos = rng.integers(0, R, (B, S))
    nh = N if rank == 3 else 0
    y_ref, n_oor = orc.rope(x, cos, sin, pos, inter, rd, nh)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    cd = _dev(cos, torch, cuda) if cos.size else torch.empty((0, h), dtype=torch.float16, device=cuda)
    sd = _dev(sin, torch, cuda) if sin.size else torch.empty((0, h), dtype=torch.float16, device=cuda)
    yd = lib.rope_apply(_dev(x, torch, cuda), cd, sd, _dev(pos, torch, cuda), interleaved=inter,
                        rotary_embedding_dim=rd, num_heads=nh, oor_flag=flag)
    torch.cuda.synchronize()
    compare(_host(yd), y_ref, x, rank, N, rope_passthrough_mask(shape, rank, N, rd, pos, R))
    assert int(flag.item()) == (1 if n_oor else 0)


def test_empty_and_errors_on_gpu(lib, cuda, torch_mod):
    torch = torch_mod
    x = torch.empty((0, 4, 64), dtype=torch.float16, device=cuda)
    c = torch.empty((8, 8), dtype=torch.float16, device=cuda)
    p = torch.empty((0, 4), dtype=torch.int64, device=cuda)
    y = lib.rope_apply(x, c, c, p, num_heads=4)
    assert y.shape == x.shape
    xd = torch.zeros((2, 4, 64), dtype=torch.float64, device=cuda)   # no float64 kernels
    cd = torch.zeros((8, 8), dtype=torch.float64, device=cuda)
    pp = torch.zeros((2, 4), dtype=torch.int64, device=cuda)
    with pytest.raises(lib.RopeError) as e:
        lib.rope_apply(xd, cd, cd, pp, num_heads=4)
    assert e.value.status == lib.ROPE_ERR_UNSUPPORTED
    with pytest.raises(lib.RopeError) as e:
        lib.rope_apply(x.new_zeros((2, 4, 64)), c, c, pp, num_heads=3)
    assert e.value.status == lib.ROPE_ERR_INVALID_ARG


def test_side_stream(lib, orc, cuda, torch_mod):
    torch = torch_mod
    rng = np.random.default_rng(23)
    x = rng.standard_normal((4, 64, 8 * 128)).astype(np.float16)
    inv = wl.inv_freq(10000.0, 128, 64)
    cos, sin = orc.cache_build(inv, 256, np.float16)
    pos = rng.integers(0, 256, (4, 64))
    y_ref, _ = orc.rope(x, cos, sin, pos, 0, 0, 8)
    s = torch.cuda.Stream()
    xd, cd, sd, pd = (_dev(a, torch, cuda) for a in (x, cos, sin, pos))
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        yd = lib.rope_apply(xd, cd, sd, pd, num_heads=8)
    s.synchronize()
    compare(_host(yd), y_ref, x, 3, 8, rope_passthrough_mask(x.shape, 3, 8, 0, pos, 256))


# ---------------------------------------------------------------------------
# TMA pipeline: tiles that run past the tokens and past the heads, head sizes
# from 16 to 256 elements, stage-ring phases that wrap many times, in place
# ---------------------------------------------------------------------------

TMA_SHAPES = [
    # name, kind, rank, dtype, B, S, N, H, rd, inter
    ("r3_head_groups", "rope", 3, "f16", 2, 9, 300, 64, 0, 0),      # 300 heads: two head groups
    ("r4_both_tails", "rope", 4, "f16", 2, 70, 5, 128, 0, 1),       # S and N tails
    ("r4_f32_h256", "rope", 4, "f32", 2, 45, 3, 256, 64, 0),        # 1 head per tile, partial
    ("r3_decode", "rope", 3, "f16", 67, 1, 40, 128, 0, 0),
    ("r3_h16", "rope", 3, "f16", 3, 101, 7, 16, 0, 1),
    ("r3_many_rounds", "rope", 3, "f16", 8, 4096, 8, 128, 0, 0),    # ~13 tiles per CTA
    ("r4_many_rounds", "rope", 4, "f16", 4, 4096, 8, 128, 64, 1),
    ("mr3_l1", "mrope", 3, "f16", 2, 777, 28, 128, 0, 0),
    ("mr4_l0_tails", "mrope", 4, "f16", 2, 70, 5, 128, 96, 1),
    ("mr3_f32_scale", "mrope", 3, "f32", 2, 300, 6, 64, 0, 0),
]


@pytest.mark.parametrize("case", TMA_SHAPES, ids=[c[0] for c in TMA_SHAPES])
@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("schedule", ["static", "dynamic"])
def test_tma_pipeline_shapes(lib, orc, cuda, torch_mod, case, in_place, schedule):
    torch = torch_mod
    name, kind, rank, dt, B, S, N, H, rd, inter = case
    dtype = DT[dt]
    rng = np.random.default_rng(_seed(*case))
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    h = (rd or H) // 2
    R = 5000
    inv = wl.inv_freq(10000.0, rd or H, h)
    cos, sin = orc.cache_build(inv, R, dtype)
    nh = N if rank == 3 else 0
    xd = _dev(x, torch, cuda)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    scratch = torch.zeros(8, dtype=torch.int64, device=cuda) if schedule == "dynamic" else None
    if kind == "rope":
        pos = rng.integers(0, R, (B, S))
        pos.ravel()[rng.choice(pos.size, size=max(1, pos.size // 50), replace=False)] = R + 3
        y_ref, _ = orc.rope(x, cos, sin, pos, inter, rd, nh)
        with lib.variant("tma"):
            yd = lib.rope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos, torch, cuda),
                                interleaved=inter, rotary_embedding_dim=rd, num_heads=nh, oor_flag=flag,
                                out=xd if in_place else None, scratch=scratch)
        mask = rope_passthrough_mask(shape, rank, N, rd, pos, R)
    else:
        sec = (h - 2 * (h // 3), h // 3, h // 3)
        layout = 1 if name.startswith("mr3_l1") else 0
        scale = float(np.float32(0.6)) if "scale" in name else 1.0
        pos3 = rng.integers(0, R, (3, B, S))
        pos3.ravel()[rng.choice(pos3.size, size=max(1, pos3.size // 50), replace=False)] = -2
        y_ref, _ = orc.mrope(x, cos, sin, pos3, sec, layout, scale, inter, rd, nh)
        with lib.variant("tma"):
            yd = lib.mrope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos3, torch, cuda),
                                 sec, mrope_layout=layout, scale=scale, interleaved=inter,
                                 rotary_embedding_dim=rd, num_heads=nh, oor_flag=flag,
                                 out=xd if in_place else None, scratch=scratch)
        smap = orc.mrope_stream_map(sec, layout, h)
        mask = mrope_passthrough_mask(shape, rank, N, rd, pos3, R, smap, inter)
    torch.cuda.synchronize()
    compare(_host(yd), y_ref, x, rank, N, mask)
    assert int(flag.item()) == 1   # some positions were out of range; no pipeline timeout (bit 1)
    if scratch is not None:
        assert not scratch.any()   # the launch left its counters zeroed for the next one


def test_dynamic_schedule_back_to_back_and_shared_scratch(lib, orc, cuda, torch_mod):
    """Many launches in one stream share one scratch (each leaves it zeroed); results
    equal the static schedule's bit for bit."""
    torch = torch_mod
    rng = np.random.default_rng(31)
    B, S, N, H = 4, 1024, 16, 128
    x = rng.standard_normal((B, S, N * H)).astype(np.float16)
    inv = wl.inv_freq(10000.0, H, H // 2)
    cos, sin = orc.cache_build(inv, 3000, np.float16)
    pos = rng.integers(0, 3000, (B, S))
    xd, cd, sd, pd = (_dev(a, torch, cuda) for a in (x, cos, sin, pos))
    scratch = torch.zeros(8, dtype=torch.int64, device=cuda)
    with lib.variant("tma"):
        ref = lib.rope_apply(xd, cd, sd, pd, num_heads=N, scratch=None)
        outs = [lib.rope_apply(xd, cd, sd, pd, num_heads=N, scratch=scratch) for _ in range(20)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    assert not scratch.any()


def test_automatic_variant_choice(lib, orc, cuda, torch_mod):
    """The automatic choice: full-rotation RoPE runs the SIMT kernel at any size;
    partial rotation of a large X and M-RoPE of a large X run the TMA pipeline, unless
    M-RoPE's three coefficient rows per token shrink its tiles (few heads), when the
    SIMT heads kernel runs; small X always runs SIMT. Every choice still matches the
    oracle."""
    torch = torch_mod
    rng = np.random.default_rng(37)
    B, S, N, H = 2, 1024, 32, 128                 # 16 MiB of float16: above the pipeline's threshold
    x = rng.standard_normal((B, S, N * H)).astype(np.float16)
    R = 4096
    pos = rng.integers(0, R, (B, S))
    xd, pd = _dev(x, torch, cuda), _dev(pos, torch, cuda)
    cases = [(0, "rope_rows_kernel"), (64, "rope_tma_kernel")]
    tables = {}
    with lib.variant("auto"):
        for rd, family in cases:
            h = (rd or H) // 2
            cos, sin = orc.cache_build(wl.inv_freq(10000.0, rd or H, h), R, np.float16)
            tables[rd] = (_dev(cos, torch, cuda), _dev(sin, torch, cuda))
            y = lib.rope_apply(xd, *tables[rd], pd, num_heads=N, rotary_embedding_dim=rd)
            assert lib.last_kernel() == family, (rd, lib.last_kernel())
            torch.cuda.synchronize()
            y_ref, _ = orc.rope(x, cos, sin, pos, 0, rd, N)
            compare(_host(y), y_ref, x, 3, N, rope_passthrough_mask(x.shape, 3, N, rd, pos, R))
        cos, sin = orc.cache_build(wl.inv_freq(10000.0, H, H // 2), R, np.float16)
        pos3 = rng.integers(0, R, (3, B, S))
        y = lib.mrope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos3, torch, cuda),
                            (16, 24, 24), mrope_layout=1, num_heads=N)
        assert lib.last_kernel() == "rope_tma_kernel"
        torch.cuda.synchronize()
        y_ref, _ = orc.mrope(x, cos, sin, pos3, (16, 24, 24), 1, 1.0, 0, 0, N)
        smap = orc.mrope_stream_map((16, 24, 24), 1, H // 2)
        compare(_host(y), y_ref, x, 3, N, mrope_passthrough_mask(x.shape, 3, N, 0, pos3, R, smap, 0))
        # 4 heads: 16 MiB, but the pipeline's M-RoPE tile would be 5 tokens x 4 heads (5 KB)
        x4 = rng.standard_normal((2, 8192, 4 * H)).astype(np.float16)
        p4 = rng.integers(0, R, (3, 2, 8192))
        y4 = lib.mrope_apply(_dev(x4, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda),
                             _dev(p4, torch, cuda), (16, 24, 24), mrope_layout=1, num_heads=4)
        assert lib.last_kernel() == "rope_mrope_heads_kernel"
        torch.cuda.synchronize()
        y_ref4, _ = orc.mrope(x4, cos, sin, p4, (16, 24, 24), 1, 1.0, 0, 0, 4)
        compare(_host(y4), y_ref4, x4, 3, 4, mrope_passthrough_mask(x4.shape, 3, 4, 0, p4, R, smap, 0))
        small = xd[:, :64].contiguous()           # 1 MiB: SIMT whatever the rotation
        lib.rope_apply(small, *tables[64], pd[:, :64].contiguous(), num_heads=N, rotary_embedding_dim=64)
        assert lib.last_kernel() == "rope_rows_kernel"


# ---------------------------------------------------------------------------
# MRotaryEmbedding
# ---------------------------------------------------------------------------

MROPE_GRID = [c + (v,) for c in itertools.product(
    ["f16", "f32", "bf16"], [3, 4], ["l0", "l1", "stride3"], [0, 1], ["full", "partial_odd_head"],
    [1.0, 0.7], ["vector", "scalar_misaligned"])
    for v in (["simt", "tma"] if c[-1] == "vector" and c[4] == "full" else ["simt"])]


@pytest.mark.parametrize("dt,rank,layout,inter,rot,scale,path,variant", MROPE_GRID)
def test_mrope_grid(lib, orc, cuda, torch_mod, dt, rank, layout, inter, rot, scale, path, variant):
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(_seed(dt, rank, layout, inter, rot, scale, path))
    B, S, N = 2, 45, 3
    if rot == "full":
        H, rd, sec = 64, 0, (8, 12, 12)
    else:
        H, rd, sec = 37, 32, (4, 6, 6)   # odd head size, even rotary width, 5-element tail
    h = (rd or H) // 2
    R = 120
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    inv = wl.inv_freq(10000.0, rd or H, h)
    cos, sin = orc.cache_build(inv, R, dtype)
    pos3 = rng.integers(0, R, (3, B, S))
    oor = rng.random((3, B, S)) < 0.08
    pos3[oor] = rng.choice([-1, R, R + 5, 1 << 40], size=int(oor.sum()))
    nh = N if rank == 3 else 0
    scale = float(np.float32(scale))
    if layout == "stride3":
        smap = orc.mrope_stream_map(sec, 2, h)
        y_ref, n_oor = orc.mrope_map(x, cos, sin, pos3, smap, scale, inter, rd, nh)
    else:
        lay = 0 if layout == "l0" else 1
        smap = orc.mrope_stream_map(sec, lay, h)
        y_ref, n_oor = orc.mrope(x, cos, sin, pos3, sec, lay, scale, inter, rd, nh)
    off = 1 if path == "scalar_misaligned" else 0
    xd = _dev(x, torch, cuda, off)
    args = (xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos3, torch, cuda))
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    kw = dict(scale=scale, interleaved=inter, rotary_embedding_dim=rd, num_heads=nh, oor_flag=flag)
    with lib.variant(variant):
        if layout == "stride3":
            yd = lib.mrope_apply_stream_map(*args, smap.tolist(), **kw)
        else:
            yd = lib.mrope_apply(*args, sec, mrope_layout=0 if layout == "l0" else 1, **kw)
    torch.cuda.synchronize()
    mask = mrope_passthrough_mask(shape, rank, N, rd, pos3, R, smap, inter)
    compare(_host(yd), y_ref, x, rank, N, mask)
    assert int(flag.item()) == (1 if n_oor else 0)


def _random_mrope_cases(n, seed):
    """n seeded shapes: dtype, rank, heads, head size, rotary width, a random three-way
    section of the half width (every stream at least one index), layout (incl. the stride-3
    reading), pairing, scale and token count (both sides of the 512-token switch)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        H = int([32, 64, 96, 128, 256][rng.integers(5)])
        rd = [0, H // 2, H // 4][rng.integers(3)]
        h = (rd or H) // 2
        c1, c2 = sorted(rng.choice(np.arange(1, h), size=2, replace=False).tolist())
        sec = (c1, c2 - c1, h - c2)
        out.append((["f16", "bf16", "f32"][rng.integers(3)], int(rng.choice([3, 4])), int(rng.integers(1, 13)), H,
                    int(rd), sec, ["l0", "l1", "stride3"][rng.integers(3)], int(rng.integers(2)),
                    [1.0, 0.7][rng.integers(2)], int(rng.choice([40, 150, 400]))))
    return out


RANDOM_MROPE = _random_mrope_cases(24, 77)


@pytest.mark.parametrize("variant", ["simt", "tma"])
@pytest.mark.parametrize("dt,rank,N,H,rd,sec,layout,inter,scale,S", RANDOM_MROPE)
def test_mrope_random_shapes(lib, orc, cuda, torch_mod, dt, rank, N, H, rd, sec, layout, inter, scale, S, variant):
    """Whichever kernel the variant leads to (the heads kernel, the rows kernel or the
    pipeline), every element against the oracle; 3% of the ids out of range."""
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(900 + RANDOM_MROPE.index((dt, rank, N, H, rd, sec, layout, inter, scale, S)))
    B = 2
    h = (rd or H) // 2
    R = 1000
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    cos, sin = orc.cache_build(wl.inv_freq(10000.0, rd or H, h), R, dtype)
    pos3 = rng.integers(0, R, (3, B, S))
    oor = rng.random((3, B, S)) < 0.03
    pos3[oor] = rng.choice([-1, R, R + 5, 1 << 40], size=int(oor.sum()))
    nh = N if rank == 3 else 0
    scale = float(np.float32(scale))
    if layout == "stride3":
        smap = orc.mrope_stream_map(sec, 2, h)
        y_ref, n_oor = orc.mrope_map(x, cos, sin, pos3, smap, scale, inter, rd, nh)
    else:
        lay = 0 if layout == "l0" else 1
        smap = orc.mrope_stream_map(sec, lay, h)
        y_ref, n_oor = orc.mrope(x, cos, sin, pos3, sec, lay, scale, inter, rd, nh)
    args = (_dev(x, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos3, torch, cuda))
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    kw = dict(scale=scale, interleaved=inter, rotary_embedding_dim=rd, num_heads=nh, oor_flag=flag)
    with lib.variant(variant):
        if layout == "stride3":
            yd = lib.mrope_apply_stream_map(*args, smap.tolist(), **kw)
        else:
            yd = lib.mrope_apply(*args, sec, mrope_layout=0 if layout == "l0" else 1, **kw)
    torch.cuda.synchronize()
    mask = mrope_passthrough_mask(shape, rank, N, rd, pos3, R, smap, inter)
    compare(_host(yd), y_ref, x, rank, N, mask)
    assert int(flag.item()) == (1 if n_oor else 0)


HEADS_GRID = list(itertools.product(["f16", "f32", "bf16"], [3, 4], ["l0", "l1", "stride3"], [0, 1],
                                    ["full", "partial"], [1.0, 0.7], [2, 4]))


@pytest.mark.parametrize("dt,rank,layout,inter,rot,scale,hpt", HEADS_GRID)
def test_mrope_heads_kernel(lib, orc, cuda, torch_mod, dt, rank, layout, inter, rot, scale, hpt):
    """The SIMT M-RoPE kernel on the 128-bit path: each thread merges a unit's three
    coefficient rows once and rotates 2 (below 512 tokens) or 4 heads with them. 5 heads
    (an uneven last head group either way), out-of-range ids in every stream, partial
    rotation with a tail, both pairings, scaled coefficients; 600 tokens for 4 heads per
    thread, 250 for 2."""
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(_seed(dt, rank, layout, inter, rot, scale, hpt, "heads"))
    B, S, N, H = 2, (300 if hpt == 4 else 125), 5, 64
    rd, sec = (0, (8, 12, 12)) if rot == "full" else (32, (4, 6, 6))
    h = (rd or H) // 2
    R = 700
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    cos, sin = orc.cache_build(wl.inv_freq(10000.0, rd or H, h), R, dtype)
    pos3 = rng.integers(0, R, (3, B, S))
    oor = rng.random((3, B, S)) < 0.05
    pos3[oor] = rng.choice([-1, R, R + 5, 1 << 40], size=int(oor.sum()))
    nh = N if rank == 3 else 0
    scale = float(np.float32(scale))
    if layout == "stride3":
        smap = orc.mrope_stream_map(sec, 2, h)
        y_ref, n_oor = orc.mrope_map(x, cos, sin, pos3, smap, scale, inter, rd, nh)
    else:
        lay = 0 if layout == "l0" else 1
        smap = orc.mrope_stream_map(sec, lay, h)
        y_ref, n_oor = orc.mrope(x, cos, sin, pos3, sec, lay, scale, inter, rd, nh)
    args = (_dev(x, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos3, torch, cuda))
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    kw = dict(scale=scale, interleaved=inter, rotary_embedding_dim=rd, num_heads=nh, oor_flag=flag)
    with lib.variant("simt"):
        if layout == "stride3":
            yd = lib.mrope_apply_stream_map(*args, smap.tolist(), **kw)
        else:
            yd = lib.mrope_apply(*args, sec, mrope_layout=0 if layout == "l0" else 1, **kw)
        assert lib.last_kernel() == "rope_mrope_heads_kernel"
    torch.cuda.synchronize()
    compare(_host(yd), y_ref, x, rank, N, mrope_passthrough_mask(shape, rank, N, rd, pos3, R, smap, inter))
    assert int(flag.item()) == (1 if n_oor else 0)


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
def test_mrope_kernels_agree_bitwise(lib, orc, cuda, torch_mod, dt):
    """The M-RoPE kernels give the same bits on the same tokens: 512 tokens take 4 heads
    per thread, 511 take 2, the pipeline (forced), and the per-element scalar path (X one
    element off 16-byte alignment)."""
    torch = torch_mod
    rng = np.random.default_rng(91)
    N, H, R = 6, 128, 2048
    x = cast(rng.standard_normal((1, 512, N * H)), DT[dt])
    cos, sin = orc.cache_build(wl.inv_freq(1e6, H, H // 2), R, DT[dt])
    pos3 = rng.integers(0, R, (3, 1, 512))
    pos3[1, 0, 100] = R + 1
    xd, cd, sd, pd = (_dev(a, torch, cuda) for a in (x, cos, sin, pos3))
    outs = {}
    kw = dict(mrope_layout=1, num_heads=N)
    with lib.variant("simt"):
        outs["heads4"] = lib.mrope_apply(xd, cd, sd, pd, (16, 24, 24), **kw)
        assert lib.last_kernel() == "rope_mrope_heads_kernel"
        outs["heads2"] = lib.mrope_apply(xd[:, :511].contiguous(), cd, sd, pd[:, :, :511].contiguous(), (16, 24, 24),
                                         **kw)
        assert lib.last_kernel() == "rope_mrope_heads_kernel"
        outs["scalar"] = lib.mrope_apply(_dev(x, torch, cuda, 1), cd, sd, pd, (16, 24, 24), **kw)
        assert lib.last_kernel() == "rope_rows_kernel"
    with lib.variant("tma"):
        outs["tma"] = lib.mrope_apply(xd, cd, sd, pd, (16, 24, 24), **kw)
        assert lib.last_kernel() == "rope_tma_kernel"
    torch.cuda.synchronize()
    bits = torch.int32 if dt == "f32" else torch.int16
    assert torch.equal(outs["heads4"][:, :511].view(bits), outs["heads2"].view(bits))
    assert torch.equal(outs["heads4"].view(bits), outs["tma"].view(bits))
    assert torch.equal(outs["heads4"].view(bits), outs["scalar"].view(bits))


@pytest.mark.parametrize("dt,rank,inter", list(itertools.product(["f16", "f32", "bf16"], [3, 4], [0, 1])))
@pytest.mark.parametrize("path", ["heads2", "heads4", "tma", "scalar"])
def test_mrope_in_place(lib, orc, cuda, torch_mod, dt, rank, inter, path):
    """y == x for M-RoPE on every path (each thread, or each consumer column, reads its
    elements before it writes them): partial rotation with a tail, out-of-range ids in
    every stream (pairs put back from X), 2 and 4 heads per thread, the pipeline and the
    per-element scalar path."""
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(_seed(dt, rank, inter, path, "inplace"))
    B, S, N, H, rd, sec = 2, (300 if path == "heads4" else 40), 5, 64, 48, (8, 8, 8)
    R = 400
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    cos, sin = orc.cache_build(wl.inv_freq(10000.0, rd, rd // 2), R, dtype)
    pos3 = rng.integers(0, R, (3, B, S))
    oor = rng.random((3, B, S)) < 0.05
    pos3[oor] = R + 2
    nh = N if rank == 3 else 0
    y_ref, _ = orc.mrope(x, cos, sin, pos3, sec, 1, 1.0, inter, rd, nh)
    xd = _dev(x, torch, cuda, 1 if path == "scalar" else 0)
    with lib.variant("tma" if path == "tma" else "simt"):
        out = lib.mrope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos3, torch, cuda), sec,
                              mrope_layout=1, interleaved=inter, rotary_embedding_dim=rd, num_heads=nh, out=xd)
        kernel = {"tma": "rope_tma_kernel", "scalar": "rope_rows_kernel"}.get(path, "rope_mrope_heads_kernel")
        assert lib.last_kernel() == kernel
    torch.cuda.synchronize()
    assert out.data_ptr() == xd.data_ptr()
    smap = orc.mrope_stream_map(sec, 1, rd // 2)
    compare(_host(xd), y_ref, x, rank, N, mrope_passthrough_mask(shape, rank, N, rd, pos3, R, smap, inter))


def test_mrope_equal_streams_equals_rope_on_gpu(lib, orc, cuda, torch_mod):
    """Text tokens (t = h = w) reduce M-RoPE to RotaryEmbedding, bit for bit on the GPU too."""
    torch = torch_mod
    rng = np.random.default_rng(24)
    B, S, N, H, R = 2, 77, 4, 128, 300
    x = rng.standard_normal((B, S, N * H)).astype(np.float16)
    inv = wl.inv_freq(1e6, H, H // 2)
    cos, sin = orc.cache_build(inv, R, np.float16)
    p = rng.integers(0, R, (B, S))
    xd, cd, sd = (_dev(a, torch, cuda) for a in (x, cos, sin))
    yr = lib.rope_apply(xd, cd, sd, _dev(p, torch, cuda), num_heads=N)
    for layout in (0, 1):
        ym = lib.mrope_apply(xd, cd, sd, _dev(np.stack([p, p, p]), torch, cuda), (16, 24, 24),
                             mrope_layout=layout, num_heads=N)
        torch.cuda.synchronize()
        assert torch.equal(ym.view(torch.int16), yr.view(torch.int16))


# ---------------------------------------------------------------------------
# On-the-fly coefficients and the cache build
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt,rank,inter,rd,scaling", list(itertools.product(
    ["f16", "f32", "bf16"], [3, 4], [0, 1], [0, 32], [1.0, 0.85])))
def test_fused_grid(lib, orc, cuda, torch_mod, dt, rank, inter, rd, scaling):
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(_seed(dt, rank, inter, rd, scaling))
    B, S, N, H = 5, 13, 6, 64
    h = (rd or H) // 2
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    inv = wl.inv_freq(1e6, rd or H, h)
    pos = rng.integers(0, 32768, (B, S))
    pos[0, 0], pos[1, 2] = 0, 32767
    scaling = float(np.float32(scaling))
    nh = N if rank == 3 else 0
    y_ref = orc.rope_fused(x, inv, pos, scaling, inter, rd, nh)
    xd, ind, pd = _dev(x, torch, cuda), _dev(inv, torch, cuda), _dev(pos, torch, cuda)
    yf = lib.rope_apply_fused(xd, ind, pd, attention_scaling=scaling, interleaved=inter,
                              rotary_embedding_dim=rd, num_heads=nh)
    torch.cuda.synchronize()
    compare(_host(yf), y_ref, x, rank, N, rope_passthrough_mask(shape, rank, N, rd, None, 0))
    # fused == gathering the library's own cache, bit for bit
    cd, sd = lib.rope_cache_build(ind, 32768, _tdt(torch, dt),
                                  attention_scaling=scaling)
    yc = lib.rope_apply(xd, cd, sd, pd, interleaved=inter, rotary_embedding_dim=rd, num_heads=nh)
    torch.cuda.synchronize()
    bits = _bits(torch, dt)
    assert torch.equal(yc.view(bits), yf.view(bits))


@pytest.mark.parametrize("dt,rank,layout,inter,rd,scale,path", [c + ("vector",) for c in itertools.product(
    ["f16", "f32", "bf16"], [3, 4], [0, 1], [0, 1], [0, 32], [1.0, 0.7])] + [
    ("f16", 3, 1, 0, 0, 0.7, "scalar_misaligned"), ("f32", 4, 0, 1, 32, 1.0, "scalar_misaligned"),
    ("f16", 3, 1, 1, 10, 0.7, "scalar_shape")])
def test_mrope_fused_grid(lib, orc, cuda, torch_mod, dt, rank, layout, inter, rd, scale, path):
    """M-RoPE on the fly against the oracle; where every position lies inside a
    rope_cache_build table, bit for bit equal to mrope_apply over that table."""
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(_seed(dt, rank, layout, inter, rd, scale, path))
    B, S, N, H = 4, 29, 5, 64 if path != "scalar_shape" else 14
    h = (rd or H) // 2
    sec = (h - 2 * (h // 3), h // 3, h // 3)
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    inv = wl.inv_freq(1e6, rd or H, h)
    R = 8192
    pos3 = rng.integers(0, R, (3, B, S))
    scale = float(np.float32(scale))
    nh = N if rank == 3 else 0
    off = 1 if path == "scalar_misaligned" else 0
    y_ref = orc.mrope_fused(x, inv, pos3, sec, layout, scale, 0.9, inter, rd, nh)
    xd, ind, pd = _dev(x, torch, cuda, off), _dev(inv, torch, cuda), _dev(pos3, torch, cuda)
    yf = lib.mrope_apply_fused(xd, ind, pd, sec, mrope_layout=layout, scale=scale, attention_scaling=0.9,
                               interleaved=inter, rotary_embedding_dim=rd, num_heads=nh)
    torch.cuda.synchronize()
    assert lib.last_kernel() == "rope_fused_kernel"
    compare(_host(yf), y_ref, x, rank, N, rope_passthrough_mask(shape, rank, N, rd, None, 0))
    cd, sd = lib.rope_cache_build(ind, R, _tdt(torch, dt),
                                  attention_scaling=0.9)
    yc = lib.mrope_apply(xd, cd, sd, pd, sec, mrope_layout=layout, scale=scale, interleaved=inter,
                         rotary_embedding_dim=rd, num_heads=nh)
    torch.cuda.synchronize()
    bits = _bits(torch, dt)
    assert torch.equal(yc.view(bits), yf.view(bits))


def _random_fused_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        H = int([32, 64, 96, 128, 256][rng.integers(5)])
        out.append((["f16", "bf16", "f32"][rng.integers(3)], int(rng.choice([3, 4])), int(rng.integers(1, 9)), H,
                    [0, H // 2][rng.integers(2)], int(rng.integers(2)), float([1e4, 1e6, 5e6][rng.integers(3)]),
                    float([1.0, 0.7071067690849304, 1.25, -0.5][rng.integers(4)])))
    return out


RANDOM_FUSED = _random_fused_cases(16, 31)


@pytest.mark.parametrize("dt,rank,N,H,rd,inter,base,scaling", RANDOM_FUSED)
def test_fused_random_shapes(lib, orc, cuda, torch_mod, dt, rank, N, H, rd, inter, base, scaling):
    """On-the-fly RoPE, whose 16-bit coefficients come from float32 sincos wherever that
    provably gives the binary64 result: positions in [0, 65536) bit for bit equal to
    gathering rope_cache_build's 65536-row table, and positions out to +-2^20 against the
    oracle."""
    torch = torch_mod
    dtype = DT[dt]
    rng = np.random.default_rng(1300 + RANDOM_FUSED.index((dt, rank, N, H, rd, inter, base, scaling)))
    B, S = 3, 37
    h = (rd or H) // 2
    shape = _x_shape(rank, B, S, N, H)
    x = cast(rng.standard_normal(shape), dtype)
    inv = wl.inv_freq(base, rd or H, h)
    nh = N if rank == 3 else 0
    xd, ind = _dev(x, torch, cuda), _dev(inv, torch, cuda)
    kw = dict(attention_scaling=scaling, interleaved=inter, rotary_embedding_dim=rd, num_heads=nh)
    # inside a 65536-row table: the fused result equals the cached one bit for bit
    pos = rng.integers(0, 1 << 16, (B, S))
    pd = _dev(pos, torch, cuda)
    yf = lib.rope_apply_fused(xd, ind, pd, **kw)
    cd, sd = lib.rope_cache_build(ind, 1 << 16, _tdt(torch, dt), attention_scaling=scaling)
    yc = lib.rope_apply(xd, cd, sd, pd, interleaved=inter, rotary_embedding_dim=rd, num_heads=nh)
    torch.cuda.synchronize()
    bits = _bits(torch, dt)
    assert torch.equal(yc.view(bits), yf.view(bits))
    compare(_host(yf), orc.rope_fused(x, inv, pos, scaling, inter, rd, nh), x, rank, N,
            rope_passthrough_mask(shape, rank, N, rd, None, 0))
    # far positions, negative ones included: against the oracle
    pos = rng.integers(-(1 << 20), 1 << 20, (B, S))
    yf = lib.rope_apply_fused(xd, ind, _dev(pos, torch, cuda), **kw)
    torch.cuda.synchronize()
    compare(_host(yf), orc.rope_fused(x, inv, pos, scaling, inter, rd, nh), x, rank, N,
            rope_passthrough_mask(shape, rank, N, rd, None, 0))


def test_mrope_fused_any_position(lib, orc, cuda, torch_mod):
    """No table, so no position is out of range: large and negative ids rotate too."""
    torch = torch_mod
    rng = np.random.default_rng(91)
    B, S, N, H = 2, 16, 4, 128
    x = rng.standard_normal((B, S, N * H)).astype(np.float16)
    inv = wl.inv_freq(1e6, H, H // 2)
    pos3 = rng.integers(-(1 << 20), 1 << 40, (3, B, S))
    y_ref = orc.mrope_fused(x, inv, pos3, (16, 24, 24), 1, 1.0, 1.0, 0, 0, N)
    yf = lib.mrope_apply_fused(_dev(x, torch, cuda), _dev(inv, torch, cuda), _dev(pos3, torch, cuda),
                               (16, 24, 24), mrope_layout=1, num_heads=N)
    torch.cuda.synchronize()
    compare(_host(yf), y_ref, x, 3, N, None)


@pytest.mark.parametrize("dt,base,scaling", list(itertools.product(["f16", "f32", "bf16"], [1e4, 1e6],
                                                                    [1.0, 0.7071067690849304])))
def test_cache_build_vs_oracle(lib, orc, cuda, torch_mod, dt, base, scaling):
    torch = torch_mod
    dtype = DT[dt]
    rows, half = 8192, 64
    inv = wl.inv_freq(base, 2 * half, half)
    c_ref, s_ref = orc.cache_build(inv, rows, dtype, scaling)
    cd, sd = lib.rope_cache_build(_dev(inv, torch, cuda), rows,
                                  _tdt(torch, dt),
                                  attention_scaling=scaling)
    torch.cuda.synchronize()
    for got, ref in ((_host(cd), c_ref), (_host(sd), s_ref)):
        if dtype in (np.float16, BF16):
            from parity_util import f16_ordinal
            d = np.abs(f16_ordinal(got) - f16_ordinal(ref))
        else:
            gi, ri = got.view(np.int32).astype(np.int64), ref.view(np.int32).astype(np.int64)
            d = np.abs(gi - ri)
        # cos/sin of the float32 angle are evaluated in binary64 on both sides and rounded to
        # float32: the two libm results differ only when they straddle a rounding boundary
        assert d.max() <= 1
        assert (d == 0).mean() >= 0.99999


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("scaling", [1.0, 0.7, -0.5])
def test_cache_build_long_angles(lib, orc, cuda, torch_mod, dt, scaling):
    """Angles up to 131072 rad on 16-bit storage, where most values come from float32
    sincos kept only when the rounding chain cannot tell it from the binary64 one: the
    same bar as above (the two binary64 libraries may round apart at a float32 boundary),
    here with a count -- at most 1 in 10^6 values may differ, by one unit."""
    torch = torch_mod
    dtype = DT[dt]
    rows, half = 1 << 17, 64
    inv = wl.inv_freq(1e6, 2 * half, half)
    c_ref, s_ref = orc.cache_build(inv, rows, dtype, scaling)
    cd, sd = lib.rope_cache_build(_dev(inv, torch, cuda), rows, _tdt(torch, dt), attention_scaling=scaling)
    torch.cuda.synchronize()
    from parity_util import f16_ordinal
    for got, ref in ((_host(cd), c_ref), (_host(sd), s_ref)):
        d = np.abs(f16_ordinal(got) - f16_ordinal(ref))
        assert d.max() <= 1
        assert int((d != 0).sum()) <= ref.size // 10 ** 6


# ---------------------------------------------------------------------------
# Full-size workloads, launched exactly as the benchmark launches them
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", [n for n, w in wl.WORKLOADS.items() if w.kind != "qkv"])
def test_workload_full_size(lib, orc, cuda, torch_mod, name):
    torch = torch_mod
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    x, pos, inv = inp["x"], inp["position_ids"], inp["inv_freq"]
    dtype = wl.storage_dtype(w.dtype)
    tdt = {"float32": torch.float32, "float16": torch.float16, "bfloat16": torch.bfloat16}[w.dtype]
    nh = w.num_heads if w.rank == 3 else 0
    xd, ind = _dev(x, torch, cuda), _dev(inv, torch, cuda)
    if w.kind == "rope" and w.positions == "none":
        cos, sin = orc.cache_build(inv, w.tokens, dtype)   # row (b, s) at position s (B = 1)
        cos, sin = cos.reshape(w.batch, w.seq, w.half), sin.reshape(w.batch, w.seq, w.half)
        y_ref, _ = orc.rope(x, cos, sin, None, w.interleaved, w.rotary_embedding_dim, nh)
        yd = lib.rope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), None,
                            interleaved=w.interleaved, rotary_embedding_dim=w.rotary_embedding_dim,
                            num_heads=nh)
        mask = rope_passthrough_mask(x.shape, w.rank, w.num_heads, w.rotary_embedding_dim, None, 0)
    elif w.kind == "rope":
        cd, sd = lib.rope_cache_build(ind, w.cache_rows, tdt)
        cos, sin = orc.cache_build(inv, w.cache_rows, dtype)
        y_ref, _ = orc.rope(x, cos, sin, pos, w.interleaved, w.rotary_embedding_dim, nh)
        yd = lib.rope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos, torch, cuda),
                            interleaved=w.interleaved, rotary_embedding_dim=w.rotary_embedding_dim,
                            num_heads=nh)
        mask = rope_passthrough_mask(x.shape, w.rank, w.num_heads, w.rotary_embedding_dim, pos,
                                     w.cache_rows)
        torch.cuda.synchronize()
        # the library's own cache gives the same result as the oracle's table
        yc = lib.rope_apply(xd, cd, sd, _dev(pos, torch, cuda), interleaved=w.interleaved,
                            rotary_embedding_dim=w.rotary_embedding_dim, num_heads=nh)
        torch.cuda.synchronize()
        compare(_host(yc), y_ref, x, w.rank, w.num_heads, mask)
    elif w.kind == "mrope":
        cos, sin = orc.cache_build(inv, w.cache_rows, dtype)
        y_ref, n_oor = orc.mrope(x, cos, sin, pos, w.mrope_section, w.mrope_layout, w.scale,
                                 w.interleaved, w.rotary_embedding_dim, nh)
        assert n_oor > 0
        flag = torch.zeros(1, dtype=torch.int32, device=cuda)
        yd = lib.mrope_apply(xd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos, torch, cuda),
                             w.mrope_section, mrope_layout=w.mrope_layout, scale=w.scale,
                             interleaved=w.interleaved, rotary_embedding_dim=w.rotary_embedding_dim,
                             num_heads=nh, oor_flag=flag)
        smap = orc.mrope_stream_map(w.mrope_section, w.mrope_layout, w.half)
        mask = mrope_passthrough_mask(x.shape, w.rank, w.num_heads, w.rotary_embedding_dim, pos,
                                      w.cache_rows, smap, w.interleaved)
        torch.cuda.synchronize()
        assert int(flag.item()) == 1
    elif w.kind == "mrope_fused":
        y_ref = orc.mrope_fused(x, inv, pos, w.mrope_section, w.mrope_layout, w.scale, w.attention_scaling,
                                w.interleaved, w.rotary_embedding_dim, nh)
        yd = lib.mrope_apply_fused(xd, ind, _dev(pos, torch, cuda), w.mrope_section, mrope_layout=w.mrope_layout,
                                   scale=w.scale, attention_scaling=w.attention_scaling, interleaved=w.interleaved,
                                   rotary_embedding_dim=w.rotary_embedding_dim, num_heads=nh)
        mask = rope_passthrough_mask(x.shape, w.rank, w.num_heads, w.rotary_embedding_dim, None, 0)
        torch.cuda.synchronize()
    else:  # fused decode, and the cached path it replaces
        y_ref = orc.rope_fused(x, inv, pos, w.attention_scaling, w.interleaved, w.rotary_embedding_dim, nh)
        pd = _dev(pos, torch, cuda)
        yd = lib.rope_apply_fused(xd, ind, pd, attention_scaling=w.attention_scaling,
                                  interleaved=w.interleaved, rotary_embedding_dim=w.rotary_embedding_dim,
                                  num_heads=nh)
        cd, sd = lib.rope_cache_build(ind, w.cache_rows, tdt, attention_scaling=w.attention_scaling)
        yc = lib.rope_apply(xd, cd, sd, pd, interleaved=w.interleaved,
                            rotary_embedding_dim=w.rotary_embedding_dim, num_heads=nh)
        torch.cuda.synchronize()
        assert torch.equal(yc.view(torch.int16), yd.view(torch.int16))
        mask = rope_passthrough_mask(x.shape, w.rank, w.num_heads, w.rotary_embedding_dim, None, 0)
    torch.cuda.synchronize()
    stats = compare(_host(yd), y_ref, x, w.rank, w.num_heads, mask)
    print(name, stats)


@pytest.mark.parametrize("variant,kernel", [("auto", "rope_tma_kernel"), ("simt", "rope_mrope_heads_kernel")])
@pytest.mark.parametrize("dt", ["float16", "bfloat16"])
def test_mrope_full_size_stride3_reading(lib, orc, cuda, torch_mod, variant, kernel, dt):
    """The M-RoPE workload ((2, 8192, 28 x 128), sections [16, 24, 24], 1 % of ids past the
    table) under the other reading of the interleaved layout that the MRotaryEmbedding
    README names without printing: stride-3 slots, h at i % 3 == 1 below 3 * 24, w at
    i % 3 == 2 below 3 * 24, t elsewhere. For [16, 24, 24] that map differs from the
    count-honouring one the library takes for layout 1, so it goes through
    mrope_apply_stream_map, at full size, on both kernels."""
    torch = torch_mod
    w = wl.WORKLOADS["mrope_r3_f16_layout1"]
    inp = wl.make_inputs(w.with_shape(dtype=dt))
    x, pos, inv = inp["x"], inp["position_ids"], inp["inv_freq"]
    dtype = wl.storage_dtype(dt)
    smap = orc.mrope_stream_map(w.mrope_section, 2, w.half)
    assert not np.array_equal(smap, orc.mrope_stream_map(w.mrope_section, 1, w.half))
    assert np.bincount(smap, minlength=3).tolist() == [22, 21, 21]
    cos, sin = orc.cache_build(inv, w.cache_rows, dtype)
    y_ref, n_oor = orc.mrope_map(x, cos, sin, pos, smap, w.scale, w.interleaved, w.rotary_embedding_dim,
                                 w.num_heads)
    assert n_oor > 0
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    with lib.variant(variant):
        yd = lib.mrope_apply_stream_map(_dev(x, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda),
                                        _dev(pos, torch, cuda), smap, scale=w.scale, interleaved=w.interleaved,
                                        rotary_embedding_dim=w.rotary_embedding_dim, num_heads=w.num_heads,
                                        oor_flag=flag)
    torch.cuda.synchronize()
    assert lib.last_kernel() == kernel
    assert int(flag.item()) == 1
    mask = mrope_passthrough_mask(x.shape, w.rank, w.num_heads, w.rotary_embedding_dim, pos, w.cache_rows, smap,
                                  w.interleaved)
    stats = compare(_host(yd), y_ref, x, w.rank, w.num_heads, mask)
    print("stride-3 reading", dt, variant, stats)
