"""GPU parity for mrope_apply_qkv (M-RoPE Q/K rotation with grouped-query heads, the
optional QK-RMSNorm and the key/value cache append) against oracle_mrope_qkv, through
the C ABI.

Sources: "com.microsoft.MRotaryEmbedding" README (Description, Inputs/positionIds,
Attributes); "com.microsoft.SparseAttention" README (Description, Inputs); onnxruntime PR
"Add RotaryEmbedding fusion for Qwen3 on-the-fly RoPE patterns" (Qwen3 Architecture).

Every case spans several CTAs with a ragged tail of tokens, pairs whose stream position is
out of range (copied through), and in cache mode rows past the end of the cache (skipped).
The bar is the one every parity test here uses: pass-through elements bit-exact, rotated
float32 within 1e-5, float16 / bfloat16 within 1 ulp; with the norm, the bound derived in
test_gpu_qkv.compare_norm.
"""

import itertools

import numpy as np
import pytest

from parity_util import BF16, cast, compare, mrope_passthrough_mask
from test_gpu_qkv import _dev, _heads, _host, compare_norm

pytestmark = pytest.mark.gpu

NPDT = {"f16": np.float16, "f32": np.float32, "bf16": BF16}


def _run(lib, orc, torch, cuda, dt, packed, cache, inter, rot, layout, norm, H=64, Nq=8, Nkv=2, B=3, S=37, R=64,
         L=80, scale=1.0, seed=0, variant="auto", kernel="rope_qkv_kernel", dynamic=False, past=None):
    rng = np.random.default_rng(2000 + seed)
    npdt = NPDT[dt]
    rd = 0 if rot == "full" else H // 2
    rdw = rd or H
    h = rdw // 2
    sec = {64: (16, 24, 24), 32: (8, 12, 12), 16: (4, 6, 6), 8: (2, 3, 3), 6: (2, 2, 2), 3: (1, 1, 1),
           128: (32, 48, 48), 48: (16, 16, 16), 40: (16, 12, 12), 24: (8, 8, 8)}[h]
    Ntot = Nq + 2 * Nkv
    x = rng.standard_normal((B, S, Ntot * H))
    if norm:
        x = x * rng.uniform(0.1, 10.0, (B, S, Ntot, 1)).repeat(H, -1).reshape(B, S, Ntot * H)
    qkv = cast(x, npdt)
    q, k, v = _heads(qkv, B, S, 0, Nq, Ntot, H), _heads(qkv, B, S, Nq, Nq + Nkv, Ntot, H), \
        _heads(qkv, B, S, Nq + Nkv, Ntot, Ntot, H)
    theta = rng.uniform(-np.pi, np.pi, (R, h))
    cos, sin = cast(np.cos(theta), npdt), cast(np.sin(theta), npdt)
    pos = rng.integers(0, R, (3, B, S))
    pos[0, 0, 5], pos[1, 1, 0], pos[2, -1, -1], pos[1, 0, 9] = R + 3, -1, R, 2 ** 40
    past = np.array([0, 11, 50], dtype=np.int32)[:B] if past is None else np.asarray(past, dtype=np.int32)
    nkw = {}
    if norm:
        nkw = dict(q_norm_weight=cast(rng.uniform(0.5, 2.0, H), npdt), k_norm_weight=cast(rng.uniform(0.5, 2.0, H),
                                                                                        npdt), epsilon=1e-6)
    kc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt) if cache else None
    vc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt) if cache else None
    q_ref, k_ref, kc_ref, vc_ref, n_oor, n_skip = orc.mrope_qkv(
        qkv if packed else q, cos, sin, pos, sec, layout, scale, num_heads=Nq, kv_num_heads=Nkv,
        key=None if packed else k, value=None if (packed or not cache) else v, interleaved=inter,
        rotary_embedding_dim=rd, k_cache=kc0, v_cache=vc0, past_seq_lens=past if cache else None, **nkw)
    assert n_oor > 0 and (n_skip > 0) == bool(cache)

    dv = lambda a: None if a is None else _dev(a, torch, cuda)  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    kc_d, vc_d = dv(kc0), dv(vc0)
    scratch = torch.zeros(8, dtype=torch.int64, device=cuda) if dynamic else None
    dkw = {kk: (dv(vv) if isinstance(vv, np.ndarray) else vv) for kk, vv in nkw.items()}
    with lib.variant(variant):
        qo, ko = lib.mrope_apply_qkv(dv(qkv if packed else q), dv(cos), dv(sin), _dev(pos, torch, cuda), sec,
                                     mrope_layout=layout, scale=scale, num_heads=Nq, kv_num_heads=Nkv,
                                     key=None if packed else dv(k), value=None if (packed or not cache) else dv(v),
                                     interleaved=inter, rotary_embedding_dim=rd, k_cache=kc_d, v_cache=vc_d,
                                     past_seq_lens=_dev(past, torch, cuda) if cache else None, status=status,
                                     scratch=scratch, **dkw)
    torch.cuda.synchronize()
    assert lib.last_kernel() == kernel
    if dynamic:
        assert not bool(scratch.any())
    assert int(status.item()) == 1 | (4 if n_skip else 0)
    smap = orc.mrope_stream_map(sec, layout, h)
    cmp = (lambda got, ref, src, N: compare_norm(got, ref, N, H, rdw, inter)) if norm else \
        (lambda got, ref, src, N: compare(got, ref, src, 3, N,
                                          mrope_passthrough_mask(got.shape, 3, N, rd, pos, R, smap, inter)))
    cmp(_host(qo), q_ref, q, Nq)
    if not cache:
        cmp(_host(ko), k_ref, k, Nkv)
        return
    assert ko is None
    # V rows are copies and every other row of both caches keeps its bits
    assert np.array_equal(_host(vc_d).view(np.uint8), vc_ref.view(np.uint8))
    kc_g = _host(kc_d)
    written = np.zeros((B, L), dtype=bool)
    rows = []
    for b in range(B):
        for s in range(S):
            row = past[b] + s
            if 0 <= row < L:
                written[b, row] = True
                rows.append((b, s, row))
    assert np.array_equal(kc_g.transpose(0, 2, 1, 3)[~written].view(np.uint8),
                          kc0.transpose(0, 2, 1, 3)[~written].view(np.uint8))
    # the written K rows, as a (1, n_rows, Nkv*H) sequence, against the oracle's rows
    got = np.stack([kc_g[b, :, row].reshape(-1) for b, s, row in rows])[None]
    ref = np.stack([kc_ref[b, :, row].reshape(-1) for b, s, row in rows])[None]
    if norm:
        compare_norm(got, ref, Nkv, H, rdw, inter)
    else:
        src = np.stack([k.reshape(B, S, Nkv * H)[b, s] for b, s, row in rows])[None]
        p_rows = np.stack([pos[:, b, s] for b, s, row in rows], axis=1)[:, None, :]
        compare(got, ref, src, 3, Nkv, mrope_passthrough_mask(got.shape, 3, Nkv, rd, p_rows, R, smap, inter))


GRID = list(itertools.product(["f16", "f32", "bf16"], [0, 1], [0, 1], [0, 1], ["full", "partial"], [0, 1], [0, 1]))


@pytest.mark.parametrize("variant", ["auto", "tma"])
@pytest.mark.parametrize("dt,packed,cache,inter,rot,layout,norm", GRID)
def test_mrope_qkv_grid(lib, orc, cuda, dt, packed, cache, inter, rot, layout, norm, variant):
    """At these sizes the automatic choice is the SIMT kernel; forced onto the TMA pipeline
    every case takes it except the norm with partial rotation (the tail is normalised too).
    Half of the pipeline cases draw their tiles from a scratch counter."""
    import torch

    case = GRID.index((dt, packed, cache, inter, rot, layout, norm))
    tma = variant == "tma" and not (norm and rot == "partial")
    _run(lib, orc, torch, cuda, dt, packed, cache, inter, rot, layout, norm,
         scale=0.75 if (inter + layout) % 2 else 1.0, seed=case, variant=variant,
         kernel="rope_qkv_tma_kernel" if tma else "rope_qkv_kernel", dynamic=tma and case % 2 == 1)


# Shapes whose roles get different tiles on the pipeline (tokens x heads per tile, from the
# planner): e.g. H 128 with 32 Q and 8 K/V heads gives Q 4 x 32, K 13 x 8, V 16 x 8; H 256
# with 16 and 2 gives Q 4 x 16, K 14 x 2, V 16 x 2. Sequence lengths leave ragged tiles in
# every role, and cache rows run past the cache's end.
MROPE_QKV_TMA_SHAPES = [
    # dt, H, Nq, Nkv, B, S, packed, cache, inter, rot, layout, norm, L (cache rows)
    ("f16", 128, 32, 8, 2, 41, 1, 1, 0, "full", 1, 1, 45),
    ("bf16", 128, 32, 8, 3, 29, 0, 1, 1, "partial", 0, 0, 60),
    ("f16", 256, 16, 2, 2, 33, 1, 1, 0, "full", 1, 1, 40),
    ("f32", 128, 12, 4, 3, 23, 0, 0, 1, "full", 0, 0, 80),
    ("f16", 64, 24, 8, 2, 50, 1, 0, 0, "full", 1, 1, 80),
    ("bf16", 128, 40, 8, 3, 12, 1, 1, 1, "full", 1, 1, 45),
]


@pytest.mark.parametrize("schedule", ["static", "dynamic"])
@pytest.mark.parametrize("dt,H,Nq,Nkv,B,S,packed,cache,inter,rot,layout,norm,L", MROPE_QKV_TMA_SHAPES)
def test_mrope_qkv_tma_shapes(lib, orc, cuda, dt, H, Nq, Nkv, B, S, packed, cache, inter, rot, layout, norm, L,
                              schedule):
    """The pipeline with a tile shape per role, tiles dealt round robin or drawn from a
    scratch counter."""
    import torch

    case = (dt, H, Nq, Nkv, B, S, packed, cache, inter, rot, layout, norm, L)
    _run(lib, orc, torch, cuda, dt, packed, cache, inter, rot, layout, norm, H=H, Nq=Nq, Nkv=Nkv, B=B, S=S,
         L=L, scale=0.75 if layout == 0 else 1.0, seed=300 + MROPE_QKV_TMA_SHAPES.index(case), variant="tma",
         kernel="rope_qkv_tma_kernel", dynamic=schedule == "dynamic")


@pytest.mark.parametrize("variant", ["simt", "tma"])
@pytest.mark.parametrize("norm", [0, 1])
def test_mrope_qkv_negative_past_lengths(lib, orc, cuda, variant, norm):
    """A negative past length puts a batch's first cache rows below 0: those rows are
    skipped (status bit 2); on the pipeline a tile starting below row 0 is stored row by row."""
    import torch

    _run(lib, orc, torch, cuda, "f16", 1, 1, 0, "full", 1, norm, H=128, Nq=16, Nkv=8, B=2, S=40, L=48,
         seed=40 + norm, variant=variant, kernel="rope_qkv_tma_kernel" if variant == "tma" else "rope_qkv_kernel",
         past=[-21, 3])


@pytest.mark.parametrize("dt,H", [("f16", 96), ("f16", 80), ("bf16", 96), ("f32", 48)])
@pytest.mark.parametrize("cache", [0, 1])
def test_mrope_qkv_tma_unit_counts(lib, orc, cuda, dt, H, cache):
    """Rows of 6 or 5 pair units (not a power of two): the pipeline takes them without the
    norm; with the norm they stay on the SIMT kernel."""
    import torch

    for norm in (0, 1):
        _run(lib, orc, torch, cuda, dt, 1, cache, 0, "full", 1, norm, H=H, Nq=12, Nkv=4, B=2, S=33, L=40,
             seed=H + cache + 2 * norm, variant="tma", kernel="rope_qkv_kernel" if norm else "rope_qkv_tma_kernel")


def test_mrope_qkv_multi_head_attention_in_place_and_empty(lib, orc, cuda):
    """kv_num_heads == num_heads with q_out == query and k_out == key (separate inputs), and
    an empty sequence."""
    import torch

    rng = np.random.default_rng(4)
    B, S, N, H, R = 2, 50, 4, 64, 100
    q = rng.standard_normal((B, S, N * H)).astype(np.float16)
    k = rng.standard_normal((B, S, N * H)).astype(np.float16)
    theta = rng.uniform(-np.pi, np.pi, (R, H // 2))
    cos, sin = np.cos(theta).astype(np.float16), np.sin(theta).astype(np.float16)
    pos = rng.integers(0, R, (3, B, S))
    sec = (8, 12, 12)
    q_ref, k_ref, _, _, n_oor, _ = orc.mrope_qkv(q, cos, sin, pos, sec, 1, 1.0, num_heads=N, kv_num_heads=N, key=k)
    assert n_oor == 0
    qd, kd = _dev(q, torch, cuda), _dev(k, torch, cuda)
    qo, ko = lib.mrope_apply_qkv(qd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos, torch, cuda), sec,
                                 mrope_layout=1, num_heads=N, kv_num_heads=N, key=kd, q_out=qd, k_out=kd)
    torch.cuda.synchronize()
    assert qo.data_ptr() == qd.data_ptr() and ko.data_ptr() == kd.data_ptr()
    smap = orc.mrope_stream_map(sec, 1, H // 2)
    for got, ref, src in ((qd, q_ref, q), (kd, k_ref, k)):
        compare(_host(got), ref, src, 3, N, mrope_passthrough_mask(src.shape, 3, N, 0, pos, R, smap, 0))
    e = torch.zeros((2, 0, N * H), dtype=torch.float16, device=cuda)
    qo, ko = lib.mrope_apply_qkv(e, _dev(cos, torch, cuda), _dev(sin, torch, cuda),
                                 torch.zeros((3, 2, 0), dtype=torch.int64, device=cuda), sec, num_heads=N,
                                 kv_num_heads=N, key=torch.zeros_like(e))
    assert qo.shape == (2, 0, N * H) and ko.shape == (2, 0, N * H)


@pytest.mark.parametrize("dt,H", [("f16", 12), ("f32", 6)])
def test_mrope_qkv_scalar_path(lib, orc, cuda, dt, H):
    """Head rows that are not whole 16-byte vectors: the single-element path."""
    import torch

    _run(lib, orc, torch, cuda, dt, 1, 1, 0, "full", 1, 0, H=H, seed=H)


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("norm", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
def test_mrope_qkv_tma_bits_equal_simt(lib, cuda, dt, norm, layout):
    """The two kernels round every value in the same order: Q and both caches agree bit for
    bit (Qwen2-VL-like heads: 16 Q, 8 K/V, H 128, sections [16, 24, 24])."""
    import torch

    rng = np.random.default_rng(90 + norm + 2 * layout)
    npdt = NPDT[dt]
    B, S, Nq, Nkv, H, R, L = 2, 40, 16, 8, 128, 96, 64
    Ntot = Nq + 2 * Nkv
    qkv = cast(rng.standard_normal((B, S, Ntot * H)) * 3, npdt)
    theta = rng.uniform(-np.pi, np.pi, (R, H // 2))
    cos, sin = cast(np.cos(theta), npdt), cast(np.sin(theta), npdt)
    pos = rng.integers(0, R, (3, B, S))
    pos[1, 0, 3], pos[2, 1, 7] = R, -2
    past = np.array([5, 30], dtype=np.int32)
    kw = {}
    if norm:
        kw = dict(q_norm_weight=_dev(cast(rng.uniform(0.5, 2.0, H), npdt), torch, cuda),
                  k_norm_weight=_dev(cast(rng.uniform(0.5, 2.0, H), npdt), torch, cuda), epsilon=1e-6)
    kc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt)
    out = {}
    for variant in ("simt", "tma"):
        kc, vc = _dev(kc0, torch, cuda), _dev(kc0, torch, cuda)
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        with lib.variant(variant):
            qo, _ = lib.mrope_apply_qkv(_dev(qkv, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda),
                                        _dev(pos, torch, cuda), (16, 24, 24), mrope_layout=layout, scale=0.875,
                                        num_heads=Nq, kv_num_heads=Nkv, k_cache=kc, v_cache=vc,
                                        past_seq_lens=_dev(past, torch, cuda), status=status, **kw)
        torch.cuda.synchronize()
        assert lib.last_kernel() == ("rope_qkv_tma_kernel" if variant == "tma" else "rope_qkv_kernel")
        out[variant] = [_host(t) for t in (qo, kc, vc)] + [int(status.item())]
    for a, b in zip(out["simt"][:3], out["tma"][:3]):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert out["simt"][3] == out["tma"][3] == (1 | 4)


@pytest.mark.parametrize("name,kernel", [("mrope_qkv_norm_prefill_r3_f16", "rope_qkv_tma_kernel"),
                                         ("mrope_qkv_norm_decode_r3_f16", "rope_qkv_kernel")])
def test_mrope_qkv_workload_full_size(lib, orc, cuda, name, kernel):
    """The benchmark's M-RoPE Q/K workloads as the benchmark launches them (packed [Q|K|V],
    QK-Norm, t/h/w ids with 1 % past the table, cache append): Q whole; the written K rows
    against the oracle, V rows bit for bit; every other cache row keeps its fill."""
    import torch

    from rotary_position_embedding_gb300 import workloads as wl

    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    x, inv, past, pos = inp["x"], inp["inv_freq"], inp["past_seq_lens"], inp["position_ids"]
    B, S, H, Nq, Nkv, L = w.batch, w.seq, w.head_size, w.num_heads, w.extra["kv_num_heads"], w.extra["max_len"]
    Ntot = Nq + 2 * Nkv
    cos, sin = orc.cache_build(inv, w.cache_rows, np.float16)
    nkw = dict(q_norm_weight=inp["q_norm_weight"], k_norm_weight=inp["k_norm_weight"], epsilon=w.extra["epsilon"])
    fill = 3.0
    kc0 = np.full((B, Nkv, L, H), fill, np.float16)
    q_ref, _, kc_ref, vc_ref, n_oor, n_skip = orc.mrope_qkv(x, cos, sin, pos, w.mrope_section, w.mrope_layout,
                                                            w.scale, num_heads=Nq, kv_num_heads=Nkv, k_cache=kc0,
                                                            v_cache=kc0, past_seq_lens=past, **nkw)
    assert n_oor > 0 and n_skip == 0
    kc = torch.full((B, Nkv, L, H), fill, dtype=torch.float16, device=cuda)
    vc = torch.full_like(kc, fill)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    qo, ko = lib.mrope_apply_qkv(_dev(x, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda),
                                 _dev(pos, torch, cuda), w.mrope_section, mrope_layout=w.mrope_layout, scale=w.scale,
                                 num_heads=Nq, kv_num_heads=Nkv, k_cache=kc, v_cache=vc,
                                 past_seq_lens=_dev(past, torch, cuda), status=status,
                                 q_norm_weight=_dev(nkw["q_norm_weight"], torch, cuda),
                                 k_norm_weight=_dev(nkw["k_norm_weight"], torch, cuda), epsilon=nkw["epsilon"])
    torch.cuda.synchronize()
    assert lib.last_kernel() == kernel
    assert ko is None and int(status.item()) == 1
    compare_norm(_host(qo), q_ref, Nq, H, H, 0)
    rows = past[:, None].astype(np.int64) + np.arange(S)[None, :]
    bi = torch.arange(B, device=cuda)[:, None].expand(B, S)
    ri = torch.from_numpy(rows).to(cuda)
    k_rows = _host(kc[bi, :, ri].reshape(B, S, Nkv * H))
    k_ref = kc_ref[np.arange(B)[:, None], :, rows].reshape(B, S, Nkv * H)
    compare_norm(k_rows, k_ref, Nkv, H, H, 0)
    v_rows = _host(vc[bi, :, ri].reshape(B, S, Nkv * H))
    assert np.array_equal(v_rows.view(np.uint16), _heads(x, B, S, Nq + Nkv, Ntot, Ntot, H).view(np.uint16))
    kc[bi, :, ri] = fill
    vc[bi, :, ri] = fill
    assert bool(torch.all(kc == fill)) and bool(torch.all(vc == fill))
