"""GPU parity for rope_apply_qkv (Q and K rotation with grouped-query heads and the
key/value cache append) against oracle_rope_qkv, through the C ABI.

Sources: "com.microsoft.SparseAttention" README (Description, Inputs, Attributes
do_rotary and kv_num_heads); onnxruntime PR "Add RotaryEmbedding fusion for Qwen3
on-the-fly RoPE patterns" (Verification, Qwen3 Architecture).

Every case spans several CTAs with a ragged tail of tokens, out-of-range positions
(copied through), and in cache mode rows past the end of the cache (skipped). The
bar is the one every parity test here uses: pass-through elements (tails, V heads,
out-of-range tokens, untouched cache rows) bit-exact; rotated float32 within 1e-5,
float16 within 1 ulp.
"""

import itertools

import numpy as np
import pytest

from parity_util import BF16, cast, compare, to_float64
from rotary_position_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TORCH_DT = {"f16": "float16", "f32": "float32"}


def _dev(a, torch, cuda, offset=0):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == BF16 else torch.from_numpy(a)
    if offset == 0:
        return t.to(cuda)
    flat = torch.empty(t.numel() + offset, dtype=t.dtype, device=cuda)
    v = flat[offset:].view(t.shape)
    v.copy_(t.to(cuda))
    return v


def _host(t):
    import torch

    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(BF16)
    return t.cpu().numpy()


def _heads(a, B, S, n0, n1, Ntot, H):
    """Heads [n0, n1) of a (B, S, Ntot*H) array as a contiguous (B, S, (n1-n0)*H) array."""
    return np.ascontiguousarray(a.reshape(B, S, Ntot, H)[:, :, n0:n1]).reshape(B, S, (n1 - n0) * H)


def _token_mask(B, S, N, H, rd, bad_tok):
    m = np.zeros((B, S, N, H), dtype=bool)
    m[..., rd:] = True
    m[bad_tok] = True
    return m


def _run_case(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H, offset=0, Nq=8, Nkv=2,
              B=3, S=37, R=64, L=80, seed=0, variant="auto", kernel="rope_qkv_kernel", past=None,
              dynamic=False):
    rng = np.random.default_rng(seed)
    npdt = {"f16": np.float16, "f32": np.float32, "bf16": BF16}[dt]
    rd = 0 if rot == "full" else H // 2
    h = (rd or H) // 2
    Ntot = Nq + 2 * Nkv
    qkv = cast(rng.standard_normal((B, S, Ntot * H)), npdt)
    q, k, v = _heads(qkv, B, S, 0, Nq, Ntot, H), _heads(qkv, B, S, Nq, Nq + Nkv, Ntot, H), \
        _heads(qkv, B, S, Nq + Nkv, Ntot, Ntot, H)
    theta = rng.uniform(-np.pi, np.pi, (R, h))
    cos, sin = cast(np.cos(theta), npdt), cast(np.sin(theta), npdt)
    past = np.array([0, 11, 50], dtype=np.int32)[:B] if past is None else np.asarray(past, dtype=np.int32)
    if implicit:
        pos = None
        eff = past[:, None].astype(np.int64) + np.arange(S)[None, :]
    else:
        pos = rng.integers(0, R, (B, S))
        pos[0, 5], pos[1, 0], pos[-1, -1] = R + 3, -1, R
        eff = pos
    bad_tok = (eff < 0) | (eff >= R)
    kc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt) if cache else None
    vc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt) if cache else None
    use_past = cache or implicit
    ref = orc.rope_qkv(qkv if packed else q, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv,
                       key=None if packed else k, value=None if (packed or not cache) else v,
                       interleaved=inter, rotary_embedding_dim=rd, k_cache=kc0, v_cache=vc0,
                       past_seq_lens=past if use_past else None)
    q_ref, k_ref, kc_ref, vc_ref, n_oor, n_skip = ref
    assert n_oor > 0 and (n_skip > 0) == bool(cache)

    dv = lambda a: None if a is None else _dev(a, torch, cuda, offset)  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    kc_d, vc_d = dv(kc0), dv(vc0)
    scratch = torch.zeros(8, dtype=torch.int64, device=cuda) if dynamic else None
    with lib.variant(variant):
        qo, ko = lib.rope_apply_qkv(dv(qkv if packed else q), dv(cos), dv(sin),
                                    None if pos is None else _dev(pos, torch, cuda), num_heads=Nq,
                                    kv_num_heads=Nkv, key=None if packed else dv(k),
                                    value=None if (packed or not cache) else dv(v), interleaved=inter,
                                    rotary_embedding_dim=rd, k_cache=kc_d, v_cache=vc_d,
                                    past_seq_lens=_dev(past, torch, cuda) if use_past else None, status=status,
                                    scratch=scratch)
    torch.cuda.synchronize()
    if kernel is not None:
        assert lib.last_kernel() == kernel
    if dynamic:  # the launch leaves its schedule counters at zero for the next one
        assert not bool(scratch.any())
    rdw = rd or H
    compare(_host(qo), q_ref, q, 3, Nq, _token_mask(B, S, Nq, H, rdw, bad_tok))
    if not cache:
        assert ko is not None
        compare(_host(ko), k_ref, k, 3, Nkv, _token_mask(B, S, Nkv, H, rdw, bad_tok))
    else:
        assert ko is None
        # V cache: bit for bit (new rows are copies, the rest untouched)
        assert np.array_equal(_host(vc_d).view(np.uint8), vc_ref.view(np.uint8))
        # K cache: what pass-through means per row -- the old row, or the new token's K
        src = kc0.copy()
        mask = np.ones((B, L, Nkv, H), dtype=bool)          # token-major view of (B, Nkv, L, H)
        k4 = k.reshape(B, S, Nkv, H)
        for b in range(B):
            for s in range(S):
                row = past[b] + s
                if 0 <= row < L:
                    src[b, :, row] = k4[b, s]
                    mask[b, row] = False
                    mask[b, row, :, rdw:] = True
                    if bad_tok[b, s]:
                        mask[b, row] = True
        compare(_host(kc_d), kc_ref, src, 4, Nkv, mask)
    want = 1 | (4 if n_skip else 0)
    assert int(status.item()) == want


QKV_GRID = list(itertools.product(["f16", "f32", "bf16"], [0, 1], [0, 1], [0, 1], ["full", "partial"], [0, 1]))
# the heads-per-thread kernel (the automatic choice at these sizes) and the TMA pipeline (forced)
QKV_KERNELS = {"auto": "rope_qkv_heads_kernel", "tma": "rope_qkv_tma_kernel"}


@pytest.mark.parametrize("variant", list(QKV_KERNELS))
@pytest.mark.parametrize("dt,packed,cache,inter,rot,implicit", QKV_GRID)
def test_qkv_grid(lib, orc, cuda, dt, packed, cache, inter, rot, implicit, variant):
    """S = 37 leaves a ragged last token tile; past lengths 0, 11 and 50 with an 80-row
    cache put whole tiles inside the cache, tiles that cross its end and tiles past it."""
    import torch

    _run_case(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H=64,
              seed=QKV_GRID.index((dt, packed, cache, inter, rot, implicit)), variant=variant,
              kernel=QKV_KERNELS[variant])


# Pipelined kernel geometry: head sizes 32-256 (pair units per row 2-16), one to eight heads
# per tile (kv heads 1, 2, 8; MHA), one-token tiles (S = 1, decode), tiles of 16 tokens.
QKV_TMA_SHAPES = [
    # dt, H, Nq, Nkv, B, S, packed, cache, inter, rot, implicit, R (table rows), L (cache rows)
    ("f16", 128, 32, 8, 2, 40, 1, 1, 0, "full", 1, 48, 45),
    ("f16", 128, 32, 8, 3, 1, 1, 1, 0, "full", 1, 40, 45),
    ("bf16", 128, 16, 8, 2, 33, 0, 1, 1, "partial", 0, 64, 40),
    ("f16", 256, 8, 1, 2, 21, 1, 1, 0, "full", 0, 64, 28),
    ("f32", 128, 6, 3, 2, 19, 0, 0, 1, "full", 1, 25, 80),
    ("f32", 32, 4, 4, 3, 50, 0, 1, 0, "partial", 0, 64, 80),
    ("f16", 32, 12, 4, 2, 64, 1, 0, 0, "full", 0, 64, 80),
]


@pytest.mark.parametrize("schedule", ["static", "dynamic"])
@pytest.mark.parametrize("dt,H,Nq,Nkv,B,S,packed,cache,inter,rot,implicit,R,L", QKV_TMA_SHAPES)
def test_qkv_tma_shapes(lib, orc, cuda, dt, H, Nq, Nkv, B, S, packed, cache, inter, rot, implicit, R, L,
                        schedule):
    """Every case has out-of-range positions and, in cache mode, rows past the cache's end;
    tiles dealt round robin (no scratch) or drawn from a scratch counter."""
    import torch

    case = (dt, H, Nq, Nkv, B, S, packed, cache, inter, rot, implicit, R, L)
    _run_case(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H=H, Nq=Nq, Nkv=Nkv, B=B, S=S,
              R=R, L=L, seed=QKV_TMA_SHAPES.index(case), variant="tma", kernel="rope_qkv_tma_kernel",
              dynamic=schedule == "dynamic")


@pytest.mark.parametrize("dt,H,offset", [("f16", 12, 0), ("f32", 6, 0), ("f16", 64, 1), ("f32", 64, 1)])
@pytest.mark.parametrize("cache", [0, 1])
def test_qkv_scalar_path(lib, orc, cuda, dt, H, offset, cache):
    """Head rows that are not whole 16-byte vectors, or misaligned buffers: the scalar path."""
    import torch

    _run_case(lib, orc, torch, cuda, dt, 0, cache, 1, "partial" if H % 4 == 0 else "full", 0, H=H,
              offset=offset, seed=7 + H + offset)


def test_qkv_multi_head_attention_and_in_place(lib, orc, cuda):
    """kv_num_heads == num_heads, q_out == query and k_out == key (separate inputs)."""
    import torch

    rng = np.random.default_rng(3)
    B, S, N, H, R = 2, 50, 4, 32, 100
    q = rng.standard_normal((B, S, N * H)).astype(np.float16)
    k = rng.standard_normal((B, S, N * H)).astype(np.float16)
    theta = rng.uniform(-np.pi, np.pi, (R, H // 2))
    cos, sin = np.cos(theta).astype(np.float16), np.sin(theta).astype(np.float16)
    pos = rng.integers(0, R, (B, S))
    q_ref, k_ref, _, _, _, _ = orc.rope_qkv(q, cos, sin, pos, num_heads=N, kv_num_heads=N, key=k)
    qd, kd = _dev(q, torch, cuda), _dev(k, torch, cuda)
    qo, ko = lib.rope_apply_qkv(qd, _dev(cos, torch, cuda), _dev(sin, torch, cuda), _dev(pos, torch, cuda),
                                num_heads=N, kv_num_heads=N, key=kd, q_out=qd, k_out=kd)
    torch.cuda.synchronize()
    assert qo.data_ptr() == qd.data_ptr() and ko.data_ptr() == kd.data_ptr()
    compare(_host(qd), q_ref, q, 3, N, _token_mask(B, S, N, H, H, np.zeros((B, S), bool)))
    compare(_host(kd), k_ref, k, 3, N, _token_mask(B, S, N, H, H, np.zeros((B, S), bool)))


def test_qkv_empty_and_rejects(lib, cuda):
    import torch

    q = torch.zeros((2, 0, 64), dtype=torch.float16, device=cuda)
    c = torch.zeros((8, 4), dtype=torch.float16, device=cuda)
    qo, ko = lib.rope_apply_qkv(q, c, c, None, num_heads=2, kv_num_heads=1,
                                key=torch.zeros((2, 0, 32), dtype=torch.float16, device=cuda))
    assert qo.shape == (2, 0, 64) and ko.shape == (2, 0, 32)
    with pytest.raises(lib.RopeError):
        lib.rope_apply_qkv(torch.zeros((1, 4, 96), dtype=torch.float16, device=cuda), c, c, None,
                           num_heads=3, kv_num_heads=2,
                           key=torch.zeros((1, 4, 64), dtype=torch.float16, device=cuda))


def expected_qkv_kernel(auto, norm, qkv_bytes, Nq, Nkv, cache):
    """The automatic choice for whole-width rotation on the 128-bit path: QK-Norm takes
    the TMA pipeline from 8 MiB of [Q|K|V] on; plain RoPE takes the heads-per-thread
    kernel, except in cache mode with Nq <= 2*Nkv from 128 MiB on (the pipeline)."""
    if not auto:
        return "rope_qkv_heads_kernel"
    if norm:
        return "rope_qkv_tma_kernel" if qkv_bytes >= 8 << 20 else "rope_qkv_heads_kernel"
    if cache and Nq <= 2 * Nkv and qkv_bytes >= 128 << 20:
        return "rope_qkv_tma_kernel"
    return "rope_qkv_heads_kernel"


# The automatic choice at its boundaries (kernel numerics are tested above): plain RoPE takes the
# heads kernel except in cache mode with Nq <= 2*Nkv from 128 MiB; QK-Norm and partial rotation
# take the pipeline from 8 MiB.
DISPATCH_CASES = [
    # Nq, Nkv, B, S, rd (0: full), cache, norm, kernel
    (32, 8, 4, 2048, 0, 1, 0, "rope_qkv_heads_kernel"),     # 100.7 MB, the Qwen3-8B prefill
    (8, 8, 1, 22000, 0, 1, 0, "rope_qkv_tma_kernel"),       # MHA, 135.2 MB >= 128 MiB
    (8, 8, 1, 21000, 0, 1, 0, "rope_qkv_heads_kernel"),     # MHA, 129.0 MB < 128 MiB
    (16, 8, 1, 17000, 0, 1, 0, "rope_qkv_tma_kernel"),      # Nq = 2*Nkv, 139.3 MB
    (8, 8, 1, 22000, 0, 0, 0, "rope_qkv_heads_kernel"),     # MHA without caches
    (32, 8, 1, 1024, 0, 1, 1, "rope_qkv_tma_kernel"),       # QK-Norm, 12.6 MB
    (32, 8, 1, 256, 0, 1, 1, "rope_qkv_heads_kernel"),      # QK-Norm, 3.1 MB
    (32, 8, 1, 1024, 64, 1, 0, "rope_qkv_tma_kernel"),      # partial rotation, 12.6 MB
    (32, 8, 1, 256, 64, 1, 0, "rope_qkv_heads_kernel"),     # partial rotation, 3.1 MB
    (32, 8, 256, 1, 0, 1, 0, "rope_qkv_heads_kernel"),      # decode
]


@pytest.mark.parametrize("Nq,Nkv,B,S,rd,cache,norm,kernel", DISPATCH_CASES)
def test_qkv_automatic_choice(lib, cuda, Nq, Nkv, B, S, rd, cache, norm, kernel):
    import torch

    H = 128
    f16 = torch.float16
    qkv = torch.zeros((B, S, (Nq + 2 * Nkv) * H), dtype=f16, device=cuda)
    half = (rd or H) // 2
    c = torch.ones((S + 64, half), dtype=f16, device=cuda)
    past = torch.zeros(B, dtype=torch.int32, device=cuda)
    kw = {}
    if cache:
        kc = torch.zeros((B, Nkv, S, H), dtype=f16, device=cuda)
        kw = dict(k_cache=kc, v_cache=torch.zeros_like(kc), past_seq_lens=past)
    if norm:
        w = torch.ones(H, dtype=f16, device=cuda)
        kw.update(q_norm_weight=w, k_norm_weight=w)
    if not cache:  # plain RoPE without caches: K comes out rotated, V is not read
        qkv = torch.zeros((B, S, Nq * H), dtype=f16, device=cuda)
        kw.update(key=torch.zeros((B, S, Nkv * H), dtype=f16, device=cuda), past_seq_lens=past)
    with lib.variant("auto"):
        lib.rope_apply_qkv(qkv, c, c, None, num_heads=Nq, kv_num_heads=Nkv, rotary_embedding_dim=rd, **kw)
    torch.cuda.synchronize()
    assert lib.last_kernel() == kernel
    del qkv, kw
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", ["auto", "auto_dynamic", "simt"])
@pytest.mark.parametrize("name", [n for n, w in wl.WORKLOADS.items() if w.kind == "qkv"])
def test_qkv_workload_full_size(lib, orc, cuda, name, variant):
    """The benchmark's own shapes and launch (packed [Q|K|V], implicit positions past[b] + s,
    cache append). Q is compared whole; the written cache rows are compared with the oracle's
    rotated K and with V bit for bit; every other cache row must still hold its fill."""
    import torch

    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    x, inv, past = inp["x"], inp["inv_freq"], inp["past_seq_lens"]
    B, S, H, Nq, Nkv, L = w.batch, w.seq, w.head_size, w.num_heads, w.extra["kv_num_heads"], w.extra["max_len"]
    Ntot = Nq + 2 * Nkv
    cos, sin = orc.cache_build(inv, w.cache_rows, np.float16)
    pos = past[:, None].astype(np.int64) + np.arange(S)[None, :]
    assert pos.max() < min(L, w.cache_rows)
    q_ref, k_ref, _, _, n_oor, _ = orc.rope_qkv(x, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv)
    assert n_oor == 0
    fill = 3.0
    kc = torch.full((B, Nkv, L, H), fill, dtype=torch.float16, device=cuda)
    vc = torch.full_like(kc, fill)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    norm = bool(w.extra.get("rms_norm"))
    nkw = {}
    if norm:
        nkw = dict(q_norm_weight=inp["q_norm_weight"], k_norm_weight=inp["k_norm_weight"],
                   epsilon=w.extra["epsilon"])
        q_ref, k_ref, _, _, _, _ = orc.rope_qkv(x, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv, **nkw)
        nkw = {**nkw, "q_norm_weight": _dev(nkw["q_norm_weight"], torch, cuda),
               "k_norm_weight": _dev(nkw["k_norm_weight"], torch, cuda)}
    scratch = torch.zeros(8, dtype=torch.int64, device=cuda) if variant == "auto_dynamic" else None
    with lib.variant("simt" if variant == "simt" else "auto"):
        qo, ko = lib.rope_apply_qkv(_dev(x, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda), None,
                                    num_heads=Nq, kv_num_heads=Nkv, k_cache=kc, v_cache=vc,
                                    past_seq_lens=_dev(past, torch, cuda), status=status, scratch=scratch, **nkw)
    torch.cuda.synchronize()
    assert lib.last_kernel() == expected_qkv_kernel(variant != "simt", norm, x.nbytes, Nq, Nkv, cache=True)
    assert ko is None and int(status.item()) == 0
    none_bad = np.zeros((B, S), dtype=bool)
    bi = torch.arange(B, device=cuda)[:, None].expand(B, S)
    ri = torch.from_numpy(pos).to(cuda)
    k_rows = _host(kc[bi, :, ri].reshape(B, S, Nkv * H))
    v_rows = _host(vc[bi, :, ri].reshape(B, S, Nkv * H))
    if norm:
        compare_norm(_host(qo), q_ref, Nq, H, H, 0)
        compare_norm(k_rows, k_ref, Nkv, H, H, 0)
    else:
        compare(_host(qo), q_ref, _heads(x, B, S, 0, Nq, Ntot, H), 3, Nq,
                _token_mask(B, S, Nq, H, H, none_bad))
        compare(k_rows, k_ref, _heads(x, B, S, Nq, Nq + Nkv, Ntot, H), 3, Nkv,
                _token_mask(B, S, Nkv, H, H, none_bad))
    assert np.array_equal(v_rows.view(np.uint16), _heads(x, B, S, Nq + Nkv, Ntot, Ntot, H).view(np.uint16))
    kc[bi, :, ri] = fill
    vc[bi, :, ri] = fill
    assert bool(torch.all(kc == fill)) and bool(torch.all(vc == fill))


@pytest.mark.parametrize("variant", list(QKV_KERNELS))
@pytest.mark.parametrize("implicit", [0, 1])
def test_qkv_negative_past_lengths(lib, orc, cuda, variant, implicit):
    """A negative past length puts a batch's first cache rows below 0: those rows are
    skipped (status bit 2) -- on the pipelined kernel a tile starting below row 0 is stored
    row by row, never by a tensor store at a negative row -- and with implicit positions
    their positions are negative, so those tokens are copied through."""
    import torch

    _run_case(lib, orc, torch, cuda, "f16", 1, 1, 0, "full", implicit, H=128, Nq=16, Nkv=8, B=2, S=40, R=64,
              L=48, seed=5 + implicit, variant=variant, kernel=QKV_KERNELS[variant], past=[-21, 3])


# rope_qkv_heads_kernel's head groups: 4 heads of a role per thread from 4096 tokens on
# (16-bit RoPE), 2 below, for float32 and with QK-Norm, and a short last group where a
# role's head count is not a multiple of the width.
HEADS_SHAPES = [
    # dt, H, Nq, Nkv, S (B = 3), packed, cache, inter, rot, implicit, norm
    ("f16", 64, 8, 4, 1400, 1, 1, 0, "full", 0, 0),     # 4 per thread, 4200 tokens
    ("bf16", 64, 6, 3, 1400, 1, 1, 1, "full", 0, 0),    # 4 per thread: Q groups 4 + 2, K and V 3
    ("f16", 128, 6, 3, 37, 0, 1, 0, "full", 1, 0),      # 2 per thread, K and V groups 2 + 1
    ("f16", 64, 8, 1, 37, 1, 1, 0, "full", 0, 0),       # one K/V head
    ("f32", 64, 6, 3, 37, 1, 0, 1, "partial", 0, 0),    # float32, short group, no cache, tail units
    ("f16", 64, 6, 3, 37, 1, 1, 0, "full", 0, 1),       # QK-Norm, short group
    ("bf16", 128, 5, 1, 37, 0, 1, 1, "full", 1, 1),     # QK-Norm, odd Q heads, one K/V head
]


@pytest.mark.parametrize("dt,H,Nq,Nkv,S,packed,cache,inter,rot,implicit,norm", HEADS_SHAPES)
def test_qkv_heads_kernel_groups(lib, orc, cuda, dt, H, Nq, Nkv, S, packed, cache, inter, rot, implicit, norm):
    """Out-of-range tokens copied through, cache rows past the end skipped, every
    element against the oracle."""
    import torch

    case = (dt, H, Nq, Nkv, S, packed, cache, inter, rot, implicit, norm)
    run = _run_norm_case if norm else _run_case
    run(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H=H, Nq=Nq, Nkv=Nkv, S=S,
        seed=300 + HEADS_SHAPES.index(case), kernel="rope_qkv_heads_kernel")


def _random_qkv_cases(n, seed):
    """n seeded shapes: dtype, head size, K/V heads, group size (short head groups included),
    packing, caches, pairing, rotary width, implicit positions, QK-Norm. S in [31, 40] with
    B = 3 keeps out-of-range positions and skipped cache rows in every case."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        dt = ["f16", "bf16", "f32"][rng.integers(3)]
        H = int([32, 64, 96, 128, 256][rng.integers(5)])
        Nkv = int(rng.integers(1, 5))
        Nq = Nkv * int(rng.integers(1, 6))
        norm = bool(rng.integers(2))
        rot = "full" if norm or rng.integers(2) else "partial"
        out.append((dt, H, Nq, Nkv, int(rng.integers(31, 41)), int(rng.integers(2)), int(rng.integers(2)),
                    int(rng.integers(2)), rot, int(rng.integers(2)), norm))
    return out


RANDOM_QKV = _random_qkv_cases(24, 2024)


@pytest.mark.parametrize("variant", ["simt", "tma"])
@pytest.mark.parametrize("dt,H,Nq,Nkv,S,packed,cache,inter,rot,implicit,norm", RANDOM_QKV)
def test_qkv_random_shapes(lib, orc, cuda, dt, H, Nq, Nkv, S, packed, cache, inter, rot, implicit, norm, variant):
    """Whichever kernel the variant leads to (the heads kernel, the one-head kernel or the
    pipeline), every element against the oracle."""
    import torch

    seed = 500 + RANDOM_QKV.index((dt, H, Nq, Nkv, S, packed, cache, inter, rot, implicit, norm))
    run = _run_norm_case if norm else _run_case
    run(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H=H, Nq=Nq, Nkv=Nkv, S=S, seed=seed,
        variant=variant, kernel=None)


def test_qkv_rows_kernel_vector_path(lib, orc, cuda):
    """A token whose head groups would need more than a CTA's 512 threads (128 Q heads
    of 256 values) takes the one-head-per-thread kernel on the 128-bit path."""
    import torch

    _run_case(lib, orc, torch, cuda, "f16", 1, 1, 0, "full", 0, H=256, Nq=128, Nkv=8, S=7, L=52, seed=9,
              kernel="rope_qkv_kernel")


@pytest.mark.parametrize("dt,H", [("f16", 96), ("f16", 80), ("bf16", 96), ("f32", 48)])
@pytest.mark.parametrize("cache", [0, 1])
def test_qkv_tma_unit_counts(lib, orc, cuda, dt, H, cache):
    """Rows of 6, 5 and 6 pair units (not a power of two): the pipelined kernel without the
    norm takes them; with the norm they stay on the SIMT kernel."""
    import torch

    _run_case(lib, orc, torch, cuda, dt, 1, cache, 0, "full", 0, H=H, Nq=12, Nkv=4, B=2, S=33, L=40,
              seed=H + cache, variant="tma", kernel="rope_qkv_tma_kernel")
    _run_norm_case(lib, orc, torch, cuda, dt, 1, cache, 0, "full", 0, H=H, Nq=12, Nkv=4, B=2, S=33, L=40,
                   seed=H + cache, variant="tma", kernel="rope_qkv_kernel")


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("norm", [0, 1])
@pytest.mark.parametrize("inter", [0, 1])
def test_qkv_tma_bits_equal_simt(lib, cuda, dt, norm, inter):
    """The Q/K kernels round every value in the same order (the pipelined one on packed
    16-bit words and float32 pairs, lane by lane as the scalar code rounds), so their
    outputs agree bit for bit: Q, and every row of both caches."""
    import torch

    rng = np.random.default_rng(77 + norm + 2 * inter)
    npdt = {"f16": np.float16, "f32": np.float32, "bf16": BF16}[dt]
    B, S, Nq, Nkv, H, R, L = 2, 40, 32, 8, 128, 96, 64
    Ntot = Nq + 2 * Nkv
    qkv = cast(rng.standard_normal((B, S, Ntot * H)) * rng.uniform(0.1, 10.0, (B, S, Ntot, 1)).repeat(H, -1)
               .reshape(B, S, Ntot * H), npdt)
    theta = rng.uniform(-np.pi, np.pi, (R, H // 2))
    cos, sin = cast(np.cos(theta), npdt), cast(np.sin(theta), npdt)
    pos = rng.integers(0, R, (B, S))
    pos[0, 3], pos[1, 7] = R, -2
    past = np.array([5, 30], dtype=np.int32)
    kw = {}
    if norm:
        kw = dict(q_norm_weight=_dev(cast(rng.uniform(0.5, 2.0, H), npdt), torch, cuda),
                  k_norm_weight=_dev(cast(rng.uniform(0.5, 2.0, H), npdt), torch, cuda), epsilon=1e-6)
    kc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt)
    out = {}
    # the heads-per-thread kernel, the pipeline on both schedules and (without the norm,
    # whose sum of squares the scalar path adds in another order) the one-head-per-thread
    # kernel on the scalar path (every buffer one element off 16-byte alignment)
    runs = [("simt", False, 0, "rope_qkv_heads_kernel"), ("tma", False, 0, "rope_qkv_tma_kernel"),
            ("tma", True, 0, "rope_qkv_tma_kernel")]
    if not norm:
        runs.append(("simt", False, 1, "rope_qkv_kernel"))
    for variant, dyn, off, kernel in runs:
        dv = lambda a: _dev(a, torch, cuda, off)  # noqa: E731
        kc, vc = dv(kc0), dv(kc0)
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        scratch = torch.zeros(8, dtype=torch.int64, device=cuda) if dyn else None
        with lib.variant(variant):
            qo, _ = lib.rope_apply_qkv(dv(qkv), dv(cos), dv(sin), _dev(pos, torch, cuda), num_heads=Nq,
                                       kv_num_heads=Nkv, interleaved=inter, k_cache=kc, v_cache=vc,
                                       past_seq_lens=_dev(past, torch, cuda), status=status, scratch=scratch,
                                       q_out=dv(np.zeros((B, S, Nq * H), npdt)), **kw)
        torch.cuda.synchronize()
        assert lib.last_kernel() == kernel
        out[(variant, dyn, off)] = [_host(t) for t in (qo, kc, vc)] + [int(status.item())]
    first = out[("simt", False, 0)]
    for key in out:
        for a, b in zip(first[:3], out[key][:3]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
        assert out[key][3] == (1 | 4)


# ---------------------------------------------------------------------------
# QK-RMSNorm before the rotation (rope_apply_qkv_rmsnorm)
# ---------------------------------------------------------------------------

def _ulp(v, dtype):
    """ulp of float64 values v in storage type dtype (float16, bfloat16 bits, float32)."""
    a = np.abs(v)
    if dtype == np.float16:
        return 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -14))) - 10)
    if dtype == BF16:
        return 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7)
    return 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 23)


def compare_norm(got, ref, N, H, rd, inter):
    """Outputs of RMS-normalised, rotated heads against the oracle.

    The kernel forms r = 1/sqrt(mean(x^2) + eps) in float32 -- per-lane fused
    multiply-adds of 2V squares, a shuffle tree of at most 5 additions, the
    mean, epsilon, a correctly rounded sqrt and division: relative error at
    most about 11 units of 2^-24 (6.6e-7) -- the oracle in binary64.
      float16: that moves T(x*r) by at most one float16 ulp and T(w*T(x*r))
        (w <= 2) by at most two ulps of z; the rotation maps a change of z
        into at most |c| + |s| <= sqrt(2) times as much in the output, and
        rounds once more. Bound: 1 ulp of the result + 3 ulps of the pair's
        magnitude (which bounds |z| and which the rotation preserves). Such
        flips need x*r within 6.6e-7 of a rounding boundary (a 2^-11 grid),
        which the worst case puts at 0.3 % of the elements; r's actual error
        is far below that bound, and over every norm case here (grids, tile
        shapes, full-size workloads) at least 99.965 % of float16 and
        99.993 % of bfloat16 elements match bit for bit, so at least 99.9 %
        must.
      float32: r's error carries into z at ~1.3e-6 relative (two more
        roundings) and through the float32 rotation (one more product and
        the final rounding). Bound: 1 ulp of the result + 3e-6 of the pair's
        magnitude; no bit-exact fraction is expected."""
    assert got.shape == ref.shape and got.dtype == ref.dtype
    dtype = ref.dtype.type
    g = to_float64(got).reshape(-1, N, H)
    r = to_float64(ref).reshape(-1, N, H)
    h = rd // 2
    i0 = np.arange(h) * 2 if inter else np.arange(h)
    i1 = i0 + 1 if inter else i0 + h
    rho = np.abs(r)
    pr = np.sqrt(r[..., i0] ** 2 + r[..., i1] ** 2)
    rho[..., i0] = np.maximum(rho[..., i0], pr)
    rho[..., i1] = np.maximum(rho[..., i1], pr)
    if dtype in (np.float16, BF16):
        tol = _ulp(r, dtype) + 3 * _ulp(rho, dtype)
    else:
        tol = _ulp(r, dtype) + 3e-6 * rho
    d = np.abs(g - r)
    bad = d > tol
    assert not bad.any(), f"{int(bad.sum())} elements beyond the bound; worst excess {float((d - tol).max())}"
    exact = float((d == 0).mean())
    worst = float((d / _ulp(rho, dtype)).max()) if d.size else 0.0
    print(f"compare_norm {np.dtype(dtype).name if dtype is not BF16 else 'bfloat16'}: bit-exact {exact:.6f}, "
          f"worst {worst:.2f} ulps of the pair magnitude")
    if dtype in (np.float16, BF16):
        assert exact >= 0.999, f"only {exact:.5f} of the elements are bit-exact"
    return exact


def _run_norm_case(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H, offset=0, Nq=8, Nkv=2,
                   B=3, S=37, R=64, L=80, seed=0, eps=1e-6, variant="auto", kernel=None):
    rng = np.random.default_rng(1000 + seed)
    npdt = {"f16": np.float16, "f32": np.float32, "bf16": BF16}[dt]
    rd = 0 if rot == "full" else H // 2
    rdw = rd or H
    h = rdw // 2
    Ntot = Nq + 2 * Nkv
    qkv = cast(rng.standard_normal((B, S, Ntot * H)) * rng.uniform(0.1, 10.0, (B, S, Ntot, 1)).repeat(H, -1)
               .reshape(B, S, Ntot * H), npdt)
    q, k, v = _heads(qkv, B, S, 0, Nq, Ntot, H), _heads(qkv, B, S, Nq, Nq + Nkv, Ntot, H), \
        _heads(qkv, B, S, Nq + Nkv, Ntot, Ntot, H)
    wq = cast(rng.uniform(0.5, 2.0, H), npdt)
    wk = cast(rng.uniform(0.5, 2.0, H), npdt)
    theta = rng.uniform(-np.pi, np.pi, (R, h))
    cos, sin = cast(np.cos(theta), npdt), cast(np.sin(theta), npdt)
    past = np.array([0, 11, 50], dtype=np.int32)[:B]
    if implicit:
        pos = None
    else:
        pos = rng.integers(0, R, (B, S))
        pos[0, 5], pos[1, 0], pos[-1, -1] = R + 3, -1, R
    kc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt) if cache else None
    vc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt) if cache else None
    use_past = cache or implicit
    q_ref, k_ref, kc_ref, vc_ref, n_oor, n_skip = orc.rope_qkv(
        qkv if packed else q, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv, key=None if packed else k,
        value=None if (packed or not cache) else v, interleaved=inter, rotary_embedding_dim=rd, k_cache=kc0,
        v_cache=vc0, past_seq_lens=past if use_past else None, q_norm_weight=wq, k_norm_weight=wk, epsilon=eps)
    dv = lambda a: None if a is None else _dev(a, torch, cuda, offset)  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    kc_d, vc_d = dv(kc0), dv(vc0)
    with lib.variant(variant):
        qo, ko = lib.rope_apply_qkv(dv(qkv if packed else q), dv(cos), dv(sin),
                                    None if pos is None else _dev(pos, torch, cuda), num_heads=Nq,
                                    kv_num_heads=Nkv, key=None if packed else dv(k),
                                    value=None if (packed or not cache) else dv(v), interleaved=inter,
                                    rotary_embedding_dim=rd, k_cache=kc_d, v_cache=vc_d,
                                    past_seq_lens=_dev(past, torch, cuda) if use_past else None, status=status,
                                    q_norm_weight=dv(wq), k_norm_weight=dv(wk), epsilon=eps)
    torch.cuda.synchronize()
    if kernel is not None:
        assert lib.last_kernel() == kernel
    compare_norm(_host(qo), q_ref, Nq, H, rdw, inter)
    if not cache:
        compare_norm(_host(ko), k_ref, Nkv, H, rdw, inter)
    else:
        kc_g, vc_g = _host(kc_d), _host(vc_d)
        assert np.array_equal(vc_g.view(np.uint8), vc_ref.view(np.uint8))   # V: copies, rest untouched
        written = np.zeros((B, L), dtype=bool)
        for b in range(B):
            rows = past[b] + np.arange(S)
            written[b, rows[(rows >= 0) & (rows < L)]] = True
        # untouched K rows keep their bits; written rows within the norm bound
        assert np.array_equal(kc_g.transpose(0, 2, 1, 3)[~written].view(np.uint8),
                              kc0.transpose(0, 2, 1, 3)[~written].view(np.uint8))
        compare_norm(np.ascontiguousarray(kc_g.transpose(0, 2, 1, 3)[written]),
                     np.ascontiguousarray(kc_ref.transpose(0, 2, 1, 3)[written]), Nkv, H, rdw, inter)
    assert int(status.item()) == (1 if n_oor else 0) | (4 if n_skip else 0)


NORM_GRID = list(itertools.product(["f16", "f32", "bf16"], [0, 1], [0, 1], ["full", "partial"], [(0, 0), (1, 1)]))


@pytest.mark.parametrize("variant", list(QKV_KERNELS))
@pytest.mark.parametrize("dt,cache,inter,rot,pk_impl", NORM_GRID)
def test_qkv_rmsnorm_grid(lib, orc, cuda, dt, cache, inter, rot, pk_impl, variant):
    """Forced onto the TMA pipeline, full rotation takes it; partial rotation with the
    norm (the tail is normalised too) stays on the SIMT kernel."""
    import torch

    packed, implicit = pk_impl
    kernel = QKV_KERNELS[variant] if rot == "full" else "rope_qkv_kernel"
    _run_norm_case(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H=64,
                   seed=NORM_GRID.index((dt, cache, inter, rot, pk_impl)), variant=variant, kernel=kernel)


@pytest.mark.parametrize("dt,H,Nq,Nkv,B,S,packed,cache,inter,implicit", [
    ("f16", 128, 32, 8, 2, 40, 1, 1, 0, 1),
    ("bf16", 128, 16, 8, 3, 1, 1, 1, 1, 1),
    ("f16", 256, 8, 1, 2, 21, 0, 1, 0, 0),
    ("f32", 128, 6, 3, 2, 19, 0, 0, 1, 0),
    ("f16", 32, 12, 4, 2, 64, 1, 0, 0, 0),
])
def test_qkv_rmsnorm_tma_shapes(lib, orc, cuda, dt, H, Nq, Nkv, B, S, packed, cache, inter, implicit):
    """The pipelined norm: lane groups of 2 to 16 units, one to eight heads per tile."""
    import torch

    _run_norm_case(lib, orc, torch, cuda, dt, packed, cache, inter, "full", implicit, H=H, Nq=Nq, Nkv=Nkv, B=B,
                   S=S, L=45, seed=H + S, variant="tma", kernel="rope_qkv_tma_kernel")


@pytest.mark.parametrize("dt,H,offset,rot", [("f16", 128, 0, "full"), ("f16", 256, 0, "full"),
                                             ("f32", 128, 0, "full"), ("f16", 12, 0, "full"),
                                             ("f16", 32, 1, "full"), ("f32", 16, 1, "partial")])
def test_qkv_rmsnorm_head_sizes_and_scalar_path(lib, orc, cuda, dt, H, offset, rot):
    """Head sizes whose units fill 4 to 32 lanes, and the single-element path."""
    import torch

    _run_norm_case(lib, orc, torch, cuda, dt, 1, 1, 0, rot, 1, H=H, offset=offset, seed=H + offset)


def test_qkv_rmsnorm_zero_head_and_unsupported(lib, orc, cuda):
    """An all-zero head normalises to zeros (epsilon > 0); a head too wide for one
    32-lane group is refused before any launch."""
    import torch

    B, S, N, H = 1, 4, 2, 64
    q = torch.zeros((B, S, N * H), dtype=torch.float16, device=cuda)
    w = torch.ones(H, dtype=torch.float16, device=cuda)
    c = torch.ones((8, H // 2), dtype=torch.float16, device=cuda)
    qo, ko = lib.rope_apply_qkv(q, c, c, None, num_heads=N, kv_num_heads=N, key=q.clone(), q_norm_weight=w,
                                k_norm_weight=w)
    torch.cuda.synchronize()
    assert not qo.any() and not ko.any()
    big = torch.zeros((1, 2, 2 * 1024), dtype=torch.float16, device=cuda)
    wb = torch.ones(1024, dtype=torch.float16, device=cuda)
    cb = torch.ones((8, 512), dtype=torch.float16, device=cuda)
    with pytest.raises(lib.RopeError):
        lib.rope_apply_qkv(big, cb, cb, None, num_heads=1, kv_num_heads=1,
                           key=torch.zeros((1, 2, 1024), dtype=torch.float16, device=cuda), q_norm_weight=wb,
                           k_norm_weight=wb)


# ---------------------------------------------------------------------------
# QK-RMSNorm where r is exact: the 1-ulp bar with no allowance for r
# ---------------------------------------------------------------------------

_FOUR_SQUARES = {}


def _four_squares(R, top=15):
    """Four non-negative integers <= top whose squares add up to R, or None."""
    if R not in _FOUR_SQUARES:
        sol = None
        for a in range(top + 1):
            for b in range(a, top + 1):
                for c in range(b, top + 1):
                    d2 = R - a * a - b * b - c * c
                    if d2 < c * c:
                        break
                    d = int(round(d2 ** 0.5))
                    if d * d == d2 and d <= top:
                        sol = (a, b, c, d)
                        break
                if sol:
                    break
            if sol:
                break
        _FOUR_SQUARES[R] = sol
    return _FOUR_SQUARES[R]


def exact_mean_square_heads(rng, nheads, H):
    """`nheads` heads of H values n * 2^e (integers |n| <= 15, one e in [-8, 2] per
    head) whose squares add up to exactly 64 * H * 4^e: the mean square is the
    power of four 4^(3+e), so with epsilon 0 r = 2^-(3+e) is exact in every
    precision, and every partial sum of squares (integers times 4^e below 2^24) is
    exact in float32 as well. Returns float64 values, (nheads, H)."""
    out = np.empty((nheads, H))
    for i in range(nheads):
        while True:
            n = rng.integers(-13, 14, H - 4)
            sol = _four_squares(64 * H - int((n * n).sum()))
            if sol is not None and 64 * H - int((n * n).sum()) >= 0:
                break
        vals = np.concatenate([n, np.array(sol) * rng.choice([-1, 1], 4)]).astype(np.float64)
        rng.shuffle(vals)
        assert (vals * vals).sum() == 64 * H
        out[i] = vals * 2.0 ** int(rng.integers(-8, 3))
    return out


@pytest.mark.parametrize("variant", list(QKV_KERNELS))
@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("H,inter", [(128, 0), (64, 1)])
def test_qkv_rmsnorm_exact_r_one_ulp(lib, orc, cuda, variant, dt, H, inter):
    """Heads whose mean square is a power of four, epsilon 0: r = 1/sqrt(mean(x^2)) is
    a power of two on both sides, so the normalised z = T(w * T(x * r)) is the same
    value on the GPU and in the oracle, and what is left is the rotation's single
    rounding. Every output element -- rotated Q and K, out-of-range tokens (z copied),
    appended K rows -- within 1 ulp (float32: 1e-5) of the oracle, the copied z and V
    bit-exact. Packed [Q|K|V] with the cache append, on both Q/K kernels."""
    import torch

    rng = np.random.default_rng(77 + H + {"f16": 0, "bf16": 1, "f32": 2}[dt] + 10 * inter)
    npdt = {"f16": np.float16, "f32": np.float32, "bf16": BF16}[dt]
    B, S, Nq, Nkv, R, L = 3, 37, 8, 2, 64, 80
    Ntot = Nq + 2 * Nkv
    heads = exact_mean_square_heads(rng, B * S * Ntot, H)
    qkv = cast(heads.reshape(B, S, Ntot * H), npdt)
    assert np.array_equal(to_float64(qkv).reshape(-1, H), heads)          # the values are exact in T
    wq = cast(rng.uniform(0.5, 2.0, H), npdt)
    wk = cast(rng.uniform(0.5, 2.0, H), npdt)
    theta = rng.uniform(-np.pi, np.pi, (R, H // 2))
    cos, sin = cast(np.cos(theta), npdt), cast(np.sin(theta), npdt)
    past = np.array([0, 11, 50], dtype=np.int32)
    pos = rng.integers(0, R, (B, S))
    pos[0, 5], pos[1, 0], pos[-1, -1] = R + 3, -1, R
    bad = (pos < 0) | (pos >= R)
    kc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt)
    vc0 = cast(rng.standard_normal((B, Nkv, L, H)), npdt)
    q_ref, _, kc_ref, vc_ref, n_oor, n_skip = orc.rope_qkv(
        qkv, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv, interleaved=inter, k_cache=kc0, v_cache=vc0,
        past_seq_lens=past, q_norm_weight=wq, k_norm_weight=wk, epsilon=0.0)
    assert n_oor > 0 and n_skip > 0
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    kc_d, vc_d = _dev(kc0, torch, cuda), _dev(vc0, torch, cuda)
    with lib.variant(variant):
        qo, _ = lib.rope_apply_qkv(_dev(qkv, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda),
                                   _dev(pos, torch, cuda), num_heads=Nq, kv_num_heads=Nkv, interleaved=inter,
                                   k_cache=kc_d, v_cache=vc_d, past_seq_lens=_dev(past, torch, cuda),
                                   status=status, q_norm_weight=_dev(wq, torch, cuda),
                                   k_norm_weight=_dev(wk, torch, cuda), epsilon=0.0)
    torch.cuda.synchronize()
    assert lib.last_kernel() == QKV_KERNELS[variant]
    assert int(status.item()) == 1 | 4
    q_got = _host(qo)
    bits = np.uint32 if dt == "f32" else np.uint16
    # out-of-range tokens carry z itself: bit-exact with the oracle's z
    qg, qr = q_got.reshape(B, S, Nq, H), q_ref.reshape(B, S, Nq, H)
    assert np.array_equal(qg[bad].view(bits), qr[bad].view(bits))
    st_q = compare(q_got, q_ref, q_ref, 3, Nq)
    kc_g, vc_g = _host(kc_d), _host(vc_d)
    assert np.array_equal(vc_g.view(bits), vc_ref.view(bits))            # V rows copied, the rest untouched
    kt_g, kt_r = kc_g.transpose(0, 2, 1, 3), kc_ref.transpose(0, 2, 1, 3)  # (B, L, Nkv, H)
    st_k = compare(np.ascontiguousarray(kt_g).reshape(B, L, Nkv * H),
                   np.ascontiguousarray(kt_r).reshape(B, L, Nkv * H), kt_r.reshape(B, L, Nkv * H), 3, Nkv)
    print(f"exact-r {dt} H={H}: Q {st_q}, K cache {st_k}")
