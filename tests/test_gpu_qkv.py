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

from parity_util import compare
from rotary_position_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TORCH_DT = {"f16": "float16", "f32": "float32"}


def _dev(a, torch, cuda, offset=0):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if offset == 0:
        return t.to(cuda)
    flat = torch.empty(t.numel() + offset, dtype=t.dtype, device=cuda)
    v = flat[offset:].view(t.shape)
    v.copy_(t.to(cuda))
    return v


def _heads(a, B, S, n0, n1, Ntot, H):
    """Heads [n0, n1) of a (B, S, Ntot*H) array as a contiguous (B, S, (n1-n0)*H) array."""
    return np.ascontiguousarray(a.reshape(B, S, Ntot, H)[:, :, n0:n1]).reshape(B, S, (n1 - n0) * H)


def _token_mask(B, S, N, H, rd, bad_tok):
    m = np.zeros((B, S, N, H), dtype=bool)
    m[..., rd:] = True
    m[bad_tok] = True
    return m


def _run_case(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H, offset=0, Nq=8, Nkv=2,
              B=3, S=37, R=64, L=80, seed=0):
    rng = np.random.default_rng(seed)
    npdt = np.float16 if dt == "f16" else np.float32
    rd = 0 if rot == "full" else H // 2
    h = (rd or H) // 2
    Ntot = Nq + 2 * Nkv
    qkv = rng.standard_normal((B, S, Ntot * H)).astype(npdt)
    q, k, v = _heads(qkv, B, S, 0, Nq, Ntot, H), _heads(qkv, B, S, Nq, Nq + Nkv, Ntot, H), \
        _heads(qkv, B, S, Nq + Nkv, Ntot, Ntot, H)
    theta = rng.uniform(-np.pi, np.pi, (R, h))
    cos, sin = np.cos(theta).astype(npdt), np.sin(theta).astype(npdt)
    past = np.array([0, 11, 50], dtype=np.int32)[:B]
    if implicit:
        pos = None
        eff = past[:, None].astype(np.int64) + np.arange(S)[None, :]
    else:
        pos = rng.integers(0, R, (B, S))
        pos[0, 5], pos[1, 0], pos[-1, -1] = R + 3, -1, R
        eff = pos
    bad_tok = (eff < 0) | (eff >= R)
    kc0 = rng.standard_normal((B, Nkv, L, H)).astype(npdt) if cache else None
    vc0 = rng.standard_normal((B, Nkv, L, H)).astype(npdt) if cache else None
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
    qo, ko = lib.rope_apply_qkv(dv(qkv if packed else q), dv(cos), dv(sin),
                                None if pos is None else _dev(pos, torch, cuda), num_heads=Nq,
                                kv_num_heads=Nkv, key=None if packed else dv(k),
                                value=None if (packed or not cache) else dv(v), interleaved=inter,
                                rotary_embedding_dim=rd, k_cache=kc_d, v_cache=vc_d,
                                past_seq_lens=_dev(past, torch, cuda) if use_past else None, status=status)
    torch.cuda.synchronize()
    assert lib.last_kernel() == "rope_qkv_kernel"
    rdw = rd or H
    compare(qo.cpu().numpy(), q_ref, q, 3, Nq, _token_mask(B, S, Nq, H, rdw, bad_tok))
    if not cache:
        assert ko is not None
        compare(ko.cpu().numpy(), k_ref, k, 3, Nkv, _token_mask(B, S, Nkv, H, rdw, bad_tok))
    else:
        assert ko is None
        # V cache: bit for bit (new rows are copies, the rest untouched)
        assert np.array_equal(vc_d.cpu().numpy().view(np.uint8), vc_ref.view(np.uint8))
        # K cache: what pass-through means per row -- the old row, or the new token's K
        src = kc0.copy()
        mask = np.ones((B, L, Nkv, H), dtype=bool)          # token-major view of (B, Nkv, L, H)
        k4 = k.reshape(B, S, Nkv, H)
        for b in range(B):
            for s in range(S):
                row = past[b] + s
                if row < L:
                    src[b, :, row] = k4[b, s]
                    mask[b, row] = False
                    mask[b, row, :, rdw:] = True
                    if bad_tok[b, s]:
                        mask[b, row] = True
        compare(kc_d.cpu().numpy(), kc_ref, src, 4, Nkv, mask)
    want = 1 | (4 if n_skip else 0)
    assert int(status.item()) == want


QKV_GRID = list(itertools.product(["f16", "f32"], [0, 1], [0, 1], [0, 1], ["full", "partial"], [0, 1]))


@pytest.mark.parametrize("dt,packed,cache,inter,rot,implicit", QKV_GRID)
def test_qkv_grid(lib, orc, cuda, dt, packed, cache, inter, rot, implicit):
    import torch

    _run_case(lib, orc, torch, cuda, dt, packed, cache, inter, rot, implicit, H=64,
              seed=QKV_GRID.index((dt, packed, cache, inter, rot, implicit)))


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
    compare(qd.cpu().numpy(), q_ref, q, 3, N, _token_mask(B, S, N, H, H, np.zeros((B, S), bool)))
    compare(kd.cpu().numpy(), k_ref, k, 3, N, _token_mask(B, S, N, H, H, np.zeros((B, S), bool)))


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


@pytest.mark.parametrize("name", [n for n, w in wl.WORKLOADS.items() if w.kind == "qkv"])
def test_qkv_workload_full_size(lib, orc, cuda, name):
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
    qo, ko = lib.rope_apply_qkv(_dev(x, torch, cuda), _dev(cos, torch, cuda), _dev(sin, torch, cuda), None,
                                num_heads=Nq, kv_num_heads=Nkv, k_cache=kc, v_cache=vc,
                                past_seq_lens=_dev(past, torch, cuda), status=status)
    torch.cuda.synchronize()
    assert ko is None and int(status.item()) == 0
    none_bad = np.zeros((B, S), dtype=bool)
    compare(qo.cpu().numpy(), q_ref, _heads(x, B, S, 0, Nq, Ntot, H), 3, Nq,
            _token_mask(B, S, Nq, H, H, none_bad))
    bi = torch.arange(B, device=cuda)[:, None].expand(B, S)
    ri = torch.from_numpy(pos).to(cuda)
    k_rows = kc[bi, :, ri].reshape(B, S, Nkv * H).cpu().numpy()
    v_rows = vc[bi, :, ri].reshape(B, S, Nkv * H).cpu().numpy()
    compare(k_rows, k_ref, _heads(x, B, S, Nq, Nq + Nkv, Ntot, H), 3, Nkv, _token_mask(B, S, Nkv, H, H, none_bad))
    assert np.array_equal(v_rows.view(np.uint16), _heads(x, B, S, Nq + Nkv, Ntot, Ntot, H).view(np.uint16))
    kc[bi, :, ri] = fill
    vc[bi, :, ri] = fill
    assert bool(torch.all(kc == fill)) and bool(torch.all(vc == fill))
