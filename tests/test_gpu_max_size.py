"""Inputs past 2^31 elements: the kernels' element offsets must not wrap.

X holds 9 * 65536 tokens of 32 heads of 128 float16 values: 2,415,919,104
elements, 4.8 GB, and Y as much again. It is drawn on the device from a seeded
generator, and positions come from a seeded host generator. The oracle
recomputes sampled tokens one by one: the first token, the last token (the
highest addresses) and tokens spread over the whole tensor, all heads each.
The cases cover the SIMT kernel (full rotation, rank 3 and rank 4) and the TMA
pipeline (partial rotation and M-RoPE), each through the automatic variant
choice, as the benchmark launches them, the SIMT M-RoPE kernel (several heads per
thread) by the SIMT variant; and the Q/K op (RoPE on both Q/K
kernels, M-RoPE on the pipeline) over a packed [Q|K|V] of 3.2 G elements.
"""

import numpy as np
import pytest

from parity_util import compare, mrope_passthrough_mask, rope_passthrough_mask
from rotary_position_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

B, S, N, H = 9, 65536, 32, 128
R = 8192          # cos/sin table rows
SAMPLES = 48


def _sample_tokens(rng):
    idx = [(0, 0), (B - 1, S - 1), (B - 1, S - 2), (B // 2, S // 2)]
    idx += [(int(b), int(s)) for b, s in zip(rng.integers(0, B, SAMPLES), rng.integers(0, S, SAMPLES))]
    return idx


@pytest.mark.parametrize("case,kernel", [("rope_full_rank3", "rope_rows_kernel"),
                                         ("rope_full_rank4", "rope_rows_kernel"),
                                         ("rope_partial_rank3", "rope_tma_kernel"),
                                         ("mrope_rank3", "rope_tma_kernel"),
                                         ("mrope_rank3_simt", "rope_mrope_heads_kernel")])
def test_over_two_to_the_31_elements(lib, orc, cuda, case, kernel):
    import torch

    simt = case.endswith("_simt")
    case = case[:-len("_simt")] if simt else case

    assert B * S * N * H > 2 ** 31
    rank = 4 if case.endswith("rank4") else 3
    shape = (B, N, S, H) if rank == 4 else (B, S, N * H)
    rd = 64 if case == "rope_partial_rank3" else 0
    half = (rd or H) // 2
    gen = torch.Generator(device=cuda)
    gen.manual_seed(0)
    xd = torch.randn(shape, generator=gen, device=cuda, dtype=torch.float16)
    rng = np.random.default_rng(1)
    inv = wl.inv_freq(10000.0, rd or H, half)
    cos, sin = orc.cache_build(inv, R, np.float16)
    cd, sd = torch.from_numpy(cos).to(cuda), torch.from_numpy(sin).to(cuda)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    nh = N if rank == 3 else 0
    if case == "mrope_rank3":
        pos = rng.integers(0, R, (3, B, S))
        pos[1, B - 1, S - 1] = R + 5          # the last token's h stream is past the table
        section = (16, 24, 24)
        with lib.variant("simt" if simt else "auto"):
            yd = lib.mrope_apply(xd, cd, sd, torch.from_numpy(pos).to(cuda), section, mrope_layout=1,
                                 num_heads=N, oor_flag=flag)
    else:
        pos = rng.integers(0, R, (B, S))
        pos[B - 1, S - 1] = R + 5             # the last token is past the table: copied through
        yd = lib.rope_apply(xd, cd, sd, torch.from_numpy(pos).to(cuda), rotary_embedding_dim=rd,
                            num_heads=nh, oor_flag=flag)
    torch.cuda.synchronize()
    assert lib.last_kernel() == kernel
    assert int(flag.item()) == 1

    idx = _sample_tokens(rng)
    bi = torch.tensor([b for b, _ in idx], device=cuda)
    si = torch.tensor([s for _, s in idx], device=cuda)
    if rank == 3:
        xs, ys = xd[bi, si], yd[bi, si]                     # (k, N*H)
    else:
        xs = xd[bi, :, si].reshape(len(idx), N * H)         # (k, N, H) -> token rows
        ys = yd[bi, :, si].reshape(len(idx), N * H)
    x_s = xs.cpu().numpy()[None]                             # (1, k, N*H): the sampled tokens as one sequence
    y_s = ys.cpu().numpy()[None]
    if case == "mrope_rank3":
        p_s = np.stack([pos[:, b, s] for b, s in idx], axis=1)[:, None, :]   # (3, 1, k)
        y_ref, n_oor = orc.mrope(x_s, cos, sin, p_s, section, 1, 1.0, 0, 0, N)
        assert n_oor > 0
        smap = orc.mrope_stream_map(section, 1, half)
        mask = mrope_passthrough_mask(x_s.shape, 3, N, 0, p_s, R, smap, 0)
    else:
        p_s = np.array([[pos[b, s] for b, s in idx]])        # (1, k)
        y_ref, n_oor = orc.rope(x_s, cos, sin, p_s, 0, rd, N)
        assert n_oor == 1
        mask = rope_passthrough_mask(x_s.shape, 3, N, rd, p_s, R)
    compare(y_s, y_ref, x_s, 3, N, mask)
    del xd, yd
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# The Q/K op past 2^31 elements: packed [Q|K|V] of 8 x 65536 tokens x 48 heads
# of 128 float16 values (3.2 G elements, 6.4 GB), rotated K and V appended to
# (8, 8, 65536, 128) caches at rows past[b] + s with past = 0. The oracle
# recomputes sampled tokens as one packed sequence without caches: Q and K
# against it, the K cache rows against its K, the V rows bit for bit.
# ---------------------------------------------------------------------------
QB, QS, QNQ, QNKV, QH = 8, 65536, 32, 8, 128


@pytest.mark.parametrize("op,variant,kernel", [("rope", "auto", "rope_qkv_heads_kernel"),
                                               ("rope", "tma", "rope_qkv_tma_kernel"),
                                               ("mrope", "auto", "rope_qkv_tma_kernel"),
                                               ("mrope", "simt", "rope_qkv_kernel")])
def test_qkv_over_two_to_the_31_elements(lib, orc, cuda, op, variant, kernel):
    import torch

    Ntot = QNQ + 2 * QNKV
    assert QB * QS * Ntot * QH > 2 ** 31
    gen = torch.Generator(device=cuda)
    gen.manual_seed(3)
    xd = torch.randn((QB, QS, Ntot * QH), generator=gen, device=cuda, dtype=torch.float16)
    rng = np.random.default_rng(4)
    inv = wl.inv_freq(10000.0, QH, QH // 2)
    cos, sin = orc.cache_build(inv, R, np.float16)
    cd, sd = torch.from_numpy(cos).to(cuda), torch.from_numpy(sin).to(cuda)
    kc = torch.zeros((QB, QNKV, QS, QH), dtype=torch.float16, device=cuda)
    vc = torch.zeros_like(kc)
    past = torch.zeros(QB, dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    section = (16, 24, 24)
    with lib.variant(variant):
        if op == "mrope":
            pos = rng.integers(0, R, (3, QB, QS))
            pos[2, QB - 1, QS - 1] = R + 5  # the last token's w stream is past the table
            qo, ko = lib.mrope_apply_qkv(xd, cd, sd, torch.from_numpy(pos).to(cuda), section, mrope_layout=1,
                                         num_heads=QNQ, kv_num_heads=QNKV, k_cache=kc, v_cache=vc,
                                         past_seq_lens=past, status=status)
        else:
            pos = rng.integers(0, R, (QB, QS))
            pos[QB - 1, QS - 1] = R + 5       # the last token is past the table: copied through
            qo, ko = lib.rope_apply_qkv(xd, cd, sd, torch.from_numpy(pos).to(cuda), num_heads=QNQ,
                                        kv_num_heads=QNKV, k_cache=kc, v_cache=vc, past_seq_lens=past,
                                        status=status)
    torch.cuda.synchronize()
    assert lib.last_kernel() == kernel
    assert ko is None and int(status.item()) == 1

    idx = [(0, 0), (QB - 1, QS - 1), (QB - 1, QS - 2), (QB // 2, QS // 2)]
    idx += [(int(b), int(s)) for b, s in zip(rng.integers(0, QB, SAMPLES), rng.integers(0, QS, SAMPLES))]
    bi = torch.tensor([b for b, _ in idx], device=cuda)
    si = torch.tensor([s for _, s in idx], device=cuda)
    x_s = xd[bi, si].cpu().numpy()[None]                      # (1, k, Ntot*H)
    q_s = qo[bi, si].cpu().numpy()[None]                      # (1, k, Nq*H)
    k_s = kc[bi, :, si].reshape(len(idx), QNKV * QH).cpu().numpy()[None]   # rows past[b] + s = s
    v_s = vc[bi, :, si].reshape(len(idx), QNKV * QH).cpu().numpy()[None]
    xq = x_s[:, :, :QNQ * QH]
    xk = x_s[:, :, QNQ * QH:(QNQ + QNKV) * QH]
    xv = x_s[:, :, (QNQ + QNKV) * QH:]
    if op == "mrope":
        p_s = np.stack([pos[:, b, s] for b, s in idx], axis=1)[:, None, :]   # (3, 1, k)
        q_ref, k_ref, _, _, n_oor, _ = orc.mrope_qkv(x_s, cos, sin, p_s, section, 1, 1.0, num_heads=QNQ,
                                                     kv_num_heads=QNKV)
        smap = orc.mrope_stream_map(section, 1, QH // 2)
        mq = mrope_passthrough_mask(xq.shape, 3, QNQ, 0, p_s, R, smap, 0)
        mk = mrope_passthrough_mask(xk.shape, 3, QNKV, 0, p_s, R, smap, 0)
    else:
        p_s = np.array([[pos[b, s] for b, s in idx]])          # (1, k)
        q_ref, k_ref, _, _, n_oor, _ = orc.rope_qkv(x_s, cos, sin, p_s, num_heads=QNQ, kv_num_heads=QNKV)
        mq = rope_passthrough_mask(xq.shape, 3, QNQ, 0, p_s, R)
        mk = rope_passthrough_mask(xk.shape, 3, QNKV, 0, p_s, R)
    assert n_oor > 0
    compare(q_s, q_ref, xq, 3, QNQ, mq)
    compare(k_s, k_ref, xk, 3, QNKV, mk)
    assert np.array_equal(v_s.view(np.uint16), xv.view(np.uint16))
    del xd, qo, kc, vc
    torch.cuda.empty_cache()
