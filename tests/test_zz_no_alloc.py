"""rope_apply_no_alloc: the RotaryEmbedding entry point for callers that cannot
allocate device memory (code inside CUDA stream capture, plugins handed only
their input and output buffers, callers without a device allocator). It takes
the dynamic tile schedule's scratch from a fixed array in the library's own
device memory instead of a caller buffer.

Checked through the C ABI against rope_apply on the same inputs, three calls in
a row (each call finds the array as the one before left it, so a counter left
behind by one call would show on the next), with the tolerance every parity
test here uses. Both cases are shapes the pipelined kernel takes (partial
rotation, 16 MiB of float16), the only kernel that uses the scratch; each call
asserts that this kernel ran. This file is collected last so that a run
stopping at the first failure has run every other test already; it also passes
alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest

from parity_util import compare, rope_passthrough_mask
from rotary_position_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _call(so, fn, x, y, cos, sin, pos, N, rd, inter, stream, scratch=None, with_scratch=False):
    xs = (ctypes.c_int64 * x.dim())(*x.shape)
    cs = (ctypes.c_int64 * cos.dim())(*cos.shape)
    args = [1, x.dim(), xs, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), cos.dim(), cs,
            ctypes.c_void_p(cos.data_ptr()), ctypes.c_void_p(sin.data_ptr()), ctypes.c_void_p(pos.data_ptr()),
            inter, rd, N, None]
    if with_scratch:
        args.append(scratch)
    args.append(ctypes.c_void_p(stream))
    return fn(*args)


@pytest.mark.parametrize("rank,inter,rd", [(3, 0, 64), (4, 1, 64)])
def test_no_alloc_matches_rope_apply(lib, orc, cuda, rank, inter, rd):
    import torch

    so = lib.load_library()
    prev = lib.get_variant()
    lib.set_variant("auto")
    try:
        rng = np.random.default_rng(41 + rank)
        B, S, N, H = 2, 1024, 32, 128           # 16 MiB of float16, partial rotation: the pipelined kernel
        shape = (B, S, N * H) if rank == 3 else (B, N, S, H)
        x = rng.standard_normal(shape).astype(np.float16)
        h = rd // 2
        R = 4096
        cos, sin = orc.cache_build(wl.inv_freq(10000.0, rd, h), R, np.float16)
        pos = rng.integers(0, R, (B, S))
        pos[1, 7] = R + 1                       # one token past the table: copied through
        nh = N if rank == 3 else 0
        y_ref, _ = orc.rope(x, cos, sin, pos, inter, rd, nh)
        xd = torch.from_numpy(x).to(cuda)
        cd, sd, pd = (torch.from_numpy(a).to(cuda) for a in (cos, sin, pos))
        stream = torch.cuda.current_stream().cuda_stream

        y_api = torch.empty_like(xd)
        assert _call(so, so.rope_apply, xd, y_api, cd, sd, pd, nh, rd, inter, stream, None, True) == 0
        assert lib.last_kernel() == "rope_tma_kernel"
        mask = rope_passthrough_mask(shape, rank, N, rd, pos, R)
        for _ in range(3):
            y_na = torch.full_like(xd, float("nan"))
            st = _call(so, so.rope_apply_no_alloc, xd, y_na, cd, sd, pd, nh, rd, inter, stream)
            assert st == 0, so.rope_last_error().decode()
            assert lib.last_kernel() == "rope_tma_kernel"   # the kernel that uses the static scratch
            torch.cuda.synchronize()
            got = y_na.cpu().numpy()
            compare(got, y_api.cpu().numpy(), x, rank, N, mask)   # against the existing entry point
            compare(got, y_ref, x, rank, N, mask)                 # and against the oracle
    finally:
        lib.set_variant(prev)
