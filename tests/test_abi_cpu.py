"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/rope.h declares, and rejects malformed arguments with the
right status before any CUDA call. The host-side M-RoPE stream map is checked
against the oracle's independent construction."""

import ctypes
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rope.h")

F32, F16 = 0, 1
OK, INVALID, UNSUPPORTED = 0, 1, 2


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    fns = declared_functions()
    for name in ("rope_apply", "mrope_apply", "mrope_apply_stream_map", "mrope_stream_map",
                 "rope_apply_fused", "rope_cache_build", "rope_status_string", "rope_last_error",
                 "rope_set_variant", "rope_get_variant", "rope_last_kernel", "rope_apply_no_alloc",
                 "rope_apply_qkv", "rope_apply_qkv_rmsnorm", "mrope_apply_fused", "mrope_apply_qkv"):
        assert name in fns


def test_library_exports_every_declared_symbol(lib):
    so = lib.load_library()
    for name in declared_functions():
        assert hasattr(so, name), name
    if shutil.which("nm"):
        out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                             text=True, check=True).stdout
        exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
        assert set(declared_functions()) <= exported
    assert set(declared_functions()) == set(lib.SIGNATURES)


def _i64(*v):
    return (ctypes.c_int64 * len(v))(*v)


FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: every case fails before a CUDA call
FAKE2 = ctypes.c_void_p(0x20000)


def _rope(so, **kw):
    a = dict(dtype=F16, rank=3, xs=_i64(2, 4, 64), x=FAKE, y=FAKE2, crank=2, cs=_i64(16, 8), cos=FAKE,
             sin=FAKE, pos=FAKE, inter=0, rd=0, nh=4, flag=None, scratch=None, stream=None)
    a.update(kw)
    return so.rope_apply(a["dtype"], a["rank"], a["xs"], a["x"], a["y"], a["crank"], a["cs"], a["cos"],
                         a["sin"], a["pos"], a["inter"], a["rd"], a["nh"], a["flag"], a["scratch"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=99), UNSUPPORTED),                      # unknown element type codes
    (dict(dtype=2, nh=3), INVALID),                     # bfloat16 passes the type gate; the shape is checked
    (dict(rank=5, xs=_i64(1, 1, 1, 1, 1)), INVALID),
    (dict(nh=0), INVALID),                              # rank 3 needs num_heads
    (dict(nh=3), INVALID),                              # 64 % 3 != 0
    (dict(xs=_i64(2, 4, 60), nh=4, cs=_i64(16, 7)), INVALID),  # head size 15 is odd
    (dict(inter=2), INVALID),
    (dict(rd=-2), INVALID),
    (dict(rd=18), INVALID),                             # rd > head size 16
    (dict(rd=6), INVALID),                              # width 8 * 2 != 6
    (dict(rd=7, cs=_i64(16, 3)), INVALID),              # odd rotary width
    (dict(cs=_i64(16, 4)), INVALID),                    # width * 2 != 16
    (dict(crank=3, cs=_i64(2, 4, 8)), INVALID),         # a 3-D cache takes no position_ids
    (dict(pos=None, crank=2), INVALID),                 # a 2-D cache needs position_ids
    (dict(crank=1, cs=_i64(16)), INVALID),
    (dict(pos=None, crank=3, cs=_i64(2, 5, 8)), INVALID),   # 3-D cache must be (B, S, rd/2)
    (dict(xs=_i64(2, -1, 64)), INVALID),
    (dict(rank=4, xs=_i64(2, 4, 5, 16), nh=3), INVALID),    # num_heads != N
    (dict(x=ctypes.c_void_p(0x10001)), INVALID),        # misaligned float16 pointer
    (dict(pos=ctypes.c_void_p(0x10004)), INVALID),      # misaligned int64 pointer
    (dict(x=None), INVALID),
    (dict(scratch=ctypes.c_void_p(0x20004)), INVALID),  # misaligned scratch
])
def test_rope_apply_rejects_before_launch(lib, kw, status):
    so = lib.load_library()
    st = _rope(so, **kw)
    assert st == status, so.rope_last_error().decode()
    assert so.rope_last_error().decode() != ""


def test_empty_inputs_launch_nothing(lib):
    so = lib.load_library()
    for xs in (_i64(0, 4, 64), _i64(2, 0, 64)):
        assert _rope(so, xs=xs, x=None, y=None, cos=None, sin=None) == OK
    assert so.rope_last_error().decode() == ""


def _mrope(so, **kw):
    a = dict(dtype=F16, rank=3, xs=_i64(2, 4, 32), x=FAKE, y=FAKE2, rows=16, cos=FAKE, sin=FAKE,
             pos=FAKE, sec=(ctypes.c_int32 * 3)(2, 1, 1), layout=0, scale=1.0, inter=0, rd=0, nh=4,
             packed=0, flag=None, scratch=None, stream=None)
    a.update(kw)
    return so.mrope_apply(a["dtype"], a["rank"], a["xs"], a["x"], a["y"], a["rows"], a["cos"], a["sin"],
                          a["pos"], a["sec"], a["layout"], a["scale"], a["inter"], a["rd"], a["nh"],
                          a["packed"], a["flag"], a["scratch"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(packed=1), UNSUPPORTED),
    (dict(packed=2), INVALID),
    (dict(layout=2), INVALID),
    (dict(sec=(ctypes.c_int32 * 3)(2, 1, 2)), INVALID),     # sums to 5, rd/2 is 4
    (dict(sec=(ctypes.c_int32 * 3)(5, -1, 0)), INVALID),
    (dict(sec=None), INVALID),
    (dict(xs=_i64(2, 4, 36), nh=4), INVALID),               # head 9, rd 0 -> odd full width
    (dict(dtype=99), UNSUPPORTED),
    (dict(rows=-1), INVALID),
    (dict(pos=None), INVALID),
    (dict(xs=_i64(2, 4, 4 * 2100), rd=0, sec=(ctypes.c_int32 * 3)(1050, 0, 0)), UNSUPPORTED),
])
def test_mrope_apply_rejects_before_launch(lib, kw, status):
    so = lib.load_library()
    st = _mrope(so, **kw)
    assert st == status, so.rope_last_error().decode()


def test_mrope_odd_head_with_even_rotary_width_is_accepted_by_checks(lib):
    """Odd head size is valid when rotary_embedding_dim is a smaller even number
    (MRotaryEmbedding README, Attributes/rotary_embedding_dim); with an empty
    batch the call returns OK without launching."""
    so = lib.load_library()
    assert _mrope(so, xs=_i64(0, 4, 36), nh=4, rd=8, sec=(ctypes.c_int32 * 3)(2, 1, 1)) == OK


def test_fused_and_cache_build_reject_before_launch(lib):
    so = lib.load_library()
    st = so.rope_apply_fused(F16, 3, _i64(2, 4, 64), FAKE, FAKE2, None, 1.0, FAKE, 0, 0, 4, None)
    assert st == INVALID  # inv_freq NULL
    st = so.rope_apply_fused(F16, 3, _i64(2, 4, 64), FAKE, FAKE2, FAKE, 1.0, None, 0, 0, 4, None)
    assert st == INVALID  # positions required
    assert so.rope_cache_build(F16, FAKE, 0, 10, 1.0, FAKE, FAKE2, None) == INVALID
    assert so.rope_cache_build(F16, FAKE, 4, -1, 1.0, FAKE, FAKE2, None) == INVALID
    assert so.rope_cache_build(7, FAKE, 4, 10, 1.0, FAKE, FAKE2, None) == UNSUPPORTED
    assert so.rope_cache_build(F16, FAKE, 4, 0, 1.0, None, None, None) == OK


def test_variant_selection(lib):
    so = lib.load_library()
    assert lib.get_variant() == "auto"
    with lib.variant("tma"):
        assert so.rope_get_variant() == 2
        with lib.variant("simt"):
            assert lib.get_variant() == "simt"
        assert lib.get_variant() == "tma"
    assert lib.get_variant() == "auto"
    assert so.rope_set_variant(7) == INVALID


def test_status_strings(lib):
    so = lib.load_library()
    assert so.rope_status_string(0) == b"ROPE_OK"
    assert so.rope_status_string(3) == b"ROPE_ERR_CUDA"


def test_stream_map_matches_oracle(lib, orc):
    """The library's host map (cycle pointer) and the oracle's (round by round)
    are written independently; they must agree for layouts 0 and 1."""
    rng = np.random.default_rng(0)
    cases = [(16, 24, 24), (24, 20, 20), (2, 1, 1), (0, 0, 5), (7, 0, 3), (1, 30, 1), (64, 0, 0)]
    cases += [tuple(int(v) for v in rng.integers(0, 40, 3)) for _ in range(300)]
    for sec in cases:
        half = sum(sec)
        if half == 0:
            continue
        for layout in (0, 1):
            got = lib.mrope_stream_map(sec, layout, half)
            exp = orc.mrope_stream_map(sec, layout, half).tolist()
            assert got == exp, (sec, layout)
    with pytest.raises(lib.RopeError) as e:
        lib.mrope_stream_map((1, 2, 3), 0, 7)
    assert e.value.status == INVALID


FAKE3 = ctypes.c_void_p(0x30000)
FAKE4 = ctypes.c_void_p(0x40000)


def _qkv(so, **kw):
    a = dict(dtype=F16, B=2, S=4, nq=8, nkv=2, H=16, q=FAKE, k=FAKE2, v=None, cos=FAKE3, sin=FAKE3, rows=32,
             pos=FAKE4, past=None, inter=0, rd=0, q_out=ctypes.c_void_p(0x50000),
             k_out=ctypes.c_void_p(0x60000), kc=None, vc=None, max_len=0, flag=None, scratch=None, stream=None)
    a.update(kw)
    return so.rope_apply_qkv(a["dtype"], a["B"], a["S"], a["nq"], a["nkv"], a["H"], a["q"], a["k"], a["v"],
                             a["cos"], a["sin"], a["rows"], a["pos"], a["past"], a["inter"], a["rd"],
                             a["q_out"], a["k_out"], a["kc"], a["vc"], a["max_len"], a["flag"], a["scratch"],
                             a["stream"])


CACHE = dict(v=ctypes.c_void_p(0x70000), k_out=None, kc=ctypes.c_void_p(0x80000), vc=ctypes.c_void_p(0x90000),
             past=ctypes.c_void_p(0xa0000), max_len=64)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=99), UNSUPPORTED),
    (dict(nkv=3), INVALID),                              # kv_num_heads must divide num_heads
    (dict(nq=0), INVALID),
    (dict(nkv=0), INVALID),
    (dict(H=15), INVALID),                               # odd head size
    (dict(H=0), INVALID),
    (dict(inter=2), INVALID),
    (dict(rd=18), INVALID),
    (dict(rd=5), INVALID),
    (dict(B=-1), INVALID),
    (dict(rows=-1), INVALID),
    (dict(k=None, v=ctypes.c_void_p(0x70000)), INVALID),  # value without key
    (dict(v=ctypes.c_void_p(0x70000)), INVALID),         # value is only read in cache mode
    (dict(k_out=None), INVALID),                         # no cache and no k_out
    (dict(vc=ctypes.c_void_p(0x90000)), INVALID),        # v_cache without k_cache
    (dict(CACHE, vc=None), INVALID),                     # k_cache without v_cache
    (dict(CACHE, past=None), INVALID),                   # cache rows need past_seq_lens
    (dict(CACHE, v=None), INVALID),                      # separate inputs need value in cache mode
    (dict(CACHE, k_out=ctypes.c_void_p(0x60000)), INVALID),   # k_out and a cache
    (dict(CACHE, max_len=0), INVALID),
    (dict(k=None, q_out=FAKE), INVALID),                 # q_out aliasing a packed query
    (dict(q=ctypes.c_void_p(0x10001)), INVALID),         # misaligned float16 pointer
    (dict(pos=ctypes.c_void_p(0x40004)), INVALID),       # misaligned int64 pointer
    (dict(CACHE, past=ctypes.c_void_p(0xa0002)), INVALID),   # misaligned int32 pointer
    (dict(scratch=ctypes.c_void_p(0xd0004)), INVALID),   # scratch not 8-byte aligned
    (dict(q_out=None), INVALID),
])
def test_rope_apply_qkv_rejects_before_launch(lib, kw, status):
    so = lib.load_library()
    st = _qkv(so, **kw)
    assert st == status, so.rope_last_error().decode()
    assert so.rope_last_error().decode() != ""


def test_rope_apply_qkv_empty_launches_nothing(lib):
    so = lib.load_library()
    assert _qkv(so, S=0, q=None, k=None, q_out=None, k_out=ctypes.c_void_p(0x60000)) == OK
    assert _qkv(so, B=0) == OK


def _qkv_norm(so, **kw):
    a = dict(dtype=F16, B=2, S=4, nq=8, nkv=2, H=16, q=FAKE, k=FAKE2, v=None, qw=ctypes.c_void_p(0xb0000),
             kw_=ctypes.c_void_p(0xc0000), eps=1e-6, cos=FAKE3, sin=FAKE3, rows=32, pos=FAKE4, past=None, inter=0,
             rd=0, q_out=ctypes.c_void_p(0x50000), k_out=ctypes.c_void_p(0x60000), kc=None, vc=None, max_len=0,
             flag=None, scratch=None, stream=None)
    a.update(kw)
    return so.rope_apply_qkv_rmsnorm(a["dtype"], a["B"], a["S"], a["nq"], a["nkv"], a["H"], a["q"], a["k"],
                                     a["v"], a["qw"], a["kw_"], a["eps"], a["cos"], a["sin"], a["rows"], a["pos"],
                                     a["past"], a["inter"], a["rd"], a["q_out"], a["k_out"], a["kc"], a["vc"],
                                     a["max_len"], a["flag"], a["scratch"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(qw=None), INVALID),                            # both weights are required
    (dict(kw_=None), INVALID),
    (dict(eps=-1e-6), INVALID),
    (dict(eps=float("inf")), INVALID),
    (dict(eps=float("nan")), INVALID),
    (dict(qw=ctypes.c_void_p(0xb0001)), INVALID),        # misaligned weight
    (dict(nkv=3), INVALID),                              # the rope_apply_qkv contracts still apply
    (dict(H=1024, rows=32), UNSUPPORTED),                # 64 units of 16 bytes: more than one 32-lane group
    (dict(H=64, rd=32, q=ctypes.c_void_p(0x10002)), UNSUPPORTED),  # scalar path: 16 pairs + 32 tail elements
])
def test_rope_apply_qkv_rmsnorm_rejects_before_launch(lib, kw, status):
    so = lib.load_library()
    st = _qkv_norm(so, **kw)
    assert st == status, so.rope_last_error().decode()
    assert so.rope_last_error().decode() != ""


def _mrope_fused(so, **kw):
    a = dict(dtype=F16, rank=3, xs=_i64(2, 4, 32), x=FAKE, y=FAKE2, inv=FAKE3, scaling=1.0, pos=FAKE4,
             sec=(ctypes.c_int32 * 3)(2, 1, 1), layout=0, scale=1.0, inter=0, rd=0, nh=4, stream=None)
    a.update(kw)
    return so.mrope_apply_fused(a["dtype"], a["rank"], a["xs"], a["x"], a["y"], a["inv"], a["scaling"], a["pos"],
                                a["sec"], a["layout"], a["scale"], a["inter"], a["rd"], a["nh"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=99), UNSUPPORTED),
    (dict(sec=None), INVALID),
    (dict(sec=(ctypes.c_int32 * 3)(2, 2, 1)), INVALID),     # sections must sum to rd/2 = 4
    (dict(sec=(ctypes.c_int32 * 3)(5, -1, 0)), INVALID),
    (dict(layout=2), INVALID),
    (dict(inter=3), INVALID),
    (dict(nh=3), INVALID),
    (dict(pos=None), INVALID),
    (dict(inv=ctypes.c_void_p(0x30002)), INVALID),           # misaligned float32 inv_freq
    (dict(x=None), INVALID),
])
def test_mrope_apply_fused_rejects_before_launch(lib, kw, status):
    so = lib.load_library()
    st = _mrope_fused(so, **kw)
    assert st == status, so.rope_last_error().decode()
    assert so.rope_last_error().decode() != ""


def _mqkv(so, **kw):
    a = dict(dtype=F16, B=2, S=4, nq=8, nkv=2, H=16, q=FAKE, k=FAKE2, v=None, qw=None, kw_=None, eps=1e-6,
             cos=FAKE3, sin=FAKE3, rows=32, pos=FAKE4, sec=(2, 3, 3), layout=1, scale=1.0, past=None, inter=0,
             rd=0, q_out=ctypes.c_void_p(0x50000), k_out=ctypes.c_void_p(0x60000), kc=None, vc=None, max_len=0,
             flag=None, scratch=None, stream=None)
    a.update(kw)
    sec = None if a["sec"] is None else (ctypes.c_int32 * 3)(*a["sec"])
    return so.mrope_apply_qkv(a["dtype"], a["B"], a["S"], a["nq"], a["nkv"], a["H"], a["q"], a["k"], a["v"],
                              a["qw"], a["kw_"], a["eps"], a["cos"], a["sin"], a["rows"], a["pos"], sec,
                              a["layout"], a["scale"], a["past"], a["inter"], a["rd"], a["q_out"], a["k_out"],
                              a["kc"], a["vc"], a["max_len"], a["flag"], a["scratch"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(sec=None), INVALID),                           # the section is required
    (dict(pos=None), INVALID),                           # so are the three position streams
    (dict(sec=(2, 3, 2)), INVALID),                      # sections must sum to rd/2
    (dict(sec=(-1, 5, 4)), INVALID),
    (dict(layout=2), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(qw=ctypes.c_void_p(0xb0000)), INVALID),        # a norm needs both weights
    (dict(nkv=3), INVALID),                              # the rope_apply_qkv contract still holds
    (dict(H=15), INVALID),
    (dict(rd=8, sec=(2, 3, 3)), INVALID),                # rd 8: sections must sum to 4
    (dict(pos=ctypes.c_void_p(0x40004)), INVALID),       # misaligned int64 positions
    (dict(dtype=99), UNSUPPORTED),
])
def test_mrope_apply_qkv_rejects_before_launch(lib, kw, status):
    so = lib.load_library()
    st = _mqkv(so, **kw)
    assert st == status, so.rope_last_error().decode()
    assert so.rope_last_error().decode() != ""


def test_mrope_apply_qkv_empty_launches_nothing(lib):
    so = lib.load_library()
    assert _mqkv(so, B=0, pos=None) == OK
    assert _mqkv(so, S=0, pos=None, q=None, k=None, q_out=None) == OK
