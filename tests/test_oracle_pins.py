"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- an independent library routine, a hand-worked example, exact
rational arithmetic, a closed form, an invariant, or a brute-force matrix
formulation -- so that a dropped term, a wrong sign, a wrong index or a
transposed operand in the oracle fails at least one of them.

Sources cited by page title and section:
  RotaryEmbedding manifest  -- "ai.onnx.RotaryEmbedding" WebGPU manifest.json
  MRotaryEmbedding README   -- "com.microsoft.MRotaryEmbedding" README
  Qwen3 fusion PR           -- onnxruntime PR "Add RotaryEmbedding fusion for
                               Qwen3 on-the-fly RoPE patterns"
"""

import itertools
import json
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest

from rotary_position_embedding_gb300 import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# binary16 conversion against numpy's independent implementation
# --------------------------------------------------------------------------

def test_half_to_double_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros and infinities keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_double_to_half_midpoints_and_random(orc):
    finite = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (finite[:-1] + finite[1:]) / 2.0          # every tie point (exact in binary64)
    rng = np.random.default_rng(7)
    rand = rng.standard_normal(20000) * np.exp2(rng.integers(-30, 17, 20000))
    edge = np.array([65504.0, 65519.999, 65520.0, 70000.0, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001,
                     2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12), 0.0])
    vals = np.concatenate([mids, -mids, finite, rand, edge, -edge, np.nextafter(mids, 0),
                           np.nextafter(mids, np.inf)])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.double_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# hand-worked example (Qwen3 fusion PR, apply_rotary_pos_emb / rotate_half)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_hand_example(orc, dtype):
    g = _gold("hand_example.json")
    x = np.array(g["x"], dtype=dtype).reshape(1, 1, g["head_size"])
    for case in g["cases"]:
        c = np.array(case["cos"], dtype=dtype).reshape(1, -1)
        s = np.array(case["sin"], dtype=dtype).reshape(1, -1)
        pos = np.zeros((1, 1), dtype=np.int64)
        y, n_oor = orc.rope(x, c, s, pos, case["interleaved"], case["rotary_embedding_dim"], 1)
        assert n_oor == 0
        assert y.ravel().tolist() == case["y"], case["name"]
        # the same head as rank 4 (B, N, S, H) = (1, 1, 1, 4)
        y4, _ = orc.rope(x.reshape(1, 1, 1, -1), c, s, pos, case["interleaved"],
                         case["rotary_embedding_dim"])
        assert y4.ravel().tolist() == case["y"], case["name"]


# --------------------------------------------------------------------------
# the printed half-split form: x*cat(c,c) + rotate_half(x)*cat(s,s)
# --------------------------------------------------------------------------

def _rotate_half_form(x, c, s):
    """The Qwen3 fusion PR's modelling form, for one (..., H) block in binary64."""
    h = x.shape[-1] // 2
    cc = np.concatenate([c, c], axis=-1)
    ss = np.concatenate([s, s], axis=-1)
    rh = np.concatenate([-x[..., h:], x[..., :h]], axis=-1)
    return x * cc + rh * ss


def test_half_split_matches_rotate_half_form_fp32(orc):
    rng = np.random.default_rng(11)
    B, S, N, H = 2, 5, 3, 16
    x = rng.standard_normal((B, S, N * H)).astype(np.float32)
    rows = 9
    cos = rng.uniform(-1, 1, (rows, H // 2)).astype(np.float32)
    sin = rng.uniform(-1, 1, (rows, H // 2)).astype(np.float32)
    pos = rng.integers(0, rows, (B, S))
    y, _ = orc.rope(x, cos, sin, pos, 0, 0, N)
    xd = x.astype(np.float64).reshape(B, S, N, H)
    c = cos.astype(np.float64)[pos][:, :, None, :]
    s = sin.astype(np.float64)[pos][:, :, None, :]
    ref = _rotate_half_form(xd, c, s).astype(np.float32)
    assert np.array_equal(y.reshape(B, S, N, H), ref)


# --------------------------------------------------------------------------
# exact rational arithmetic: fp16 outputs are the correctly rounded result
# --------------------------------------------------------------------------

def _round_half_exact(q: Fraction):
    """Nearest float16 to the exact rational q, ties to even (no binary64 step)."""
    f = float(q)
    lo = np.float16(f)
    cands = {float(lo)}
    for d in (np.inf, -np.inf):
        cands.add(float(np.nextafter(lo, np.float16(d))))
    best = None
    for cnd in sorted(cands):
        if not np.isfinite(cnd):
            continue
        err = abs(Fraction(cnd) - q)
        even = (int(np.float16(cnd).view(np.uint16)) & 1) == 0
        key = (err, not even)
        if best is None or key < best[0]:
            best = (key, cnd)
    return best[1]


def test_fp16_rotation_is_correctly_rounded(orc):
    rng = np.random.default_rng(3)
    B, S, N, H = 1, 4, 2, 8
    x = (rng.standard_normal((B, S, N * H)) * 3).astype(np.float16)
    cos = rng.uniform(-1, 1, (S, H // 2)).astype(np.float16)
    sin = rng.uniform(-1, 1, (S, H // 2)).astype(np.float16)
    pos = np.arange(S)[None, :]
    for inter in (0, 1):
        y, _ = orc.rope(x, cos, sin, pos, inter, 0, N)
        xr = x.reshape(S, N, H)
        yr = y.reshape(S, N, H)
        h = H // 2
        for s_, n, i in itertools.product(range(S), range(N), range(h)):
            j0, j1 = (2 * i, 2 * i + 1) if inter else (i, i + h)
            x0, x1 = Fraction(float(xr[s_, n, j0])), Fraction(float(xr[s_, n, j1]))
            c, s = Fraction(float(cos[s_, i])), Fraction(float(sin[s_, i]))
            assert float(yr[s_, n, j0]) == _round_half_exact(x0 * c - x1 * s)
            assert float(yr[s_, n, j1]) == _round_half_exact(x1 * c + x0 * s)


# --------------------------------------------------------------------------
# closed forms and invariants
# --------------------------------------------------------------------------

def test_complex_multiply_closed_form(orc):
    """Each pair is (x0 + i x1) * (c + i s); fp32 outputs round that product once."""
    rng = np.random.default_rng(5)
    B, N, S, H = 2, 3, 6, 12
    x = rng.standard_normal((B, N, S, H)).astype(np.float32)
    theta = rng.uniform(-np.pi, np.pi, (B, S, H // 2))
    cos = np.cos(theta).astype(np.float32)
    sin = np.sin(theta).astype(np.float32)
    for inter in (0, 1):
        y, _ = orc.rope(x, cos, sin, None, inter, 0)
        h = H // 2
        idx0 = np.arange(h) * 2 if inter else np.arange(h)
        idx1 = idx0 + 1 if inter else idx0 + h
        z = x[..., idx0].astype(np.complex128) + 1j * x[..., idx1].astype(np.complex128)
        w = cos.astype(np.float64)[:, None, :, :] + 1j * sin.astype(np.float64)[:, None, :, :]
        prod = z * w
        assert np.array_equal(y[..., idx0], prod.real.astype(np.float32))
        assert np.array_equal(y[..., idx1], prod.imag.astype(np.float32))


def test_norm_preserved_when_unit_coefficients(orc):
    rng = np.random.default_rng(6)
    B, S, N, H = 2, 7, 4, 32
    x = rng.standard_normal((B, S, N * H)).astype(np.float32)
    theta = rng.uniform(0, 2 * np.pi, (B, S, H // 2))
    cos, sin = np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)
    y, _ = orc.rope(x, cos, sin, None, 0, 0, N)
    xr, yr = x.reshape(B, S, N, H).astype(np.float64), y.reshape(B, S, N, H).astype(np.float64)
    h = H // 2
    nx = xr[..., :h] ** 2 + xr[..., h:] ** 2
    ny = yr[..., :h] ** 2 + yr[..., h:] ** 2
    assert np.allclose(ny, nx, rtol=8 * 2.0 ** -24, atol=1e-12)


def test_identity_at_position_zero(orc):
    rng = np.random.default_rng(8)
    for dtype in (np.float16, np.float32):
        x = rng.standard_normal((2, 3, 4, 16)).astype(dtype)
        x[x == 0] = 1  # no signed zeros: -0 + x*0 may give +0
        cos = np.ones((5, 8), dtype=dtype)
        sin = np.zeros((5, 8), dtype=dtype)
        pos = np.zeros((2, 4), dtype=np.int64)
        for inter in (0, 1):
            y, _ = orc.rope(x, cos, sin, pos, inter, 0)
            assert np.array_equal(y.view(np.uint8), x.view(np.uint8))


def test_interleaved_is_permuted_half_split(orc):
    """interleaved(P x) == P half_split(x), P: i -> 2i, i + rd/2 -> 2i + 1 (tail fixed)."""
    rng = np.random.default_rng(9)
    for dtype, rd in itertools.product((np.float16, np.float32), (0, 8)):
        B, S, N, H = 2, 5, 3, 12
        rdv = rd or H
        h = rdv // 2
        x = rng.standard_normal((B, S, N * H)).astype(dtype)
        cos = rng.uniform(-1, 1, (11, h)).astype(dtype)
        sin = rng.uniform(-1, 1, (11, h)).astype(dtype)
        pos = rng.integers(0, 11, (B, S))
        perm = np.arange(H)
        perm[2 * np.arange(h)] = np.arange(h)
        perm[2 * np.arange(h) + 1] = np.arange(h) + h
        # perm[k] = index in half-split layout of element k of the interleaved layout
        xh = x.reshape(B, S, N, H)
        xi = xh[..., perm]
        yh, _ = orc.rope(x, cos, sin, pos, 0, rd, N)
        yi, _ = orc.rope(xi.reshape(B, S, N * H), cos, sin, pos, 1, rd, N)
        lhs = yi.reshape(B, S, N, H)
        rhs = np.ascontiguousarray(yh.reshape(B, S, N, H)[..., perm])
        assert np.array_equal(lhs.view(np.uint8), rhs.view(np.uint8))


def test_tail_is_bit_copy_and_rank3_equals_rank4(orc):
    rng = np.random.default_rng(10)
    B, S, N, H, rd = 2, 6, 3, 20, 8
    for dtype in (np.float16, np.float32):
        x3 = rng.standard_normal((B, S, N * H)).astype(dtype)
        cos = rng.uniform(-1, 1, (13, rd // 2)).astype(dtype)
        sin = rng.uniform(-1, 1, (13, rd // 2)).astype(dtype)
        pos = rng.integers(0, 13, (B, S))
        for inter in (0, 1):
            y3, _ = orc.rope(x3, cos, sin, pos, inter, rd, N)
            assert np.array_equal(y3.reshape(B, S, N, H)[..., rd:].view(np.uint8),
                                  x3.reshape(B, S, N, H)[..., rd:].view(np.uint8))
            x4 = np.ascontiguousarray(x3.reshape(B, S, N, H).transpose(0, 2, 1, 3))
            y4, _ = orc.rope(x4, cos, sin, pos, inter, rd)
            assert np.array_equal(y4.transpose(0, 2, 1, 3).view(np.uint8),
                                  y3.reshape(B, S, N, H).view(np.uint8))


def test_cache3d_equals_gather(orc):
    """Without position_ids row (b, s) of a (B, S, rd/2) table is used: the same as
    gathering a 2-D table at the token's own index."""
    rng = np.random.default_rng(12)
    B, S, N, H = 3, 4, 2, 8
    x = rng.standard_normal((B, N, S, H)).astype(np.float32)
    cos = rng.uniform(-1, 1, (B, S, H // 2)).astype(np.float32)
    sin = rng.uniform(-1, 1, (B, S, H // 2)).astype(np.float32)
    y3d, _ = orc.rope(x, cos, sin, None, 0, 0)
    pos = np.arange(B * S).reshape(B, S)
    y2d, _ = orc.rope(x, cos.reshape(B * S, -1), sin.reshape(B * S, -1), pos, 0, 0)
    assert np.array_equal(y3d, y2d)


def test_rope_out_of_range_token_copies_through(orc):
    rng = np.random.default_rng(13)
    B, S, N, H, R = 2, 8, 2, 8, 5
    x = rng.standard_normal((B, S, N * H)).astype(np.float16)
    cos = rng.uniform(-1, 1, (R, H // 2)).astype(np.float16)
    sin = rng.uniform(-1, 1, (R, H // 2)).astype(np.float16)
    pos = rng.integers(0, R, (B, S))
    pos[0, 1], pos[1, 5], pos[1, 6] = -1, R, 1 << 40
    y, n = orc.rope(x, cos, sin, pos, 0, 0, N)
    assert n == 3
    bad = (pos < 0) | (pos >= R)
    assert np.array_equal(y[bad].view(np.uint16), x[bad].view(np.uint16))
    assert not np.array_equal(y[~bad], x[~bad])


# --------------------------------------------------------------------------
# M-RoPE: stream maps, reductions, out-of-range pairs, brute force
# --------------------------------------------------------------------------

def test_stream_maps_readme_and_counts(orc):
    g = _gold("mrope_readme_example.json")
    assert orc.mrope_stream_map(g["mrope_section"], 0, 4).tolist() == g["stream_map_layout0"]
    assert orc.mrope_stream_map(g["mrope_section"], 1, 4).tolist() == g["stream_map_layout1"]
    assert orc.mrope_stream_map(g["mrope_section"], 2, 4).tolist() == g["stream_map_layout1"]
    m1 = orc.mrope_stream_map([16, 24, 24], 1, 64)
    assert np.bincount(m1, minlength=3).tolist() == [16, 24, 24]
    assert m1[:48].tolist() == [0, 1, 2] * 16 and m1[48:].tolist() == [1, 2] * 8
    m2 = orc.mrope_stream_map([16, 24, 24], 2, 64)
    assert np.bincount(m2, minlength=3).tolist() == g["section_16_24_24_layout1_stride3_counts"]
    a = orc.mrope_stream_map([24, 20, 20], 1, 64)
    b = orc.mrope_stream_map([24, 20, 20], 2, 64)
    assert np.array_equal(a, b)
    assert np.bincount(a, minlength=3).tolist() == g["section_24_20_20_layout1_counts"]
    rng = np.random.default_rng(14)
    for _ in range(200):
        sec = rng.integers(0, 20, 3)
        half = int(sec.sum())
        if half == 0:
            continue
        for layout in (0, 1):
            m = orc.mrope_stream_map(sec, layout, half)
            assert np.bincount(m, minlength=3).tolist() == sec.tolist()
        m0 = orc.mrope_stream_map(sec, 0, half)
        assert np.all(np.diff(m0.astype(int)) >= 0)  # chunked: t block, h block, w block
    with pytest.raises(ValueError):
        orc.mrope_stream_map([1, 2, 3], 0, 7)


def test_mrope_equal_streams_reduce_to_rope(orc):
    rng = np.random.default_rng(15)
    B, S, N, H, R = 2, 9, 3, 16, 20
    for dtype, inter, rd in itertools.product((np.float16, np.float32), (0, 1), (0, 8)):
        h = (rd or H) // 2
        x = rng.standard_normal((B, S, N * H)).astype(dtype)
        cos = rng.uniform(-1, 1, (R, h)).astype(dtype)
        sin = rng.uniform(-1, 1, (R, h)).astype(dtype)
        p = rng.integers(0, R, (B, S))
        pos3 = np.stack([p, p, p])
        sec = [h - 2 * (h // 3), h // 3, h // 3]
        yr, _ = orc.rope(x, cos, sin, p, inter, rd, N)
        for layout in (0, 1, 2):
            m = orc.mrope_stream_map(sec, layout, h)
            ym, n = orc.mrope_map(x, cos, sin, pos3, m, 1.0, inter, rd, N)
            assert n == 0
            assert np.array_equal(ym.view(np.uint8), yr.view(np.uint8))


def test_mrope_single_section_uses_only_t(orc):
    rng = np.random.default_rng(16)
    B, S, N, H, R = 2, 5, 2, 8, 9
    x = rng.standard_normal((B, S, N * H)).astype(np.float16)
    cos = rng.uniform(-1, 1, (R, 4)).astype(np.float16)
    sin = rng.uniform(-1, 1, (R, 4)).astype(np.float16)
    t = rng.integers(0, R, (B, S))
    junk = rng.integers(-5, 2 * R, (2, B, S))
    y, n = orc.mrope(x, cos, sin, np.concatenate([t[None], junk]), [4, 0, 0], 0, 1.0, 0, 0, N)
    yr, _ = orc.rope(x, cos, sin, t, 0, 0, N)
    assert n == 0 and np.array_equal(y.view(np.uint16), yr.view(np.uint16))


def _brute_mrope(x, cos, sin, pos3, smap, scale, inter, N, dtype):
    """Per (token, head): build the H x H block-rotation matrix and apply it in binary64."""
    B, S, HN = x.shape
    H = HN // N
    h = len(smap)
    R = cos.shape[0]
    out = np.empty((B, S, N, H), dtype=np.float64)
    xr = x.reshape(B, S, N, H).astype(np.float64)
    keep = np.zeros((B, S, N, H), dtype=bool)

    def rnd(v):
        return float(np.asarray(v, dtype=np.float64).astype(dtype))

    for b, s in itertools.product(range(B), range(S)):
        M = np.eye(H)
        k = np.zeros(H, dtype=bool)
        for i in range(h):
            p = int(pos3[smap[i], b, s])
            j0, j1 = (2 * i, 2 * i + 1) if inter else (i, i + h)
            if p < 0 or p >= R:
                k[j0] = k[j1] = True
                continue
            c = rnd(float(cos[p, i]) * scale)
            sn = rnd(float(sin[p, i]) * scale)
            M[j0, j0], M[j0, j1], M[j1, j0], M[j1, j1] = c, -sn, sn, c
        for n in range(N):
            out[b, s, n] = M @ xr[b, s, n]
            keep[b, s, n] = k
    return out, keep


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("inter", [0, 1])
def test_mrope_brute_force_readme_shape(orc, layout, inter):
    """README example shape; every (t, h, w) combination of {-1, 0, 1, 2} over R = 2 rows."""
    g = _gold("mrope_readme_example.json")
    B, S, HN = g["x_shape"]
    N = g["num_heads"]
    R, h = g["cache_shape"]
    smap = g["stream_map_layout0" if layout == 0 else "stream_map_layout1"]
    rng = np.random.default_rng(17)
    combos = list(itertools.product([-1, 0, 1, 2], repeat=3))
    scale = 0.8125
    for dtype in (np.float16, np.float32):
        cos = rng.uniform(-1, 1, (R, h)).astype(dtype)
        sin = rng.uniform(-1, 1, (R, h)).astype(dtype)
        for start in range(0, len(combos), B * S):
            chunk = combos[start:start + B * S]
            chunk = chunk + [(0, 0, 0)] * (B * S - len(chunk))
            pos3 = np.array(chunk, dtype=np.int64).T.reshape(3, B, S)
            x = rng.standard_normal((B, S, HN)).astype(dtype)
            y, n = orc.mrope(x, cos, sin, pos3, g["mrope_section"], layout, scale, inter, 0, N)
            ref, keep = _brute_mrope(x, cos, sin, pos3, smap, scale, inter, N, dtype)
            yr = y.reshape(B, S, N, -1)
            xr = x.reshape(B, S, N, -1)
            assert n == int(keep.sum()) // 2
            assert np.array_equal(yr[keep].view(np.uint8), xr[keep].view(np.uint8))
            assert np.array_equal(yr[~keep], ref[~keep].astype(dtype))


def test_mrope_scale_rounds_coefficient_to_storage_type(orc):
    """The scaled coefficient is rounded to T before the rotation (README,
    Implementation variants/pairs4): with x = (1, 0) the output is exactly
    (T(c*scale), T(s*scale))."""
    for dtype in (np.float16, np.float32):
        rng = np.random.default_rng(18)
        R, h = 7, 6
        cos = rng.uniform(-1, 1, (R, h)).astype(dtype)
        sin = rng.uniform(-1, 1, (R, h)).astype(dtype)
        x = np.zeros((1, R, 2 * h), dtype=dtype)
        x[..., :h] = 1
        pos3 = np.tile(np.arange(R)[None, None, :], (3, 1, 1))
        scale = float(np.float32(0.3))   # the attribute is a float32
        y, _ = orc.mrope(x, cos, sin, pos3, [h, 0, 0], 0, scale, 0, 0, 1)
        exp_c = np.array([[Fraction(float(v)) * Fraction(scale) for v in row] for row in cos])
        exp_s = np.array([[Fraction(float(v)) * Fraction(scale) for v in row] for row in sin])
        for p in range(R):
            for i in range(h):
                if dtype == np.float16:
                    rc, rs = _round_half_exact(exp_c[p, i]), _round_half_exact(exp_s[p, i])
                else:
                    rc = float(np.float32(float(exp_c[p, i])))  # binary64 product is exact here
                    rs = float(np.float32(float(exp_s[p, i])))
                assert float(y[0, p, i]) == rc and float(y[0, p, h + i]) == rs


# --------------------------------------------------------------------------
# cache build and the on-the-fly variant
# --------------------------------------------------------------------------

def _fl32(v):
    return float(np.float32(v))


def test_cache_spot_positions_against_high_precision(orc):
    """Qwen3 fusion PR, numerical validation: cache[p] = cos(p*inv)*scaling at
    p in {0, 1, 7, 100, 1000}; checked against 60-digit mpmath on the float32
    angle, so each float32 cos/sin is the correctly rounded value."""
    g = _gold("cache_spot_positions.json")
    mpmath.mp.dps = 60
    half = g["head_dim"] // 2
    for base, scaling in itertools.product(g["bases"], g["scalings"]):
        inv = wl.inv_freq(base, g["head_dim"], half)
        rows = max(g["positions"]) + 1
        c32, s32 = orc.cache_build(inv, rows, np.float32, scaling)
        c16, s16 = orc.cache_build(inv, rows, np.float16, scaling)
        for p in g["positions"]:
            for i in range(half):
                theta = np.float32(np.float32(p) * inv[i])
                ce = mpmath.cos(mpmath.mpf(float(theta)))
                se = mpmath.sin(mpmath.mpf(float(theta)))
                with mpmath.workprec(24):     # round the 60-digit value straight to 24 bits
                    cr, sr = float(+ce), float(+se)
                exp_c = np.float32(np.float32(cr) * np.float32(scaling))
                exp_s = np.float32(np.float32(sr) * np.float32(scaling))
                assert c32[p, i] == exp_c and s32[p, i] == exp_s, (base, scaling, p, i)
                assert c16[p, i] == exp_c.astype(np.float16) and s16[p, i] == exp_s.astype(np.float16)
        # position 0 is the identity rotation scaled: cos = scaling, sin = 0
        assert np.all(c32[0] == np.float32(scaling)) and np.all(s32[0] == 0)


def test_fused_equals_cached(orc):
    """On-the-fly coefficients equal gathering the built cache (Qwen3 fusion PR)."""
    rng = np.random.default_rng(19)
    for dtype, inter, rd, rank in itertools.product((np.float16, np.float32), (0, 1), (0, 16), (3, 4)):
        B, S, N, H = 2, 6, 3, 32
        rdv = rd or H
        shape = (B, S, N * H) if rank == 3 else (B, N, S, H)
        x = rng.standard_normal(shape).astype(dtype)
        inv = wl.inv_freq(1e6, rdv, rdv // 2)
        R = 300
        pos = rng.integers(0, R, (B, S))
        cos, sin = orc.cache_build(inv, R, dtype, 0.9)
        yc, _ = orc.rope(x, cos, sin, pos, inter, rd, N if rank == 3 else 0)
        yf = orc.rope_fused(x, inv, pos, 0.9, inter, rd, N if rank == 3 else 0)
        assert np.array_equal(yc.view(np.uint8), yf.view(np.uint8))


def test_workload_inputs_are_seeded():
    w = wl.WORKLOADS["mrope_r3_f16_layout1"].with_shape(S=8192, B=1)
    a = wl.make_inputs(w)
    b = wl.make_inputs(w)
    assert np.array_equal(a["x"], b["x"]) and np.array_equal(a["position_ids"], b["position_ids"])
    pos = a["position_ids"]
    oor = pos >= w.cache_rows
    assert abs(oor.mean() - 0.01) < 0.002
    assert pos.min() >= 0
    # text spans have t == h == w (away from the ids moved past the cache)
    text = ~oor[:, 0, :1000].any(axis=0)
    assert np.all(pos[0, 0, :1000][text] == pos[1, 0, :1000][text])
    assert np.all(pos[0, 0, :1000][text] == pos[2, 0, :1000][text])


# --------------------------------------------------------------------------
# Q and K rotation with grouped-query heads and the key/value cache append
# (SparseAttention README: Description, Inputs, Attributes do_rotary and
# kv_num_heads; Qwen3 fusion PR: Verification, Qwen3 Architecture)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_qkv_hand_example_gqa(orc, dtype):
    g = _gold("qkv_hand_example.json")
    Nq, Nkv, H = g["num_heads"], g["kv_num_heads"], g["head_size"]
    q = np.array(g["q"], dtype=dtype).reshape(1, 1, Nq * H)
    k = np.array(g["k"], dtype=dtype).reshape(1, 1, Nkv * H)
    v = np.array(g["v"], dtype=dtype).reshape(1, 1, Nkv * H)
    cos, sin = np.array(g["cos"], dtype=dtype), np.array(g["sin"], dtype=dtype)
    L = g["max_cache_len"]
    fill = np.full((1, Nkv, L, H), g["cache_fill"], dtype=dtype)
    past = np.array([g["past"]], dtype=np.int32)
    for case in g["cases"]:
        inter = case["interleaved"]
        # explicit position, no cache
        qo, ko, _, _, n_oor, _ = orc.rope_qkv(q, cos, sin, np.array([[g["past"]]]), num_heads=Nq,
                                              kv_num_heads=Nkv, key=k, interleaved=inter)
        assert n_oor == 0
        assert qo.ravel().tolist() == case["q_out"] and ko.ravel().tolist() == case["k_out"]
        # cache mode, implicit position past + s, separate and packed inputs
        packed = np.concatenate([q, k, v], axis=-1)
        for kw in (dict(key=k, value=v), dict()):
            src = q if kw else packed
            qo, ko, kc, vc, _, n_skip = orc.rope_qkv(src, cos, sin, None, num_heads=Nq, kv_num_heads=Nkv,
                                                    interleaved=inter, k_cache=fill, v_cache=fill,
                                                    past_seq_lens=past, **kw)
            assert ko is None and n_skip == 0
            assert qo.ravel().tolist() == case["q_out"]
            assert kc[0, 0, 1].tolist() == case["k_out"] and vc[0, 0, 1].tolist() == g["v"]
            for row in (0, 2):
                assert (kc[0, 0, row] == g["cache_fill"]).all() and (vc[0, 0, row] == g["cache_fill"]).all()


def _qkv_inputs(rng, dtype, B=3, S=5, Nq=6, Nkv=2, H=16, R=40):
    q = rng.standard_normal((B, S, Nq * H)).astype(dtype)
    k = rng.standard_normal((B, S, Nkv * H)).astype(dtype)
    v = rng.standard_normal((B, S, Nkv * H)).astype(dtype)
    theta = rng.uniform(-np.pi, np.pi, (R, H // 2))
    return q, k, v, np.cos(theta).astype(dtype), np.sin(theta).astype(dtype)


def test_qkv_complex_multiply_closed_form(orc):
    """Every Q and K pair is (x0 + i x1) * (c + i s) at its token's position, rounded once."""
    rng = np.random.default_rng(71)
    B, S, Nq, Nkv, H, R = 3, 5, 6, 2, 16, 40
    q, k, v, cos, sin = _qkv_inputs(rng, np.float32)
    pos = rng.integers(0, R, (B, S))
    h = H // 2
    for inter in (0, 1):
        qo, ko, _, _, _, _ = orc.rope_qkv(q, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv, key=k,
                                          interleaved=inter)
        i0 = np.arange(h) * 2 if inter else np.arange(h)
        i1 = i0 + 1 if inter else i0 + h
        w = cos.astype(np.float64)[pos] + 1j * sin.astype(np.float64)[pos]   # (B, S, h)
        for x, y, n in ((q, qo, Nq), (k, ko, Nkv)):
            xr, yr = x.reshape(B, S, n, H), y.reshape(B, S, n, H)
            z = xr[..., i0].astype(np.complex128) + 1j * xr[..., i1].astype(np.complex128)
            prod = z * w[:, :, None, :]
            assert np.array_equal(yr[..., i0], prod.real.astype(np.float32))
            assert np.array_equal(yr[..., i1], prod.imag.astype(np.float32))


def test_qkv_cache_rows_values_and_skips(orc):
    """Cache mode: token s of batch b lands in row past[b] + s of both caches (K rotated at
    position past[b] + s, V bit-exact); every other row keeps its bits; rows past the end
    are skipped and counted."""
    rng = np.random.default_rng(72)
    B, S, Nq, Nkv, H, L = 3, 5, 6, 2, 16, 9
    for dtype in (np.float16, np.float32):
        q, k, v, cos, sin = _qkv_inputs(rng, dtype)
        kc0 = rng.standard_normal((B, Nkv, L, H)).astype(dtype)
        vc0 = rng.standard_normal((B, Nkv, L, H)).astype(dtype)
        past = np.array([0, 4, 6], dtype=np.int32)            # batch 2: rows 6..10, two past the end
        qo, ko, kc, vc, n_oor, n_skip = orc.rope_qkv(q, cos, sin, None, num_heads=Nq, kv_num_heads=Nkv,
                                                    key=k, value=v, k_cache=kc0, v_cache=vc0,
                                                    past_seq_lens=past)
        assert ko is None and n_oor == 0 and n_skip == 2
        # the rotation the cache must hold: explicit positions past[b] + s, no cache
        pos = past[:, None].astype(np.int64) + np.arange(S)[None, :]
        qe, ke, _, _, _, _ = orc.rope_qkv(q, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv, key=k)
        assert np.array_equal(qo.view(np.uint8), qe.view(np.uint8))
        kexp, vexp = kc0.copy(), vc0.copy()
        ke4, v4 = ke.reshape(B, S, Nkv, H), v.reshape(B, S, Nkv, H)
        for b in range(B):
            for s in range(S):
                r = past[b] + s
                if r < L:
                    kexp[b, :, r] = ke4[b, s]
                    vexp[b, :, r] = v4[b, s]
        assert np.array_equal(kc.view(np.uint8), kexp.view(np.uint8))
        assert np.array_equal(vc.view(np.uint8), vexp.view(np.uint8))


def test_qkv_reduces_to_rotary_embedding_and_packed_equals_separate(orc):
    """Q and K each come out exactly as RotaryEmbedding rotates a rank-3 X of those heads
    (including out-of-range positions and a partial rotary width), and a packed [Q|K|V]
    input gives the same bits as separate tensors."""
    rng = np.random.default_rng(73)
    B, S, Nq, Nkv, H, R = 2, 7, 8, 2, 16, 30
    for dtype in (np.float16, np.float32):
        q, k, v, cos8, sin8 = _qkv_inputs(rng, dtype, B, S, Nq, Nkv, H, R)
        for rd in (0, 8):
            cos, sin = (cos8, sin8) if rd == 0 else (cos8[:, :rd // 2].copy(), sin8[:, :rd // 2].copy())
            pos = rng.integers(0, R, (B, S))
            pos[0, 3], pos[1, 0] = R, -1
            for inter in (0, 1):
                qo, ko, _, _, n_oor, _ = orc.rope_qkv(q, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv,
                                                      key=k, interleaved=inter, rotary_embedding_dim=rd)
                assert n_oor == 2
                yq, _ = orc.rope(q, cos, sin, pos, inter, rd, Nq)
                yk, _ = orc.rope(k, cos, sin, pos, inter, rd, Nkv)
                assert np.array_equal(qo.view(np.uint8), yq.view(np.uint8))
                assert np.array_equal(ko.view(np.uint8), yk.view(np.uint8))
                packed = np.concatenate([q, k, v], axis=-1)
                qp, kp, _, _, _, _ = orc.rope_qkv(packed, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv,
                                                  interleaved=inter, rotary_embedding_dim=rd)
                assert np.array_equal(qp.view(np.uint8), qo.view(np.uint8))
                assert np.array_equal(kp.view(np.uint8), ko.view(np.uint8))


def test_qkv_implicit_positions_follow_the_cache(orc):
    """Without position_ids, token s takes position past[b] + s (s without past)."""
    rng = np.random.default_rng(74)
    B, S, Nq, Nkv, H = 3, 4, 4, 4, 8
    q, k, v, cos, sin = _qkv_inputs(rng, np.float32, B, S, Nq, Nkv, H, 20)
    past = np.array([0, 3, 9], dtype=np.int32)
    a = orc.rope_qkv(q, cos, sin, None, num_heads=Nq, kv_num_heads=Nkv, key=k, past_seq_lens=past)
    b = orc.rope_qkv(q, cos, sin, past[:, None] + np.arange(S)[None, :], num_heads=Nq, kv_num_heads=Nkv,
                     key=k)
    c = orc.rope_qkv(q, cos, sin, None, num_heads=Nq, kv_num_heads=Nkv, key=k)
    d = orc.rope_qkv(q, cos, sin, np.tile(np.arange(S), (B, 1)), num_heads=Nq, kv_num_heads=Nkv, key=k)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(c[0], d[0]) and np.array_equal(c[1], d[1])
    assert not np.array_equal(a[0], c[0])


# --------------------------------------------------------------------------
# QK-RMSNorm before the rotation (Qwen3 fusion PR: Qwen3 Architecture,
# Verification). Reading: z = T(w * T(x / sqrt(mean(x^2) + eps))) per head.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_qkv_rmsnorm_hand_example(orc, dtype):
    g = _gold("qkv_rmsnorm_hand_example.json")
    H = g["head_size"]
    arr = lambda v: np.array(v, dtype=dtype)  # noqa: E731
    q, k = arr(g["q"]).reshape(1, 1, H), arr(g["k"]).reshape(1, 1, H)
    exp = g["expected"][np.dtype(dtype).name]
    qo, ko, _, _, _, _ = orc.rope_qkv(q, arr(g["cos"]), arr(g["sin"]), np.array([[g["position"]]]),
                                      num_heads=1, kv_num_heads=1, key=k, q_norm_weight=arr(g["q_weight"]),
                                      k_norm_weight=arr(g["k_weight"]), epsilon=g["epsilon"])
    assert qo.ravel().tolist() == [float(dtype(v)) for v in exp["q_out"]]
    assert ko.ravel().tolist() == [float(dtype(v)) for v in exp["k_out"]]


def test_qkv_rmsnorm_epsilon_closed_form(orc):
    """A constant head a normalises to a / sqrt(a^2 + eps) (mpmath, rounded to T)."""
    H, a, eps = 8, 2.0, 1e-3
    for dtype in (np.float16, np.float32):
        q = np.full((1, 1, H), a, dtype=dtype)
        one = np.ones((1, H // 2), dtype=dtype)
        zero = np.zeros((1, H // 2), dtype=dtype)
        qo, _, _, _, _, _ = orc.rope_qkv(q, one, zero, np.zeros((1, 1), np.int64), num_heads=1, kv_num_heads=1,
                                         key=q.copy(), q_norm_weight=np.ones(H, dtype), k_norm_weight=np.ones(H, dtype),
                                         epsilon=eps)
        exact = mpmath.mpf(a) / mpmath.sqrt(mpmath.mpf(a) ** 2 + mpmath.mpf(eps))
        assert (qo.ravel() == dtype(float(exact))).all()
        assert float(dtype(float(exact))) != 1.0 or dtype == np.float16


def _rmsnorm_numpy(x, w, eps, H, dtype):
    """Independent formulation: numpy float64 mean of squares, rounded with astype."""
    xs = x.reshape(*x.shape[:-1], -1, H).astype(np.float64)
    r = 1.0 / np.sqrt(np.mean(xs * xs, axis=-1, keepdims=True) + eps)
    n = (xs * r).astype(dtype).astype(np.float64)
    return (n * w.astype(np.float64)).astype(dtype).reshape(x.shape)


def test_qkv_rmsnorm_equals_numpy_norm_then_rotation(orc):
    """Fused == numpy RMSNorm followed by the pinned RotaryEmbedding oracle, bit for bit, on Q
    and K (separate weights), packed and separate, partial width, out-of-range positions
    (the normalised head is copied through); V is never normalised."""
    rng = np.random.default_rng(75)
    B, S, Nq, Nkv, H, R, L = 2, 6, 4, 2, 16, 30, 12
    for dtype in (np.float16, np.float32):
        q, k, v, cos8, sin8 = _qkv_inputs(rng, dtype, B, S, Nq, Nkv, H, R)
        q = (q * 3).astype(dtype)
        wq = rng.uniform(0.5, 1.5, H).astype(dtype)
        wk = rng.uniform(0.5, 1.5, H).astype(dtype)
        eps = 1e-6
        for rd in (0, 8):
            cos, sin = (cos8, sin8) if rd == 0 else (cos8[:, :rd // 2].copy(), sin8[:, :rd // 2].copy())
            pos = rng.integers(0, R, (B, S))
            pos[1, 2] = R + 1
            zq = _rmsnorm_numpy(q, wq, eps, H, dtype)
            zk = _rmsnorm_numpy(k, wk, eps, H, dtype)
            yq, _ = orc.rope(zq, cos, sin, pos, 0, rd, Nq)
            yk, _ = orc.rope(zk, cos, sin, pos, 0, rd, Nkv)
            qo, ko, _, _, n_oor, _ = orc.rope_qkv(q, cos, sin, pos, num_heads=Nq, kv_num_heads=Nkv, key=k,
                                                  rotary_embedding_dim=rd, q_norm_weight=wq, k_norm_weight=wk,
                                                  epsilon=eps)
            assert n_oor == 1
            assert np.array_equal(qo.view(np.uint8), yq.view(np.uint8))
            assert np.array_equal(ko.view(np.uint8), yk.view(np.uint8))
            # packed input and cache mode: same Q, K in the cache rows, V copied unchanged
            packed = np.concatenate([q, k, v], axis=-1)
            past = np.array([0, 3], dtype=np.int32)
            kc0 = np.zeros((B, Nkv, L, H), dtype)
            qp, _, kc, vc, _, _ = orc.rope_qkv(packed, cos, sin, past[:, None] + np.arange(S)[None, :],
                                               num_heads=Nq, kv_num_heads=Nkv, rotary_embedding_dim=rd,
                                               k_cache=kc0, v_cache=kc0, past_seq_lens=past, q_norm_weight=wq,
                                               k_norm_weight=wk, epsilon=eps)
            pos2 = past[:, None] + np.arange(S)[None, :]
            yq2, _ = orc.rope(zq, cos, sin, pos2, 0, rd, Nq)
            yk2, _ = orc.rope(zk, cos, sin, pos2, 0, rd, Nkv)
            assert np.array_equal(qp.view(np.uint8), yq2.view(np.uint8))
            for b in range(B):
                for s in range(S):
                    row = past[b] + s
                    assert np.array_equal(kc[b, :, row].view(np.uint8),
                                          yk2.reshape(B, S, Nkv, H)[b, s].view(np.uint8))
                    assert np.array_equal(vc[b, :, row].view(np.uint8), v.reshape(B, S, Nkv, H)[b, s].view(np.uint8))


def test_qkv_rmsnorm_scale_invariant_without_epsilon(orc):
    rng = np.random.default_rng(76)
    B, S, N, H, R = 2, 3, 2, 16, 10
    for dtype in (np.float16, np.float32):
        q, k, _, cos, sin = _qkv_inputs(rng, dtype, B, S, N, N, H, R)
        w = rng.uniform(0.5, 1.5, H).astype(dtype)
        pos = rng.integers(0, R, (B, S))
        a = orc.rope_qkv(q, cos, sin, pos, num_heads=N, kv_num_heads=N, key=k, q_norm_weight=w, k_norm_weight=w,
                         epsilon=0.0)
        b = orc.rope_qkv((q * 4).astype(dtype), cos, sin, pos, num_heads=N, kv_num_heads=N,
                         key=(k / 8).astype(dtype), q_norm_weight=w, k_norm_weight=w, epsilon=0.0)
        assert np.array_equal(a[0].view(np.uint8), b[0].view(np.uint8))
        assert np.array_equal(a[1].view(np.uint8), b[1].view(np.uint8))


# --------------------------------------------------------------------------
# MRotaryEmbedding with on-the-fly coefficients (MRotaryEmbedding README:
# Description, Inputs, Attributes; Qwen3 fusion PR: Motivation and Context)
# --------------------------------------------------------------------------

def test_mrope_fused_equals_cached_table(orc):
    """On-the-fly M-RoPE == M-RoPE over the cache build's table, bit for bit, for every
    layout, pairing, scale and a partial width (all positions in range)."""
    rng = np.random.default_rng(81)
    B, S, N, H, R = 2, 9, 3, 32, 200
    for dtype in (np.float16, np.float32):
        x = rng.standard_normal((B, S, N * H)).astype(dtype)
        for rd, sec in ((0, (6, 5, 5)), (16, (4, 2, 2))):
            h = (rd or H) // 2
            inv = wl.inv_freq(10000.0, rd or H, h)
            cos, sin = orc.cache_build(inv, R, dtype, 1.25)
            pos3 = rng.integers(0, R, (3, B, S))
            for layout in (0, 1):
                for inter in (0, 1):
                    for scale in (1.0, float(np.float32(0.7))):
                        y_c, n_oor = orc.mrope(x, cos, sin, pos3, sec, layout, scale, inter, rd, N)
                        assert n_oor == 0
                        y_f = orc.mrope_fused(x, inv, pos3, sec, layout, scale, 1.25, inter, rd, N)
                        assert np.array_equal(y_f.view(np.uint8), y_c.view(np.uint8)), (dtype, rd, layout, inter)


def test_mrope_fused_equal_streams_reduce_to_fused_rope(orc):
    """Equal t/h/w streams and scale 1: exactly the on-the-fly RotaryEmbedding (which has no
    out-of-range positions either, so large and negative positions are fine)."""
    rng = np.random.default_rng(82)
    B, S, N, H = 2, 7, 2, 16
    for dtype in (np.float16, np.float32):
        x = rng.standard_normal((B, S, N * H)).astype(dtype)
        inv = wl.inv_freq(1.0e6, H, H // 2)
        pos = rng.integers(-5000, 1 << 40, (B, S))
        pos3 = np.stack([pos, pos, pos])
        y_r = orc.rope_fused(x, inv, pos, 1.0, 0, 0, N)
        for layout in (0, 1):
            y_m = orc.mrope_fused(x, inv, pos3, (4, 2, 2), layout, 1.0, 1.0, 0, 0, N)
            assert np.array_equal(y_m.view(np.uint8), y_r.view(np.uint8))


# --------------------------------------------------------------------------
# bfloat16 conversion (storage offered beyond the pages' float32/float16)
# against torch's independent implementation and exact arithmetic
# --------------------------------------------------------------------------

def test_bf16_to_double_all_patterns(orc):
    torch = pytest.importorskip("torch")
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_double_to_bf16_midpoints_and_random_float32(orc):
    """float32 inputs (so torch's float32 -> bfloat16 rounding is a single rounding):
    every bf16 midpoint, its float32 neighbours, and random values across the range."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(61)
    finite = np.arange(0, 0x7f80, dtype=np.uint32)
    mids = ((finite << 16) | 0x8000).view(np.float32)                 # exactly halfway
    vals = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0)),
                           rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(
                               -40, 38, 20000).astype(np.float32)])
    vals = vals[np.isfinite(vals)]
    vals = np.concatenate([vals, -vals])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.double_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_double_to_bf16_single_rounding_from_binary64(orc):
    """Values a hair above or below a bf16 midpoint that float32 cannot hold: a correct
    single rounding must go to the nearer neighbour (rounding through float32 first would
    land on the midpoint and tie to even)."""
    for bits in (0x3f80, 0x3f81, 0x4049, 0x0001, 0x7f7e):
        lo, hi = Fraction(orc.bf16_to_double(bits)), Fraction(orc.bf16_to_double(bits + 1))
        mid = (lo + hi) / 2
        eps = (hi - lo) / (1 << 40)
        assert orc.double_to_bf16(float(mid + eps)) == bits + 1
        assert orc.double_to_bf16(float(mid - eps)) == bits
        assert orc.double_to_bf16(float(mid)) == (bits if bits % 2 == 0 else bits + 1)


def _bf16_bits(values):
    """float32 values that bfloat16 holds exactly -> their bit patterns (truncation is exact here)."""
    f = np.asarray(values, dtype=np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(((b.astype(np.uint32) << 16).view(np.float32)), f)
    return b


def test_hand_example_bfloat16(orc):
    g = _gold("hand_example.json")
    x = _bf16_bits(g["x"]).reshape(1, 1, g["head_size"])
    for case in g["cases"]:
        c = _bf16_bits(case["cos"]).reshape(1, -1)
        s = _bf16_bits(case["sin"]).reshape(1, -1)
        y, _ = orc.rope(x, c, s, np.zeros((1, 1), np.int64), case["interleaved"], case["rotary_embedding_dim"], 1)
        assert y.dtype == np.uint16
        assert [orc.bf16_to_double(int(v)) for v in y.ravel()] == case["y"], case["name"]


def test_bfloat16_rotation_rounds_once(orc):
    """Each bf16 output is the exact rotation (rational arithmetic on the bf16 inputs)
    rounded once to nearest-even bf16."""
    rng = np.random.default_rng(62)
    H = 8
    xs = _bf16_bits(np.round(rng.standard_normal((1, 4, H)) * 64) / 64).reshape(1, 4, H)
    th = rng.uniform(-np.pi, np.pi, (4, H // 2))
    cos = (np.cos(th).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    sin = (np.sin(th).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    pos = np.arange(4).reshape(1, 4)
    y, _ = orc.rope(xs, cos, sin, pos, 0, 0, 1)
    val = lambda b: Fraction(orc.bf16_to_double(int(b)))  # noqa: E731
    for s_ in range(4):
        for i in range(H // 2):
            x0, x1 = val(xs[0, s_, i]), val(xs[0, s_, i + H // 2])
            c, sn = val(cos[s_, i]), val(sin[s_, i])
            for j, exact in ((i, x0 * c - x1 * sn), (i + H // 2, x1 * c + x0 * sn)):
                lo = orc.double_to_bf16(float(exact))
                # the exact value's nearest bf16 (float(exact) is within 2^-53 relative: no tie shifts)
                assert int(y[0, s_, j]) == lo


# ---------------------------------------------------------------------------
# M-RoPE Q/K rotation with the cache append (oracle_mrope_qkv): each Q and K head is
# one head of MRotaryEmbedding ("com.microsoft.MRotaryEmbedding" README, Description,
# Inputs/positionIds, Attributes); grouped-query heads and the cache as SparseAttention.
# ---------------------------------------------------------------------------

def test_mrope_qkv_reduces_to_mrope_per_head(orc):
    """Q heads and K heads equal the pinned M-RoPE oracle run on Q and on K alone, bit for bit:
    both layouts, both pairings, a partial width, a scale, and pairs whose stream position is
    out of range (copied through); packed input equals separate input."""
    rng = np.random.default_rng(81)
    B, S, Nq, Nkv, H, R = 2, 7, 6, 2, 16, 30
    for dtype in (np.float16, np.float32):
        q, k, v, cos8, sin8 = _qkv_inputs(rng, dtype, B, S, Nq, Nkv, H, R)
        for rd, sec in ((0, (2, 3, 3)), (8, (2, 1, 1))):
            cos, sin = (cos8, sin8) if rd == 0 else (cos8[:, :rd // 2].copy(), sin8[:, :rd // 2].copy())
            pos = rng.integers(0, R, (3, B, S))
            pos[1, 0, 3], pos[2, 1, 6], pos[0, 1, 0] = R, -1, R + 9
            for layout in (0, 1):
                for inter in (0, 1):
                    for scale in (1.0, 0.75):
                        yq, nq = orc.mrope(q, cos, sin, pos, sec, layout, scale, inter, rd, Nq)
                        yk, nk = orc.mrope(k, cos, sin, pos, sec, layout, scale, inter, rd, Nkv)
                        qo, ko, _, _, n_oor, _ = orc.mrope_qkv(q, cos, sin, pos, sec, layout, scale, num_heads=Nq,
                                                               kv_num_heads=Nkv, key=k, interleaved=inter,
                                                               rotary_embedding_dim=rd)
                        assert n_oor == nq + nk > 0
                        assert np.array_equal(qo.view(np.uint8), yq.view(np.uint8))
                        assert np.array_equal(ko.view(np.uint8), yk.view(np.uint8))
                        packed = np.concatenate([q, k, v], axis=-1)
                        qp, kp, _, _, _, _ = orc.mrope_qkv(packed, cos, sin, pos, sec, layout, scale,
                                                           num_heads=Nq, kv_num_heads=Nkv, interleaved=inter,
                                                           rotary_embedding_dim=rd)
                        assert np.array_equal(qp.view(np.uint8), qo.view(np.uint8))
                        assert np.array_equal(kp.view(np.uint8), ko.view(np.uint8))


def test_mrope_qkv_equal_streams_equal_rope_qkv(orc):
    """t = h = w and scale 1: the M-RoPE Q/K op is the pinned RotaryEmbedding Q/K op, bit for
    bit, for every layout (cache mode included, with rows past its end skipped)."""
    rng = np.random.default_rng(82)
    B, S, Nq, Nkv, H, R, L = 2, 6, 4, 2, 16, 30, 9
    q, k, v, cos, sin = _qkv_inputs(rng, np.float16, B, S, Nq, Nkv, H, R)
    p = rng.integers(0, R, (B, S))
    p[0, 2] = R + 2
    pos3 = np.stack([p, p, p])
    past = np.array([2, 5], dtype=np.int32)
    kc0 = rng.standard_normal((B, Nkv, L, H)).astype(np.float16)
    want = orc.rope_qkv(q, cos, sin, p, num_heads=Nq, kv_num_heads=Nkv, key=k, value=v, k_cache=kc0, v_cache=kc0,
                        past_seq_lens=past)
    for layout in (0, 1, 2):
        got = orc.mrope_qkv(q, cos, sin, pos3, (3, 3, 2), layout, 1.0, num_heads=Nq, kv_num_heads=Nkv, key=k,
                            value=v, k_cache=kc0, v_cache=kc0, past_seq_lens=past)
        for a, b in zip(got[:4], want[:4]):
            if a is None:
                assert b is None
            else:
                assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
        assert got[5] == want[5] > 0


def test_mrope_qkv_rmsnorm_cache_rows_and_values(orc):
    """With QK-RMSNorm: numpy RMSNorm followed by the pinned M-RoPE oracle, bit for bit, on Q
    and K; in cache mode the rotated K rows sit at past[b] + s, V rows are copies, rows outside
    [0, max_len) are not written and are counted, every other row is untouched."""
    rng = np.random.default_rng(83)
    B, S, Nq, Nkv, H, R, L = 2, 6, 4, 2, 16, 30, 9
    for dtype in (np.float16, np.float32):
        q, k, v, cos, sin = _qkv_inputs(rng, dtype, B, S, Nq, Nkv, H, R)
        q = (q * 3).astype(dtype)
        wq = rng.uniform(0.5, 1.5, H).astype(dtype)
        wk = rng.uniform(0.5, 1.5, H).astype(dtype)
        pos = rng.integers(0, R, (3, B, S))
        pos[2, 1, 1] = R
        sec = (2, 3, 3)
        zq = _rmsnorm_numpy(q, wq, 1e-6, H, dtype)
        zk = _rmsnorm_numpy(k, wk, 1e-6, H, dtype)
        yq, _ = orc.mrope(zq, cos, sin, pos, sec, 1, 1.0, 0, 0, Nq)
        yk, _ = orc.mrope(zk, cos, sin, pos, sec, 1, 1.0, 0, 0, Nkv)
        past = np.array([0, 5], dtype=np.int32)                # batch 1 runs past the 9-row cache
        kc0 = rng.standard_normal((B, Nkv, L, H)).astype(dtype)
        vc0 = rng.standard_normal((B, Nkv, L, H)).astype(dtype)
        qo, ko, kc, vc, _, n_skip = orc.mrope_qkv(q, cos, sin, pos, sec, 1, 1.0, num_heads=Nq, kv_num_heads=Nkv,
                                                  key=k, value=v, k_cache=kc0, v_cache=vc0, past_seq_lens=past,
                                                  q_norm_weight=wq, k_norm_weight=wk, epsilon=1e-6)
        assert ko is None
        assert np.array_equal(qo.view(np.uint8), yq.view(np.uint8))
        written = np.zeros((B, L), bool)
        for b in range(B):
            for s in range(S):
                row = past[b] + s
                if row >= L:
                    continue
                written[b, row] = True
                assert np.array_equal(kc[b, :, row].view(np.uint8), yk.reshape(B, S, Nkv, H)[b, s].view(np.uint8))
                assert np.array_equal(vc[b, :, row].view(np.uint8), v.reshape(B, S, Nkv, H)[b, s].view(np.uint8))
        assert n_skip == int((past[:, None] + np.arange(S)[None, :] >= L).sum()) > 0
        untouched = ~written
        assert np.array_equal(kc.transpose(0, 2, 1, 3)[untouched].view(np.uint8),
                              kc0.transpose(0, 2, 1, 3)[untouched].view(np.uint8))
        assert np.array_equal(vc.transpose(0, 2, 1, 3)[untouched].view(np.uint8),
                              vc0.transpose(0, 2, 1, 3)[untouched].view(np.uint8))
