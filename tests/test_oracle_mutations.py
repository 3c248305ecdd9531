"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each case plants one mistake in a temporary copy of the oracle's C source (a
flipped sign, a wrong pair index, a transposed row formula, a skipped
rounding, an off-by-one range check...), rebuilds that copy and runs the pin
suite against it; the suite must fail. Nothing here touches the real oracle
or the CUDA path.
"""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "sign_of_second_output": ("double y1 = x1 * c + x0 * s;", "double y1 = x1 * c - x0 * s;"),
    "interleaved_partner": ("*j1 = 2 * i + 1;", "*j1 = 2 * i + 2;"),
    "rank4_row_transposed": ("return ((b * g->N + n) * g->S + s) * g->H;",
                             "return ((b * g->S + s) * g->N + n) * g->H;"),
    "scaled_coefficient_not_rounded": (
        "double c = round_to(dt, ld(dt, cos_t, p * half + i) * (double)scale);",
        "double c = ld(dt, cos_t, p * half + i) * (double)scale;"),
    "range_check_off_by_one": ("if (p < 0 || p >= cache_rows) {", "if (p < 0 || p > cache_rows) {"),
    "angle_in_binary64": ("float theta = pf * inv;", "double theta = (double)pf * inv;"),
    "half_rounding_truncates": ("double r = nearbyint(ldexp(a, 10 - E));",
                                "double r = floor(ldexp(a, 10 - E));"),
    "interleaved_map_order": ("for (int st = 0; st < 3; ++st)\n      if (r < sec[st]) {",
                              "for (int st = 2; st >= 0; --st)\n      if (r < sec[st]) {"),
    "per_token_row_shifted": ("crow = tok * half;", "crow = tok * half + (tok > 0);"),
    "sin_from_cos_table": ("double sn = ld(dt, sin_t, crow + i);", "double sn = ld(dt, cos_t, crow + i);"),
    "scaling_dropped": ("float cs = c32 * scaling;", "float cs = c32;"),
    "qkv_cache_row_ignores_past": ("int64_t row = cache ? (int64_t)past[b] + s : 0;",
                                   "int64_t row = cache ? s : 0;"),
    "qkv_value_read_from_key": ("const void* vs = packed ? q : v;", "const void* vs = packed ? q : k;"),
    "qkv_packed_value_offset": ("int64_t vsrc = packed ? (tok * Ntot + Nq + Nkv + n) * H",
                                "int64_t vsrc = packed ? (tok * Ntot + Nq + n) * H"),
    "qkv_implicit_position_ignores_past": ("int64_t p = pos ? pos[tok] : (past ? (int64_t)past[b] + s : s);",
                                           "int64_t p = pos ? pos[tok] : s;"),
    "norm_mean_over_half_head": ("double r = 1.0 / sqrt(ss / (double)H + eps);",
                                 "double r = 1.0 / sqrt(ss / (double)(H / 2) + eps);"),
    "norm_epsilon_dropped": ("double r = 1.0 / sqrt(ss / (double)H + eps);", "double r = 1.0 / sqrt(ss / (double)H);"),
    "norm_weight_before_rounding": ("double n = round_to(dt, ld(dt, x, xb + j) * r);",
                                    "double n = ld(dt, x, xb + j) * r;"),
    "norm_key_uses_query_weight": ("rms_norm_head(dt, ks, ksrc, H, k_weight, eps, zq);",
                                   "rms_norm_head(dt, ks, ksrc, H, q_weight, eps, zq);"),
    "mrope_fused_stream_ignored": ("int64_t p = pos3[(int64_t)map[i] * ntok + tok];", "int64_t p = pos3[tok];"),
    "mrope_fused_scale_dropped": ("c = round_to(dt, c * (double)scale);", "c = round_to(dt, c);"),
    "bf16_exponent_bias": ("v = ldexp((double)(m + 128), e - 134);", "v = ldexp((double)(m + 128), e - 133);"),
    "bf16_rounding_truncates": ("double r = nearbyint(ldexp(a, 7 - E));", "double r = floor(ldexp(a, 7 - E));"),
    "mrope_qkv_stream_of_pair_ignored": ("const int64_t p = p3[map[i]];", "const int64_t p = p3[0];"),
    "mrope_qkv_positions_of_wrong_token": ("p3[st3] = pos3[st3 * B * S + tok];", "p3[st3] = pos3[st3 * B * S + b];"),
    "mrope_qkv_scale_dropped": ("const double c = round_to(dt, ld(dt, cos_t, p * half + i) * (double)scale);",
                                "const double c = round_to(dt, ld(dt, cos_t, p * half + i));"),
    "qkv_value_rotated": ("for (int64_t j = 0; j < H; ++j) cp(dt, vs, vsrc + j, v_cache, dst + j);",
                          "rope_one_head(dt, interleaved, H, rd, vs, vsrc, v_cache, dst, cos_t, sin_t, crow, valid);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(ROOT, "oracle", "rope_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} no longer in the oracle source"
    ign = shutil.ignore_patterns("_build", "*.so", "__pycache__")
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle", ignore=ign)
    (tmp_path / "oracle" / "rope_oracle.c").write_text(src.replace(old, new, 1))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests", ignore=ign)
    pkg = tmp_path / "rotary_position_embedding_gb300"
    pkg.mkdir()
    src_pkg = os.path.join(ROOT, "rotary_position_embedding_gb300")
    for f in os.listdir(src_pkg):
        if f.endswith(".py"):
            shutil.copy(os.path.join(src_pkg, f), pkg / f)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"planted mistake {name!r} passed every pin:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
