"""ctypes marshalling for the C oracle in ``rope_oracle.c``.

Test infrastructure: see the package docstring. Nothing here computes any
part of the method; every function hands contiguous numpy arrays to the C
library and returns its outputs.
"""

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rope_oracle.c")
_LIB = os.path.join(_HERE, "_build", "librope_oracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2
# numpy has no bfloat16: bfloat16 arrays travel as their uint16 bit patterns.
BF16_BITS = np.uint16

_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force=False):
    """Compile the oracle with gcc (no CUDA, no shared code with the product)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_double_to_half.argtypes = [ctypes.c_double]
            lib.oracle_double_to_half.restype = ctypes.c_uint16
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_rope.argtypes = [i32, i32, _i64p, i64, i32, i64, vp, vp, vp, i64, vp, vp, _i64p]
            lib.oracle_mrope_stream_map.argtypes = [vp, i32, i64, vp]
            lib.oracle_mrope_map.argtypes = [i32, i32, _i64p, i64, i32, i64, vp, vp, vp, i64, vp, vp,
                                             f32, vp, _i64p]
            lib.oracle_mrope.argtypes = [i32, i32, _i64p, i64, i32, i64, vp, vp, vp, i64, vp, vp, i32,
                                         f32, vp, _i64p]
            lib.oracle_rope_fused.argtypes = [i32, i32, _i64p, i64, i32, i64, vp, vp, f32, vp, vp]
            lib.oracle_cache_build.argtypes = [i32, vp, i64, i64, f32, vp, vp]
            lib.oracle_rope_qkv.argtypes = [i32, i64, i64, i64, i64, i64, i32, i64, vp, vp, vp, vp, vp, i64,
                                            vp, vp, vp, vp, vp, vp, i64, _i64p, _i64p]
            lib.oracle_rope_qkv_rmsnorm.argtypes = [i32, i64, i64, i64, i64, i64, i32, i64, vp, vp, vp, vp, vp,
                                                    ctypes.c_double, vp, vp, i64, vp, vp, vp, vp, vp, vp, i64,
                                                    _i64p, _i64p]
            lib.oracle_mrope_fused.argtypes = [i32, i32, _i64p, i64, i32, i64, vp, vp, f32, vp, vp, i32, f32,
                                               vp]
            lib.oracle_mrope_qkv.argtypes = [i32, i64, i64, i64, i64, i64, i32, i64, vp, vp, vp, vp, vp,
                                             ctypes.c_double, vp, vp, i64, vp, vp, i32, f32, vp, vp, vp, vp,
                                             vp, i64, _i64p, _i64p]
            for name in ("oracle_rope", "oracle_mrope_stream_map", "oracle_mrope_map", "oracle_mrope",
                         "oracle_rope_fused", "oracle_cache_build", "oracle_rope_qkv",
                         "oracle_rope_qkv_rmsnorm", "oracle_mrope_fused", "oracle_mrope_qkv"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _dt(a):
    if a.dtype == np.float16:
        return F16
    if a.dtype == np.float32:
        return F32
    if a.dtype == BF16_BITS:
        return BF16
    raise TypeError(f"oracle supports float16, float32 and bfloat16 (uint16 bits), got {a.dtype}")


def _c(a, dtype=None):
    if dtype is not None and np.dtype(dtype) == BF16_BITS and np.asarray(a).dtype != BF16_BITS:
        raise TypeError("bfloat16 arrays travel as uint16 bit patterns; convert before the call")
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shape(x):
    arr = (ctypes.c_int64 * 4)(*([int(d) for d in x.shape] + [0] * (4 - x.ndim)))
    return arr


def half_to_double(bits):
    return _load().oracle_half_to_double(int(bits))


def bf16_to_double(bits):
    return _load().oracle_bf16_to_double(int(bits))


def double_to_bf16(v):
    return _load().oracle_double_to_bf16(float(v))


def double_to_half(v):
    return _load().oracle_double_to_half(float(v))


def rope(x, cos, sin, position_ids=None, interleaved=0, rotary_embedding_dim=0, num_heads=0):
    """RotaryEmbedding. Returns (y, number of tokens whose position was out of range)."""
    lib = _load()
    x = _c(x)
    cos = _c(cos, x.dtype)
    sin = _c(sin, x.dtype)
    pos = None if position_ids is None else _c(position_ids, np.int64)
    rows = cos.shape[0] if pos is not None else 0
    y = np.empty_like(x)
    n = ctypes.c_int64(0)
    rc = lib.oracle_rope(_dt(x), x.ndim, _shape(x), int(num_heads), int(interleaved),
                         int(rotary_embedding_dim), _ptr(x), _ptr(cos), _ptr(sin), int(rows), _ptr(pos),
                         _ptr(y), ctypes.byref(n))
    if rc:
        raise ValueError("oracle_rope: malformed arguments")
    return y, n.value


def mrope_stream_map(section, layout, half):
    """Stream (0=t, 1=h, 2=w) of each of the rd/2 coefficient indices.

    layout 0 = chunked, 1 = interleaved (round-robin honouring the section
    counts), 2 = interleaved stride-3 reading.
    """
    lib = _load()
    sec = np.ascontiguousarray(section, dtype=np.int32)
    m = np.zeros(int(half), dtype=np.uint8)
    rc = lib.oracle_mrope_stream_map(_ptr(sec), int(layout), int(half), _ptr(m))
    if rc:
        raise ValueError("oracle_mrope_stream_map: sections do not divide the half-rotary axis")
    return m


def mrope_map(x, cos, sin, position_ids, stream_map, scale=1.0, interleaved=0, rotary_embedding_dim=0,
              num_heads=0):
    """MRotaryEmbedding with an explicit per-index stream map. Returns (y, pairs copied through)."""
    lib = _load()
    x = _c(x)
    cos = _c(cos, x.dtype)
    sin = _c(sin, x.dtype)
    pos = _c(position_ids, np.int64)
    m = _c(stream_map, np.uint8)
    y = np.empty_like(x)
    n = ctypes.c_int64(0)
    rc = lib.oracle_mrope_map(_dt(x), x.ndim, _shape(x), int(num_heads), int(interleaved),
                              int(rotary_embedding_dim), _ptr(x), _ptr(cos), _ptr(sin), int(cos.shape[0]),
                              _ptr(pos), _ptr(m), float(scale), _ptr(y), ctypes.byref(n))
    if rc:
        raise ValueError("oracle_mrope_map: malformed arguments")
    return y, n.value


def mrope(x, cos, sin, position_ids, mrope_section, mrope_layout=0, scale=1.0, interleaved=0,
          rotary_embedding_dim=0, num_heads=0):
    """MRotaryEmbedding with the map given by mrope_section/mrope_layout."""
    lib = _load()
    x = _c(x)
    cos = _c(cos, x.dtype)
    sin = _c(sin, x.dtype)
    pos = _c(position_ids, np.int64)
    sec = np.ascontiguousarray(mrope_section, dtype=np.int32)
    y = np.empty_like(x)
    n = ctypes.c_int64(0)
    rc = lib.oracle_mrope(_dt(x), x.ndim, _shape(x), int(num_heads), int(interleaved),
                          int(rotary_embedding_dim), _ptr(x), _ptr(cos), _ptr(sin), int(cos.shape[0]),
                          _ptr(pos), _ptr(sec), int(mrope_layout), float(scale), _ptr(y), ctypes.byref(n))
    if rc:
        raise ValueError("oracle_mrope: malformed arguments")
    return y, n.value


def rope_fused(x, inv_freq, position_ids, attention_scaling=1.0, interleaved=0, rotary_embedding_dim=0,
               num_heads=0):
    """Rotation with cos/sin computed from inv_freq at each position."""
    lib = _load()
    x = _c(x)
    inv = _c(inv_freq, np.float32)
    pos = _c(position_ids, np.int64)
    y = np.empty_like(x)
    rc = lib.oracle_rope_fused(_dt(x), x.ndim, _shape(x), int(num_heads), int(interleaved),
                               int(rotary_embedding_dim), _ptr(x), _ptr(inv), float(attention_scaling),
                               _ptr(pos), _ptr(y))
    if rc:
        raise ValueError("oracle_rope_fused: malformed arguments")
    return y


def mrope_fused(x, inv_freq, position_ids, mrope_section, mrope_layout=0, scale=1.0, attention_scaling=1.0,
                interleaved=0, rotary_embedding_dim=0, num_heads=0):
    """MRotaryEmbedding with cos/sin computed on the fly from inv_freq (three position streams)."""
    lib = _load()
    x = _c(x)
    inv = _c(inv_freq, np.float32)
    pos = _c(position_ids, np.int64)
    sec = np.ascontiguousarray(mrope_section, dtype=np.int32)
    y = np.empty_like(x)
    rc = lib.oracle_mrope_fused(_dt(x), x.ndim, _shape(x), int(num_heads), int(interleaved),
                                int(rotary_embedding_dim), _ptr(x), _ptr(inv), float(attention_scaling), _ptr(pos),
                                _ptr(sec), int(mrope_layout), float(scale), _ptr(y))
    if rc:
        raise ValueError("oracle_mrope_fused: malformed arguments")
    return y


def cache_build(inv_freq, rows, dtype=np.float16, attention_scaling=1.0):
    """(rows, len(inv_freq)) cos and sin tables."""
    lib = _load()
    inv = _c(inv_freq, np.float32)
    half = inv.shape[0]
    cos = np.empty((int(rows), half), dtype=dtype)
    sin = np.empty((int(rows), half), dtype=dtype)
    rc = lib.oracle_cache_build(_dt(cos), _ptr(inv), int(half), int(rows), float(attention_scaling),
                                _ptr(cos), _ptr(sin))
    if rc:
        raise ValueError("oracle_cache_build: malformed arguments")
    return cos, sin


def rope_qkv(query, cos, sin, position_ids=None, *, num_heads, kv_num_heads, key=None, value=None,
             interleaved=0, rotary_embedding_dim=0, k_cache=None, v_cache=None, past_seq_lens=None,
             q_norm_weight=None, k_norm_weight=None, epsilon=1e-6):
    """Q and K rotation with grouped-query heads and the optional cache append;
    with q_norm_weight and k_norm_weight (head-size vectors) each Q and K head
    is RMS-normalised (epsilon) before the rotation.

    query is (B, S, Nq*H), or packed (B, S, (Nq + 2*Nkv)*H) when key and value
    are None. With k_cache/v_cache (B, Nkv, max_len, H) the caches are copied,
    the new rows written and the copies returned. Returns
    (q_out, k_out or None, k_cache or None, v_cache or None, n_oor, n_skip).
    """
    lib = _load()
    q = _c(query)
    B, S, hidden = q.shape
    packed = key is None and value is None
    Ntot = num_heads + (2 * kv_num_heads if packed else 0)
    H = hidden // Ntot
    k = None if key is None else _c(key, q.dtype)
    v = None if value is None else _c(value, q.dtype)
    cos = _c(cos, q.dtype)
    sin = _c(sin, q.dtype)
    pos = None if position_ids is None else _c(position_ids, np.int64)
    past = None if past_seq_lens is None else _c(past_seq_lens, np.int32)
    q_out = np.empty((B, S, num_heads * H), dtype=q.dtype)
    cache = k_cache is not None
    k_out = None if cache else np.empty((B, S, kv_num_heads * H), dtype=q.dtype)
    kc = None if k_cache is None else np.array(k_cache, dtype=q.dtype, copy=True, order="C")
    vc = None if v_cache is None else np.array(v_cache, dtype=q.dtype, copy=True, order="C")
    max_len = kc.shape[2] if cache else 0
    n_oor, n_skip = ctypes.c_int64(0), ctypes.c_int64(0)
    if q_norm_weight is None and k_norm_weight is None:
        rc = lib.oracle_rope_qkv(_dt(q), B, S, int(num_heads), int(kv_num_heads), H, int(interleaved),
                                 int(rotary_embedding_dim), _ptr(q), _ptr(k), _ptr(v), _ptr(cos), _ptr(sin),
                                 int(cos.shape[0]), _ptr(pos), _ptr(past), _ptr(q_out), _ptr(k_out), _ptr(kc),
                                 _ptr(vc), int(max_len), ctypes.byref(n_oor), ctypes.byref(n_skip))
    else:
        qw = _c(q_norm_weight, q.dtype)
        kw = _c(k_norm_weight, q.dtype)
        rc = lib.oracle_rope_qkv_rmsnorm(_dt(q), B, S, int(num_heads), int(kv_num_heads), H, int(interleaved),
                                         int(rotary_embedding_dim), _ptr(q), _ptr(k), _ptr(v), _ptr(qw),
                                         _ptr(kw), float(epsilon), _ptr(cos), _ptr(sin), int(cos.shape[0]),
                                         _ptr(pos), _ptr(past), _ptr(q_out), _ptr(k_out), _ptr(kc), _ptr(vc),
                                         int(max_len), ctypes.byref(n_oor), ctypes.byref(n_skip))
    if rc:
        raise ValueError("oracle_rope_qkv: malformed arguments")
    return q_out, k_out, kc, vc, n_oor.value, n_skip.value


def mrope_qkv(query, cos, sin, position_ids, mrope_section, mrope_layout=0, scale=1.0, *, num_heads,
              kv_num_heads, key=None, value=None, interleaved=0, rotary_embedding_dim=0, k_cache=None,
              v_cache=None, past_seq_lens=None, q_norm_weight=None, k_norm_weight=None, epsilon=1e-6):
    """Q and K rotation with M-RoPE (position_ids (3, B, S): t, h, w), grouped-query
    heads, the optional QK-RMSNorm and the optional cache append. Arguments and
    returns as rope_qkv; n_oor counts Q and K pairs copied through."""
    lib = _load()
    q = _c(query)
    B, S, hidden = q.shape
    packed = key is None and value is None
    Ntot = num_heads + (2 * kv_num_heads if packed else 0)
    H = hidden // Ntot
    k = None if key is None else _c(key, q.dtype)
    v = None if value is None else _c(value, q.dtype)
    cos = _c(cos, q.dtype)
    sin = _c(sin, q.dtype)
    pos = _c(position_ids, np.int64)
    sec = np.ascontiguousarray(mrope_section, dtype=np.int32)
    past = None if past_seq_lens is None else _c(past_seq_lens, np.int32)
    q_out = np.empty((B, S, num_heads * H), dtype=q.dtype)
    cache = k_cache is not None
    k_out = None if cache else np.empty((B, S, kv_num_heads * H), dtype=q.dtype)
    kc = None if k_cache is None else np.array(k_cache, dtype=q.dtype, copy=True, order="C")
    vc = None if v_cache is None else np.array(v_cache, dtype=q.dtype, copy=True, order="C")
    max_len = kc.shape[2] if cache else 0
    qw = None if q_norm_weight is None else _c(q_norm_weight, q.dtype)
    kw = None if k_norm_weight is None else _c(k_norm_weight, q.dtype)
    n_oor, n_skip = ctypes.c_int64(0), ctypes.c_int64(0)
    rc = lib.oracle_mrope_qkv(_dt(q), B, S, int(num_heads), int(kv_num_heads), H, int(interleaved),
                              int(rotary_embedding_dim), _ptr(q), _ptr(k), _ptr(v), _ptr(qw), _ptr(kw),
                              float(epsilon), _ptr(cos), _ptr(sin), int(cos.shape[0]), _ptr(pos), _ptr(sec),
                              int(mrope_layout), float(scale), _ptr(past), _ptr(q_out), _ptr(k_out), _ptr(kc),
                              _ptr(vc), int(max_len), ctypes.byref(n_oor), ctypes.byref(n_skip))
    if rc:
        raise ValueError("oracle_mrope_qkv: malformed arguments")
    return q_out, k_out, kc, vc, n_oor.value, n_skip.value
