"""GB300-native rotary position embedding: RoPE, M-RoPE, on-the-fly RoPE.

A thin binding over the C ABI of ``librope_gb300.so`` (``include/rope.h``).
This module only marshals arguments -- tensor pointers, shapes, attributes,
the current CUDA stream -- and allocates outputs the way the operators' own
JavaScript API does; every step of the computation runs in the library's
CUDA kernels. PyTorch supplies device memory and streams.

There is no CPU fallback: if the library cannot be loaded, every call raises.
"""

import ctypes
import os
import threading

from .build import LIB_PATH, build_library  # noqa: F401

__all__ = [
    "RopeError", "load_library", "build_library", "rope_apply", "mrope_apply",
    "mrope_apply_stream_map", "mrope_stream_map", "rope_apply_fused", "rope_cache_build",
    "rope_apply_qkv", "mrope_apply_qkv",
    "set_variant", "get_variant", "variant",
    "ROPE_OK", "ROPE_ERR_INVALID_ARG", "ROPE_ERR_UNSUPPORTED", "ROPE_ERR_CUDA",
]

ROPE_OK, ROPE_ERR_INVALID_ARG, ROPE_ERR_UNSUPPORTED, ROPE_ERR_CUDA = 0, 1, 2, 3
ROPE_F32, ROPE_F16, ROPE_BF16 = 0, 1, 2
ROPE_SCRATCH_BYTES = 64
VARIANTS = {"auto": 0, "simt": 1, "tma": 2}
_UNSUPPORTED_DTYPE = 99  # passed through so the library reports ROPE_ERR_UNSUPPORTED

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)

# name -> argtypes (restype is the int status unless listed in _RESTYPES)
SIGNATURES = {
    "rope_apply": [_i32, _i32, _i64p, _vp, _vp, _i32, _i64p, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp,
                   _vp],
    "mrope_apply": [_i32, _i32, _i64p, _vp, _vp, _i64, _vp, _vp, _vp, _i32p, _i32, _f32, _i32, _i32,
                    _i32, _i32, _vp, _vp, _vp],
    "mrope_apply_stream_map": [_i32, _i32, _i64p, _vp, _vp, _i64, _vp, _vp, _vp, _u8p, _f32, _i32,
                               _i32, _i32, _vp, _vp, _vp],
    "mrope_stream_map": [_i32p, _i32, _i32, _u8p],
    "rope_apply_fused": [_i32, _i32, _i64p, _vp, _vp, _vp, _f32, _vp, _i32, _i32, _i32, _vp],
    "mrope_apply_fused": [_i32, _i32, _i64p, _vp, _vp, _vp, _f32, _vp, _i32p, _i32, _f32, _i32, _i32, _i32, _vp],
    "rope_cache_build": [_i32, _vp, _i32, _i64, _f32, _vp, _vp, _vp],
    "rope_apply_qkv": [_i32, _i64, _i64, _i32, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _i32,
                       _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp],
    "rope_apply_qkv_rmsnorm": [_i32, _i64, _i64, _i32, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _vp,
                               _i64, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp],
    "mrope_apply_qkv": [_i32, _i64, _i64, _i32, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _vp, _i64, _vp,
                        _i32p, _i32, _f32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp],
    "rope_apply_no_alloc": [_i32, _i32, _i64p, _vp, _vp, _i32, _i64p, _vp, _vp, _vp, _i32, _i32, _i32, _vp,
                            _vp],
    "rope_set_variant": [_i32],
    "rope_get_variant": [],
    "rope_status_string": [_i32],
    "rope_last_error": [],
    "rope_last_kernel": [],
}
_RESTYPES = {"rope_status_string": ctypes.c_char_p, "rope_last_error": ctypes.c_char_p,
             "rope_last_kernel": ctypes.c_char_p}


class RopeError(RuntimeError):
    def __init__(self, fn, status, message):
        self.status = status
        self.message = message
        names = {1: "ROPE_ERR_INVALID_ARG", 2: "ROPE_ERR_UNSUPPORTED", 3: "ROPE_ERR_CUDA"}
        super().__init__(f"{fn}: {names.get(status, status)}: {message}")


def load_library(path=None):
    """Load librope_gb300.so (built in-tree by ``build_library()``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"librope_gb300.so not found at {p}: run "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc); "
                "there is no CPU fallback")
        lib = ctypes.CDLL(p)
        for name, args in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, ctypes.c_int)
        if path is None:
            _lib = lib
        return lib


def _check(fn, status):
    if status != ROPE_OK:
        msg = load_library().rope_last_error().decode()
        raise RopeError(fn, status, msg)


# --------------------------------------------------------------------------
# marshalling helpers (torch is imported lazily: the host-only helpers work
# without it)
# --------------------------------------------------------------------------

def _dtype_code(t):
    import torch

    return {torch.float32: ROPE_F32, torch.float16: ROPE_F16, torch.bfloat16: ROPE_BF16}.get(
        t.dtype, _UNSUPPORTED_DTYPE)


def _shape(t):
    return (ctypes.c_int64 * max(1, t.dim()))(*[int(d) for d in t.shape])


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(name, t, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    return t


def _stream(x, stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    return ctypes.c_void_p(s.cuda_stream)


_scratch = {}


def _scratch_ptr(x, stream, scratch):
    """The scratch argument: None (default) -> the static schedule; a tensor ->
    that buffer (ROPE_SCRATCH_BYTES, zeroed before its first use); "auto" -> one
    zeroed buffer per (device, stream), owned by this module, so launches on one
    stream share it and streams never do."""
    import torch

    if scratch is None or scratch is False:
        return None
    if isinstance(scratch, torch.Tensor):
        _cuda("scratch", scratch)
        if scratch.numel() * scratch.element_size() < ROPE_SCRATCH_BYTES:
            raise ValueError(f"scratch needs {ROPE_SCRATCH_BYTES} bytes")
        return ctypes.c_void_p(scratch.data_ptr())
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    key = (x.device.index, s.cuda_stream)
    buf = _scratch.get(key)
    if buf is None:
        buf = torch.zeros(ROPE_SCRATCH_BYTES // 8, dtype=torch.int64, device=x.device)
        _scratch[key] = buf
    return ctypes.c_void_p(buf.data_ptr())


def _out(x, out):
    import torch

    if out is None:
        return torch.empty_like(x)
    _cuda("out", out, x.dtype)
    if out.shape != x.shape:
        raise ValueError(f"out shape {tuple(out.shape)} != x shape {tuple(x.shape)}")
    return out


# --------------------------------------------------------------------------
# public API (same names as the C ABI)
# --------------------------------------------------------------------------

def rope_apply(x, cos_cache, sin_cache, position_ids=None, *, interleaved=0, rotary_embedding_dim=0,
               num_heads=0, out=None, oor_flag=None, stream=None, scratch=None):
    """RotaryEmbedding (see ``rope_apply`` in include/rope.h). Returns Y."""
    import torch

    lib = load_library()
    _cuda("x", x)
    _cuda("cos_cache", cos_cache)
    _cuda("sin_cache", sin_cache)
    _cuda("position_ids", position_ids, torch.int64)
    _cuda("oor_flag", oor_flag, torch.int32)
    y = _out(x, out)
    with torch.cuda.device(x.device):
        st = lib.rope_apply(_dtype_code(x), x.dim(), _shape(x), _ptr(x), _ptr(y), cos_cache.dim(),
                            _shape(cos_cache), _ptr(cos_cache), _ptr(sin_cache), _ptr(position_ids),
                            int(interleaved), int(rotary_embedding_dim), int(num_heads), _ptr(oor_flag),
                            _scratch_ptr(x, stream, scratch), _stream(x, stream))
    _check("rope_apply", st)
    return y


def mrope_apply(x, cos_cache, sin_cache, position_ids, mrope_section, *, mrope_layout=0, scale=1.0,
                interleaved=0, rotary_embedding_dim=0, num_heads=0, is_packed_batching=0, out=None,
                oor_flag=None, stream=None, scratch=None):
    """MRotaryEmbedding (see ``mrope_apply`` in include/rope.h). Returns Y."""
    import torch

    lib = load_library()
    _cuda("x", x)
    _cuda("cos_cache", cos_cache)
    _cuda("sin_cache", sin_cache)
    _cuda("position_ids", position_ids, torch.int64)
    _cuda("oor_flag", oor_flag, torch.int32)
    y = _out(x, out)
    sec = (ctypes.c_int32 * 3)(*[int(v) for v in mrope_section])
    with torch.cuda.device(x.device):
        st = lib.mrope_apply(_dtype_code(x), x.dim(), _shape(x), _ptr(x), _ptr(y), int(cos_cache.shape[0]),
                             _ptr(cos_cache), _ptr(sin_cache), _ptr(position_ids), sec, int(mrope_layout),
                             float(scale), int(interleaved), int(rotary_embedding_dim), int(num_heads),
                             int(is_packed_batching), _ptr(oor_flag), _scratch_ptr(x, stream, scratch),
                             _stream(x, stream))
    _check("mrope_apply", st)
    return y


def mrope_apply_stream_map(x, cos_cache, sin_cache, position_ids, stream_map, *, scale=1.0, interleaved=0,
                           rotary_embedding_dim=0, num_heads=0, out=None, oor_flag=None, stream=None,
                           scratch=None):
    """MRotaryEmbedding with an explicit stream (0 t, 1 h, 2 w) per half-rotary index."""
    import torch

    lib = load_library()
    _cuda("x", x)
    _cuda("cos_cache", cos_cache)
    _cuda("sin_cache", sin_cache)
    _cuda("position_ids", position_ids, torch.int64)
    _cuda("oor_flag", oor_flag, torch.int32)
    y = _out(x, out)
    m = list(int(v) for v in stream_map)
    arr = (ctypes.c_uint8 * max(1, len(m)))(*m)
    with torch.cuda.device(x.device):
        st = lib.mrope_apply_stream_map(_dtype_code(x), x.dim(), _shape(x), _ptr(x), _ptr(y),
                                        int(cos_cache.shape[0]), _ptr(cos_cache), _ptr(sin_cache),
                                        _ptr(position_ids), arr, float(scale), int(interleaved),
                                        int(rotary_embedding_dim), int(num_heads), _ptr(oor_flag),
                                        _scratch_ptr(x, stream, scratch), _stream(x, stream))
    _check("mrope_apply_stream_map", st)
    return y


def mrope_stream_map(mrope_section, mrope_layout, half):
    """Host helper: the stream of each half-rotary index, as mrope_apply uses it."""
    lib = load_library()
    sec = (ctypes.c_int32 * 3)(*[int(v) for v in mrope_section])
    out = (ctypes.c_uint8 * max(1, int(half)))()
    _check("mrope_stream_map", lib.mrope_stream_map(sec, int(mrope_layout), int(half), out))
    return list(out)[: int(half)]


def rope_apply_fused(x, inv_freq, position_ids, *, attention_scaling=1.0, interleaved=0,
                     rotary_embedding_dim=0, num_heads=0, out=None, stream=None):
    """RotaryEmbedding with cos/sin computed on the fly from inv_freq."""
    import torch

    lib = load_library()
    _cuda("x", x)
    _cuda("inv_freq", inv_freq, torch.float32)
    _cuda("position_ids", position_ids, torch.int64)
    y = _out(x, out)
    with torch.cuda.device(x.device):
        st = lib.rope_apply_fused(_dtype_code(x), x.dim(), _shape(x), _ptr(x), _ptr(y), _ptr(inv_freq),
                                  float(attention_scaling), _ptr(position_ids), int(interleaved),
                                  int(rotary_embedding_dim), int(num_heads), _stream(x, stream))
    _check("rope_apply_fused", st)
    return y


def rope_apply_qkv(query, cos_cache, sin_cache, position_ids=None, *, num_heads, kv_num_heads, key=None,
                   value=None, interleaved=0, rotary_embedding_dim=0, k_cache=None, v_cache=None,
                   past_seq_lens=None, q_out=None, k_out=None, status=None, q_norm_weight=None,
                   k_norm_weight=None, epsilon=1e-6, stream=None, scratch=None):
    """Q and K rotation for grouped-query attention in one launch, optionally
    appending rotated K and V to (B, kv_num_heads, max_len, H) caches in place.
    With q_norm_weight and k_norm_weight (head_size vectors) each Q and K head
    is RMS-normalised first (rope_apply_qkv_rmsnorm).

    query is (B, S, num_heads*H), or packed [Q|K|V] (B, S, (num_heads +
    2*kv_num_heads)*H) when key and value are None. Returns (q_out, k_out);
    k_out is None in cache mode (the caches hold the result). scratch: None,
    or ROPE_SCRATCH_BYTES of zeroed device memory for the dynamic tile schedule
    (one per concurrently running stream).
    """
    import torch

    lib = load_library()
    _cuda("query", query)
    for name, t in (("key", key), ("value", value), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("cos_cache", cos_cache), ("sin_cache", sin_cache)):
        _cuda(name, t, query.dtype)
    _cuda("position_ids", position_ids, torch.int64)
    _cuda("past_seq_lens", past_seq_lens, torch.int32)
    if query.dim() != 3:
        raise ValueError("query must be (B, S, hidden)")
    B, S, hidden = query.shape
    packed = key is None and value is None
    rows_per_tok = num_heads + (2 * kv_num_heads if packed else 0)
    if hidden % rows_per_tok:
        raise ValueError(f"query hidden size {hidden} is not a multiple of {rows_per_tok} heads")
    H = hidden // rows_per_tok
    if q_out is None:
        q_out = torch.empty((B, S, num_heads * H), dtype=query.dtype, device=query.device)
    cache = k_cache is not None
    if not cache and k_out is None:
        k_out = torch.empty((B, S, kv_num_heads * H), dtype=query.dtype, device=query.device)
    max_len = k_cache.shape[2] if cache else 0
    norm = q_norm_weight is not None or k_norm_weight is not None
    _cuda("q_norm_weight", q_norm_weight, query.dtype)
    _cuda("k_norm_weight", k_norm_weight, query.dtype)
    with torch.cuda.device(query.device):
        if norm:
            st = lib.rope_apply_qkv_rmsnorm(
                _dtype_code(query), B, S, int(num_heads), int(kv_num_heads), H, _ptr(query), _ptr(key),
                _ptr(value), _ptr(q_norm_weight), _ptr(k_norm_weight), float(epsilon), _ptr(cos_cache),
                _ptr(sin_cache), int(cos_cache.shape[0]), _ptr(position_ids), _ptr(past_seq_lens),
                int(interleaved), int(rotary_embedding_dim), _ptr(q_out), _ptr(k_out), _ptr(k_cache),
                _ptr(v_cache), int(max_len), _ptr(status), _ptr(scratch), _stream(query, stream))
        else:
            st = lib.rope_apply_qkv(_dtype_code(query), B, S, int(num_heads), int(kv_num_heads), H, _ptr(query),
                                    _ptr(key), _ptr(value), _ptr(cos_cache), _ptr(sin_cache),
                                    int(cos_cache.shape[0]), _ptr(position_ids), _ptr(past_seq_lens),
                                    int(interleaved), int(rotary_embedding_dim), _ptr(q_out), _ptr(k_out),
                                    _ptr(k_cache), _ptr(v_cache), int(max_len), _ptr(status), _ptr(scratch),
                                    _stream(query, stream))
    _check("rope_apply_qkv_rmsnorm" if norm else "rope_apply_qkv", st)
    return q_out, (None if cache else k_out)


def mrope_apply_qkv(query, cos_cache, sin_cache, position_ids, mrope_section, *, num_heads, kv_num_heads,
                    mrope_layout=0, scale=1.0, key=None, value=None, interleaved=0, rotary_embedding_dim=0,
                    k_cache=None, v_cache=None, past_seq_lens=None, q_out=None, k_out=None, status=None,
                    q_norm_weight=None, k_norm_weight=None, epsilon=1e-6, stream=None, scratch=None):
    """rope_apply_qkv with M-RoPE: position_ids is (3, B, S) (t, h, w) and every Q and K
    head is rotated as mrope_apply rotates a head; optional QK-RMSNorm first. Returns
    (q_out, k_out); k_out is None in cache mode."""
    import torch

    lib = load_library()
    _cuda("query", query)
    for name, t in (("key", key), ("value", value), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("cos_cache", cos_cache), ("sin_cache", sin_cache), ("q_norm_weight", q_norm_weight),
                    ("k_norm_weight", k_norm_weight)):
        _cuda(name, t, query.dtype)
    _cuda("position_ids", position_ids, torch.int64)
    _cuda("past_seq_lens", past_seq_lens, torch.int32)
    if query.dim() != 3:
        raise ValueError("query must be (B, S, hidden)")
    B, S, hidden = query.shape
    packed = key is None and value is None
    rows_per_tok = num_heads + (2 * kv_num_heads if packed else 0)
    if hidden % rows_per_tok:
        raise ValueError(f"query hidden size {hidden} is not a multiple of {rows_per_tok} heads")
    H = hidden // rows_per_tok
    if q_out is None:
        q_out = torch.empty((B, S, num_heads * H), dtype=query.dtype, device=query.device)
    cache = k_cache is not None
    if not cache and k_out is None:
        k_out = torch.empty((B, S, kv_num_heads * H), dtype=query.dtype, device=query.device)
    max_len = k_cache.shape[2] if cache else 0
    sec = (ctypes.c_int32 * 3)(*[int(v) for v in mrope_section])
    with torch.cuda.device(query.device):
        st = lib.mrope_apply_qkv(_dtype_code(query), B, S, int(num_heads), int(kv_num_heads), H, _ptr(query),
                                 _ptr(key), _ptr(value), _ptr(q_norm_weight), _ptr(k_norm_weight), float(epsilon),
                                 _ptr(cos_cache), _ptr(sin_cache), int(cos_cache.shape[0]), _ptr(position_ids),
                                 sec, int(mrope_layout), float(scale), _ptr(past_seq_lens), int(interleaved),
                                 int(rotary_embedding_dim), _ptr(q_out), _ptr(k_out), _ptr(k_cache), _ptr(v_cache),
                                 int(max_len), _ptr(status), _ptr(scratch), _stream(query, stream))
    _check("mrope_apply_qkv", st)
    return q_out, (None if cache else k_out)


def mrope_apply_fused(x, inv_freq, position_ids, mrope_section, *, mrope_layout=0, scale=1.0,
                      attention_scaling=1.0, interleaved=0, rotary_embedding_dim=0, num_heads=0, out=None,
                      stream=None):
    """MRotaryEmbedding with cos/sin computed on the fly from inv_freq (three position streams)."""
    import torch

    lib = load_library()
    _cuda("x", x)
    _cuda("inv_freq", inv_freq, torch.float32)
    _cuda("position_ids", position_ids, torch.int64)
    y = _out(x, out)
    sec = (ctypes.c_int32 * 3)(*[int(v) for v in mrope_section])
    with torch.cuda.device(x.device):
        st = lib.mrope_apply_fused(_dtype_code(x), x.dim(), _shape(x), _ptr(x), _ptr(y), _ptr(inv_freq),
                                   float(attention_scaling), _ptr(position_ids), sec, int(mrope_layout),
                                   float(scale), int(interleaved), int(rotary_embedding_dim), int(num_heads),
                                   _stream(x, stream))
    _check("mrope_apply_fused", st)
    return y


def rope_cache_build(inv_freq, rows, dtype=None, *, attention_scaling=1.0, cos_out=None, sin_out=None,
                     stream=None):
    """(rows, len(inv_freq)) cos and sin tables. Returns (cos, sin)."""
    import torch

    lib = load_library()
    _cuda("inv_freq", inv_freq, torch.float32)
    dtype = dtype or torch.float16
    half = int(inv_freq.shape[0])
    if cos_out is None:
        cos_out = torch.empty((int(rows), half), dtype=dtype, device=inv_freq.device)
    if sin_out is None:
        sin_out = torch.empty((int(rows), half), dtype=dtype, device=inv_freq.device)
    _cuda("cos_out", cos_out, dtype)
    _cuda("sin_out", sin_out, dtype)
    code = _dtype_code(cos_out)
    with torch.cuda.device(inv_freq.device):
        st = lib.rope_cache_build(code, _ptr(inv_freq), half, int(rows), float(attention_scaling),
                                  _ptr(cos_out), _ptr(sin_out), _stream(inv_freq, stream))
    _check("rope_cache_build", st)
    return cos_out, sin_out


def set_variant(name):
    """Kernel variant for later calls in this process: "auto", "simt" or "tma"."""
    lib = load_library()
    _check("rope_set_variant", lib.rope_set_variant(VARIANTS[name]))


def get_variant():
    code = load_library().rope_get_variant()
    return {v: k for k, v in VARIANTS.items()}[code]


def last_kernel():
    """Kernel family the calling thread's last launching call used ("" before any)."""
    return load_library().rope_last_kernel().decode()


class variant:
    """Context manager: ``with variant("tma"): ...``."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        self.prev = get_variant()
        set_variant(self.name)
        return self

    def __exit__(self, *exc):
        set_variant(self.prev)
