"""Reference oracle for rotary position embedding (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path never does, and the
two share no code. The arithmetic lives in ``rope_oracle.c`` (plain C,
single-threaded, binary64 unless the definition fixes float32); this module
only compiles it and marshals numpy arrays through ctypes.
"""

from .oracle import (  # noqa: F401
    BF16_BITS,
    bf16_to_double,
    build,
    cache_build,
    double_to_bf16,
    double_to_half,
    half_to_double,
    mrope,
    mrope_fused,
    mrope_map,
    mrope_qkv,
    mrope_stream_map,
    rope,
    rope_fused,
    rope_qkv,
)
