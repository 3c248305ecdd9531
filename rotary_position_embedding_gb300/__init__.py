"""GB300-native rotary position embedding (RoPE / M-RoPE).

Placeholder during bring-up; the binding is added with the CUDA library.
"""
