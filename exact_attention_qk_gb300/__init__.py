"""GB300-native exact attention forward (FlashAttention-style) behind a C ABI.

The CUDA library `libfa.so` (built from `csrc/`) holds every kernel; `fa`
marshals arguments into it. Importing this package does not load the library;
`exact_attention_qk_gb300.fa` does, and raises if it is missing.
"""
__all__ = ["inputs", "fa", "build"]
