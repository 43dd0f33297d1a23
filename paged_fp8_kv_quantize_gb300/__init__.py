"""paged_fp8_kv_quantize_gb300 -- paged FP8 (e4m3) KV cache for decode
attention on GB300: quantize-on-append, tag-checked split-KV paged decode
attention (FP8 and BF16 caches), as a C-ABI CUDA library (libpfkv.so,
include/pfkv.h) with a thin ctypes binding.

Importing the package does not load the library; ``from
paged_fp8_kv_quantize_gb300 import abi`` does, and fails loudly if it is not
built.
"""

__all__ = ["abi", "synth", "build"]
