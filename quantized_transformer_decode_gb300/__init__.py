"""GB300-native forward pass of a Qwen3-style dense decoder over GGUF Q8_0 weights.

The compute runs in the CUDA library `libqw3.so` (C ABI declared in
include/qw3.h); `quantized_transformer_decode_gb300.qw3` is its thin ctypes
binding. `inputs` holds the seeded synthetic workloads. Importing the package
loads nothing native; `qw3.load()` does, and fails loudly when the library is
missing.
"""
