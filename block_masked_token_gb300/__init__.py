"""GB300-native (sm_103a) hot path of MARS block-masked multi-token decoding.

The compute lives in `libmars.so` (hand-written CUDA behind a C ABI declared in
include/mars.h); `block_masked_token_gb300.mars` is a thin ctypes binding with the same
entry-point names. Importing this package does not load the library; the first call
into `mars` does, and fails loudly if it was not built.
"""
__all__ = ["mars", "workloads"]
