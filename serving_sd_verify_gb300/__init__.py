"""GB300-native block verification for lossless speculative decoding.

libsdverify.so (csrc/, C ABI in include/sd_verify.h) holds the CUDA kernels;
`sd_verify` is its thin ctypes binding, `build` compiles it in-tree for
sm_103a, and `workloads` draws the seeded synthetic inputs.
"""
__all__ = ["build", "sd_verify", "workloads"]
