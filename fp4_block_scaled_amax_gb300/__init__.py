"""GB300-native FP4 block-scaled linear-layer hot path.

The compute lives in `libfp4.so` (hand-written sm_103a CUDA kernels behind a
C ABI declared in include/fp4.h).  `fp4_block_scaled_amax_gb300.fp4` is the thin
ctypes binding with the same entry-point names; `synth` draws the seeded
synthetic inputs.  Importing this package does not load the library; the first
call through the binding does, and raises if the library is missing.
"""

__all__ = ["fp4", "synth"]
