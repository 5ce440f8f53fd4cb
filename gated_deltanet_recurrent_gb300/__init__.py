"""Slot-indexed Gated DeltaNet layer for GB300 (sm_103a).

The compute lives in libgdn.so (hand-written CUDA behind the C ABI declared
in include/gdn.h); `abi` is its Python binding and `synth` the seeded
synthetic-input generators.  Importing the package loads nothing; the first
call into `abi` loads the library and raises if it has not been built.
"""
