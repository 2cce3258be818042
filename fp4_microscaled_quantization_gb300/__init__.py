"""GB300-native fused Hadamard rotation + 4-bit microscaled quantizer and
block-scaled FP4 GEMM.

The compute lives in the CUDA library ``libfp4q.so`` (C ABI declared in
``include/fp4q.h``); :mod:`.fp4q` is the thin ctypes binding with the same
names.  Importing this package loads nothing; the binding loads the library on
first use and raises if it has not been built.
"""
__all__ = ["fp4q", "synth"]
