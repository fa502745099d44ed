"""fp8bs: the FP8 (e4m3) block-scaled linear layer on B300 (sm_103a).

The compute lives in the C-ABI library ``libfp8bs.so`` (hand-written CUDA,
declared in ``include/fp8bs.h``); ``fp8_block_scaled_18_b300.fp8bs`` is the thin
ctypes binding with the same call names.  Importing the binding raises if the
library has not been built: there is no other code path.
"""
__version__ = "0.1.0"
