"""GB300-native fused reduce + residual add + RMSNorm (TokenWeave's hot path).

The compute runs in ``libtw.so`` (hand-written sm_103a CUDA behind a C ABI);
:mod:`.tw` is the thin ctypes binding and :mod:`.inputs` the seeded synthetic
input generator.  Importing the package does not load the CUDA library; the
binding loads it on first use and raises if it is missing.
"""
__all__ = ["inputs", "tw"]
