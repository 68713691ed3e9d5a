"""GB300-native quantized paged KV cache.

The compute path is the C-ABI library ``libkvq.so`` (hand-written CUDA for
sm_103a); :mod:`.kvq` is a thin ctypes binding over it.  Importing this package
does not load the library; the binding loads it on first import and raises if
it is missing.
"""
__all__ = ["kvq", "workloads"]
