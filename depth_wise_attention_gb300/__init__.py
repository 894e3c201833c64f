"""GB300-native Attention Residuals depth-wise softmax read.

The compute path is ``libattnres.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/attnres.h``); ``depth_wise_attention_gb300.attnres``
is a thin ctypes binding with the same entry-point names.  The library is
loaded on first use, and a missing library is an error: there is no fallback.
"""
__all__ = ["attnres", "inputs"]
