"""GB300-native ResidualAttention over a disaggregated, copy-on-write KV cache.

The compute path lives in ``libforkkv.so`` (C-ABI, hand-written CUDA for
sm_103a, declared in ``include/forkkv.h``).  ``forkkv`` is the thin ctypes
binding: argument marshalling only.  Importing this package does not load the
library; the first call that needs it does, and raises if it is missing.
"""
__all__ = ["forkkv", "workload"]
