"""GB300-native block-FP8 mixture-of-experts layer forward.

The compute lives in ``libmoefp8.so`` (hand-written CUDA for sm_103a behind a C ABI, declared in
``include/moefp8.h``); ``ops`` is a thin ctypes binding with the same entry-point names.  The
library is loaded on first use and a missing or unbuildable library raises -- there is no CPU
fallback.
"""
__all__ = ["ops", "workloads"]
