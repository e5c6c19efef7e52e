"""PQ-compressed KV-cache decode attention for GB300 (sm_103a).

The compute lives in ``libaqpq.so`` (hand-written CUDA behind a C ABI, see
``include/aqpq.h``); this package is the thin Python binding over it plus host
arithmetic (byte counts, split planning).  Importing the package does not load
the library; the first call does, and fails loudly if it is missing.
"""
__all__ = ["traffic"]
