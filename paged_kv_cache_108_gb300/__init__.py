"""GB300-native paged-KV decode attention.

The compute path lives in ``libpa.so`` (hand-written sm_103a CUDA kernels
behind a C ABI, declared in ``include/pa.h``).  ``ops`` is the thin Python
binding; ``pool`` wraps the native host-side block pool; ``synth`` draws the
seeded synthetic workloads.  Importing the package loads nothing native; the
first call into ``ops`` does, and fails loudly if the library is missing.
"""
__all__ = ["ops", "pool", "synth", "build"]
