"""LoPA (Lookahead Parallel Decoding) branch-verification step for GB300 (sm_103a).

The decoding path lives in liblopa.so (C ABI, include/lopa.h), built in-tree by
``build.build()``.  ``api`` marshals arguments to it; ``synth`` generates the seeded
synthetic workloads.  Nothing here computes the method in Python.
"""
__all__ = ["api", "synth", "build"]
__version__ = "0.1.0"
