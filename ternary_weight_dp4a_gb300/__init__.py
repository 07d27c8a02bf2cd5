"""GB300 (sm_103a) ternary-weight FFN decode path.

The compute lives in ``libtq.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/tq.h``).  ``ternary_weight_dp4a_gb300.tq`` is the thin
ctypes binding; ``ternary_weight_dp4a_gb300.synth`` draws seeded inputs.
Importing the package does not load the library; the first call into ``tq``
does, and raises if the CUDA library has not been built.
"""
__all__ = ["tq", "synth"]
