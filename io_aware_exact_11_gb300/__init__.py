"""Exact IO-aware tiled softmax attention for NVIDIA GB300 (sm_103a).

The compute lives in ``libfa.so`` (hand-written CUDA behind a C ABI, see
``include/fa.h``); ``io_aware_exact_11_gb300.fa`` is the thin ctypes binding.
Importing this package loads nothing: the library is opened on first use and
an error is raised if it has not been built.
"""

__all__ = ["fa", "inputs"]
