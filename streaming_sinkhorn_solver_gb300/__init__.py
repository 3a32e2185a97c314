"""GB300-native streaming Sinkhorn solver (FlashSinkhorn hot path).

The compute path is the C-ABI library ``libflashsinkhorn.so`` built from
``csrc/`` for sm_103a; ``binding`` is a thin ctypes layer over it.  Importing
this package does not load the library; the first call does, and fails loudly
if it was not built.
"""
from .workloads import WORKLOADS, make_inputs  # noqa: F401

__all__ = ["WORKLOADS", "make_inputs"]
