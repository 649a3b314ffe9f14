"""GB300-native physically sparse QSA decode.

The compute path is the C-ABI library ``libqsa.so`` (hand-written sm_103a
CUDA kernels, declared in ``include/qsa.h``); ``top_group_sparse_gb300.qsa``
is its thin ctypes binding.  Importing this package loads nothing: the
binding loads the library on first use and raises if it is missing.
"""

__all__ = ["qsa", "workloads"]
