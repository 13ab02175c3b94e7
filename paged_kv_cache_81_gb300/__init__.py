"""GB300-native paged KV-cache data movement (slot mapping, cache write, xfer_list, pack, unpack).

The compute path is the CUDA library ``libpagedkv.so`` (sm_103a), reached through
the ctypes binding in ``pagedkv``.  Importing this package loads nothing; the
library is loaded on first use and a missing library raises at once.
"""
__all__ = ["pagedkv", "workloads"]
