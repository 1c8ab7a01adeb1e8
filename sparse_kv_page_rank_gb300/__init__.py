"""LOCKS decode-step library for GB300 (sm_103a).

The compute lives in ``_lib/liblocks.so`` (C ABI in ``include/locks.h``);
``sparse_kv_page_rank_gb300.locks`` is its ctypes binding and
``sparse_kv_page_rank_gb300.runtime`` holds the device-side state of one cache
(tensors, structs, workspace) for callers that use PyTorch for memory.
Importing this package loads nothing; the library is loaded on first use.
"""
