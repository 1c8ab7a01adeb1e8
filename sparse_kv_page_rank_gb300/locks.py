"""Thin ctypes binding of liblocks.so (argument marshalling only).

Every function here has the name of the C entry point it wraps and does
nothing but turn tensors into raw device pointers, fill the C structs and
check the returned status; all compute runs in the library's CUDA kernels.
Tensors are torch tensors (device memory, streams) or raw integer pointers.
The library must have been built (``sparse_kv_page_rank_gb300.build_lib``);
a missing library raises instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "liblocks.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "locks.h")

LOCKS_OK = 0
LOCKS_ERR_INVALID_ARG = 1
LOCKS_ERR_UNSUPPORTED = 2
LOCKS_ERR_CUDA = 3
LOCKS_ERR_WORKSPACE = 4
LOCKS_ERR_DEVICE = 5
# bytes of the library-owned workspace behind locks_decode_step_static
LOCKS_STATIC_WS_BYTES = 8 << 20
LOCKS_DTYPE_BF16 = 0
LOCKS_DTYPE_F32 = 1
LOCKS_DTYPE_Q4 = 2
LOCKS_DTYPE_BF16_PACKED = 3
LOCKS_FLAG_UNFUSED = 0x1
LOCKS_FLAG_FUSED = 0x2


def q4_page_head_bytes(rank: int, page_size: int = 64) -> int:
    """Bytes of one page-head of a LOCKS_DTYPE_Q4 summary (LOCKS_Q4_BLOCK_BYTES)."""
    return (72 * rank + page_size * rank + 132 + 15) // 16 * 16
LOCKS_DEVERR_BLOCK_TABLE = 0x1
LOCKS_DEVERR_SEL_PAGE = 0x2
LOCKS_DEVERR_LENGTHS = 0x4
LOCKS_DEVERR_PAGE_ID = 0x8
LOCKS_DEVERR_TIMEOUT = 0x10


class LocksError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class locks_cache_t(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("n_summarized", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("pages_total", ctypes.c_int32),
                ("max_pages", ctypes.c_int32)]


class locks_summary_t(ctypes.Structure):
    _fields_ = [("basis_t", ctypes.c_void_p), ("coeffs", ctypes.c_void_p),
                ("rank", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class locks_params_t(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("budget_tokens", ctypes.c_int32),
                ("scale", ctypes.c_float), ("flags", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load liblocks.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"liblocks.so not built ({LIB_PATH}); run "
                               "python -m sparse_kv_page_rank_gb300.build_lib")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        C, S, R = P(locks_cache_t), P(locks_summary_t), P(locks_params_t)
        sig = {
            "locks_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "locks_workspace_size": (ctypes.c_int, [C, S, R, P(sz)]),
            "locks_workspace_init": (ctypes.c_int, [vp, sz, vp]),
            "locks_build_summaries": (ctypes.c_int, [C, S, vp, i32, vp, sz, vp]),
            "locks_select": (ctypes.c_int, [C, S, R, vp, vp, vp, vp, vp, sz, vp]),
            "locks_page_scores": (ctypes.c_int, [C, S, R, vp, vp, vp, sz, vp]),
            "locks_sparse_attend": (ctypes.c_int, [C, R, vp, vp, vp, vp, vp, vp, sz, vp]),
            "locks_decode_step": (ctypes.c_int, [C, S, R, vp, vp, vp, vp, vp, vp, sz, vp]),
            "locks_decode_step_launches": (ctypes.c_int, [C, S, R, P(i32)]),
            "locks_dense_decode": (ctypes.c_int, [C, R, vp, vp, vp, vp, sz, vp]),
            "locks_exact_page_lse": (ctypes.c_int, [C, R, vp, vp, vp]),
            "locks_get_device_error": (ctypes.c_int, [vp, P(i32), vp]),
            "locks_decode_step_static": (ctypes.c_int, [C, S, R, vp, vp, vp, vp, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def declared_symbols() -> list[str]:
    """Entry points declared in include/locks.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"LOCKS_API\s+[\w\s\*]+?\b(locks_\w+)\s*\(", text)))


def status_string(status: int) -> str:
    return lib().locks_status_string(int(status)).decode()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != LOCKS_OK:
        raise LocksError(status, what)


def make_cache(k_pool, v_pool, block_table, seq_lens, n_summarized=None, *, pages_total=None,
               num_kv_heads=None) -> locks_cache_t:
    """C struct for a paged cache given as tensors [pages_total][Hkv][P][d]."""
    pt, hkv, P, d = (k_pool.shape if k_pool is not None and hasattr(k_pool, "shape")
                     else (pages_total, num_kv_heads, 64, 128))
    return locks_cache_t(_ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(seq_lens),
                         _ptr(n_summarized), int(block_table.shape[0]), int(hkv), int(d), int(P),
                         int(pt), int(block_table.shape[1]))


def make_summary(basis_t, coeffs, rank: int, dtype: int = LOCKS_DTYPE_BF16) -> locks_summary_t:
    return locks_summary_t(_ptr(basis_t), _ptr(coeffs), int(rank), int(dtype))


def make_params(num_q_heads: int, budget_tokens: int, scale: float = 0.0, flags: int = 0) -> locks_params_t:
    return locks_params_t(int(num_q_heads), int(budget_tokens), float(scale), int(flags))


def locks_workspace_size(cache, summary, params) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().locks_workspace_size(ctypes.byref(cache), ctypes.byref(summary) if summary else None,
                                      ctypes.byref(params), ctypes.byref(n)), "locks_workspace_size")
    return int(n.value)


def locks_workspace_init(ws, nbytes: int, stream=None):
    _check(lib().locks_workspace_init(_ptr(ws), int(nbytes), _stream(stream)), "locks_workspace_init")


def locks_build_summaries(cache, summary, page_ids, n: int, ws=None, ws_bytes: int = 0, stream=None):
    _check(lib().locks_build_summaries(ctypes.byref(cache), ctypes.byref(summary), _ptr(page_ids), int(n),
                                       _ptr(ws), int(ws_bytes), _stream(stream)), "locks_build_summaries")


def locks_select(cache, summary, params, q, sel_pages, sel_count, page_lse, ws, ws_bytes: int, stream=None):
    _check(lib().locks_select(ctypes.byref(cache), ctypes.byref(summary), ctypes.byref(params), _ptr(q),
                              _ptr(sel_pages), _ptr(sel_count), _ptr(page_lse), _ptr(ws), int(ws_bytes),
                              _stream(stream)), "locks_select")


def locks_page_scores(cache, summary, params, q, page_lse, ws, ws_bytes: int, stream=None):
    _check(lib().locks_page_scores(ctypes.byref(cache), ctypes.byref(summary), ctypes.byref(params), _ptr(q),
                                   _ptr(page_lse), _ptr(ws), int(ws_bytes), _stream(stream)),
           "locks_page_scores")


def locks_sparse_attend(cache, params, q, sel_pages, sel_count, out, lse, ws, ws_bytes: int, stream=None):
    _check(lib().locks_sparse_attend(ctypes.byref(cache), ctypes.byref(params), _ptr(q), _ptr(sel_pages),
                                     _ptr(sel_count), _ptr(out), _ptr(lse), _ptr(ws), int(ws_bytes),
                                     _stream(stream)), "locks_sparse_attend")


def locks_decode_step(cache, summary, params, q, out, lse, sel_pages, sel_count, ws, ws_bytes: int,
                      stream=None):
    _check(lib().locks_decode_step(ctypes.byref(cache), ctypes.byref(summary), ctypes.byref(params), _ptr(q),
                                   _ptr(out), _ptr(lse), _ptr(sel_pages), _ptr(sel_count), _ptr(ws),
                                   int(ws_bytes), _stream(stream)), "locks_decode_step")


def locks_decode_step_static(cache, summary, params, q, out, lse, sel_pages=None, sel_count=None,
                             device_error=None, stream=None):
    """locks_decode_step in the library's own fixed device workspace (no
    workspace argument; for callers that cannot allocate device memory)."""
    _check(lib().locks_decode_step_static(ctypes.byref(cache), ctypes.byref(summary), ctypes.byref(params),
                                          _ptr(q), _ptr(out), _ptr(lse), _ptr(sel_pages), _ptr(sel_count),
                                          _ptr(device_error), _stream(stream)), "locks_decode_step_static")


def locks_decode_step_launches(cache, summary, params) -> int:
    n = ctypes.c_int32(0)
    _check(lib().locks_decode_step_launches(ctypes.byref(cache), ctypes.byref(summary), ctypes.byref(params),
                                            ctypes.byref(n)), "locks_decode_step_launches")
    return n.value


def locks_dense_decode(cache, params, q, out, lse, ws, ws_bytes: int, stream=None):
    _check(lib().locks_dense_decode(ctypes.byref(cache), ctypes.byref(params), _ptr(q), _ptr(out), _ptr(lse),
                                    _ptr(ws), int(ws_bytes), _stream(stream)), "locks_dense_decode")


def locks_exact_page_lse(cache, params, q, page_lse, stream=None):
    _check(lib().locks_exact_page_lse(ctypes.byref(cache), ctypes.byref(params), _ptr(q), _ptr(page_lse),
                                      _stream(stream)), "locks_exact_page_lse")


def locks_get_device_error(ws, stream=None) -> int:
    """Returns the device error bits (0 = none) and clears them."""
    code = ctypes.c_int32(0)
    st = lib().locks_get_device_error(_ptr(ws), ctypes.byref(code), _stream(stream))
    if st not in (LOCKS_OK, LOCKS_ERR_DEVICE):
        raise LocksError(st, "locks_get_device_error")
    return int(code.value)
