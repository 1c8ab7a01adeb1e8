"""C-ABI checks that need no GPU: the library builds, loads, exports every
entry point declared in include/locks.h, and rejects bad host arguments with
the documented status codes before launching anything."""

import ctypes
import os
import subprocess
from pathlib import Path

import pytest

from sparse_kv_page_rank_gb300 import locks as L
from sparse_kv_page_rank_gb300.build_lib import LIB, build

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    build()
    return L.lib()


def test_library_exports_every_declared_symbol(lib):
    declared = L.declared_symbols()
    assert len(declared) == 13, declared
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared:
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing but the declared API leaks out of the library
    assert {n for n in exported if n.startswith("locks_")} == set(declared)


def test_library_has_no_torch_or_driver_dependency(lib):
    out = subprocess.run(["ldd", LIB], capture_output=True, text=True).stdout
    assert "libtorch" not in out and "libcuda.so" not in out and "libc10" not in out


def test_status_strings(lib):
    assert L.status_string(0) == "LOCKS_OK"
    assert L.status_string(2) == "LOCKS_ERR_UNSUPPORTED"
    assert L.status_string(99) == "LOCKS_ERR_UNKNOWN"


def _cache(**kw):
    d = dict(k_pool=0x1000, v_pool=0x2000, block_table=0x3000, seq_lens=0x4000, n_summarized=0x5000,
             batch=1, num_kv_heads=2, head_dim=128, page_size=64, pages_total=10, max_pages=10)
    d.update(kw)
    return L.locks_cache_t(**d)


def test_sixteen_token_pages_accepted(lib):
    p = L.make_params(8, 512)
    a = L.locks_workspace_size(_cache(page_size=16, max_pages=40, pages_total=40), None, p)
    b = L.locks_workspace_size(_cache(page_size=64), None, p)
    # four times the pages per token budget: more selected pages, more candidates
    assert a > b > 0 and a % 256 == 0


def _header_q4_block_bytes(r, P):
    """Evaluates LOCKS_Q4_BLOCK_BYTES as written in include/locks.h."""
    import re
    text = (ROOT / "include" / "locks.h").read_text()
    m = re.search(r"#define LOCKS_Q4_BLOCK_BYTES\(r, P\) (.+)", text)
    expr = m.group(1).replace("(r)", str(r)).replace("(P)", str(P)).replace("/", "//")
    return eval(expr)


@pytest.mark.parametrize("r", [2, 4, 6, 8])
@pytest.mark.parametrize("P", [16, 64])
def test_q4_block_bytes_agree(r, P):
    from helpers import q4_block_bytes
    assert _header_q4_block_bytes(r, P) == L.q4_page_head_bytes(r, P) == q4_block_bytes(r, P)
    assert L.q4_page_head_bytes(r, P) % 16 == 0


def test_workspace_size_grows_with_shapes(lib):
    p = L.make_params(8, 512)
    a = L.locks_workspace_size(_cache(), None, p)
    b = L.locks_workspace_size(_cache(batch=4, max_pages=100, pages_total=400), None, p)
    assert a > 0 and b > a and a % 256 == 0


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), L.LOCKS_ERR_UNSUPPORTED),
    (dict(page_size=32), L.LOCKS_ERR_UNSUPPORTED),
    (dict(batch=0), L.LOCKS_ERR_INVALID_ARG),
    (dict(max_pages=0), L.LOCKS_ERR_INVALID_ARG),
])
def test_bad_cache_rejected(lib, kw, status):
    with pytest.raises(L.LocksError) as e:
        L.locks_workspace_size(_cache(**kw), None, L.make_params(8, 512))
    assert e.value.status == status


@pytest.mark.parametrize("params,status", [
    (L.make_params(7, 512), L.LOCKS_ERR_INVALID_ARG),      # not a multiple of Hkv
    (L.make_params(34, 512), L.LOCKS_ERR_UNSUPPORTED),     # G = 17
    (L.make_params(8, -1), L.LOCKS_ERR_INVALID_ARG),
    (L.make_params(8, 512, flags=4), L.LOCKS_ERR_INVALID_ARG),      # a reserved flag bit
    (L.make_params(8, 512, flags=3), L.LOCKS_ERR_INVALID_ARG),      # both forms requested
    (L.make_params(8, 512, scale=-1.0), L.LOCKS_ERR_INVALID_ARG),
])
def test_bad_params_rejected(lib, params, status):
    with pytest.raises(L.LocksError) as e:
        L.locks_workspace_size(_cache(), None, params)
    assert e.value.status == status


@pytest.mark.parametrize("rank,dtype,status", [
    (3, 0, L.LOCKS_ERR_UNSUPPORTED), (18, 0, L.LOCKS_ERR_UNSUPPORTED), (0, 0, L.LOCKS_ERR_UNSUPPORTED),
    (8, 1, L.LOCKS_ERR_UNSUPPORTED), (8, 7, L.LOCKS_ERR_INVALID_ARG),
])
def test_bad_summary_rejected_before_launch(lib, rank, dtype, status):
    s = L.locks_summary_t(0x10000, 0x20000, rank, dtype)
    ws = ctypes.c_void_p(0x100000)
    with pytest.raises(L.LocksError) as e:
        L.locks_select(_cache(), s, L.make_params(8, 512), 0x9000, 0xA000, 0xB000, None, ws.value, 1 << 30, 0)
    assert e.value.status == status


def test_packed_summary_needs_no_coefficient_array(lib):
    """LOCKS_DTYPE_BF16_PACKED (one block per page-head) passes the summary
    checks with coeffs NULL and stops only at the missing workspace; the
    two-array layout without coeffs is rejected."""
    p = L.make_params(8, 512)
    for dtype, status in ((L.LOCKS_DTYPE_BF16_PACKED, L.LOCKS_ERR_WORKSPACE),
                          (L.LOCKS_DTYPE_BF16, L.LOCKS_ERR_INVALID_ARG)):
        with pytest.raises(L.LocksError) as e:
            L.locks_select(_cache(), L.make_summary(0x10000, None, 8, dtype), p, 0x9000, 0xA000, 0xB000, None,
                           None, 0, 0)
        assert e.value.status == status, dtype


def test_workspace_checks_before_launch(lib):
    s = L.locks_summary_t(0x10000, 0x20000, 8, 0)
    p = L.make_params(8, 512)
    need = L.locks_workspace_size(_cache(), s, p)
    for ws, nbytes in ((None, need), (0x100010, need), (0x100000, need - 1)):
        with pytest.raises(L.LocksError) as e:
            L.locks_select(_cache(), s, p, 0x9000, 0xA000, 0xB000, None, ws, nbytes, 0)
        assert e.value.status == L.LOCKS_ERR_WORKSPACE


def test_null_pointers_rejected(lib):
    p = L.make_params(8, 512)
    with pytest.raises(L.LocksError) as e:
        L.locks_dense_decode(_cache(k_pool=None), p, 0x9000, 0xA000, None, 0x100000, 1 << 30, 0)
    assert e.value.status == L.LOCKS_ERR_INVALID_ARG
    with pytest.raises(L.LocksError) as e:
        L.locks_decode_step(_cache(), L.locks_summary_t(0x10000, 0x20000, 8, 0), p, 0x9000, 0xA000, None,
                            0xC000, None, 0x100000, 1 << 30, 0)  # sel_pages without sel_count
    assert e.value.status == L.LOCKS_ERR_INVALID_ARG
    with pytest.raises(L.LocksError) as e:
        L.locks_get_device_error(None, 0)
    assert e.value.status == L.LOCKS_ERR_INVALID_ARG


def test_misaligned_pool_rejected(lib):
    with pytest.raises(L.LocksError) as e:
        L.locks_dense_decode(_cache(k_pool=0x1008), L.make_params(8, 512), 0x9000, 0xA000, None, 0x100000,
                             1 << 30, 0)
    assert e.value.status == L.LOCKS_ERR_INVALID_ARG


def test_product_path_never_imports_oracle():
    """The binding and runtime must not reach the CPU oracle."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "sparse_kv_page_rank_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_decode_step_launches_validates_its_arguments(lib):
    """locks_decode_step_launches checks its arguments like the step itself."""
    cache, summary, params = _cache(), L.make_summary(16, 16, 8), L.make_params(8, 512)
    with pytest.raises(L.LocksError) as e:
        L.locks_decode_step_launches(cache, L.make_summary(16, 16, 3), params)
    assert e.value.status == L.LOCKS_ERR_UNSUPPORTED
    with pytest.raises(L.LocksError) as e:
        L.locks_decode_step_launches(cache, summary, L.make_params(7, 512))
    assert e.value.status == L.LOCKS_ERR_INVALID_ARG
    # the three-kernel form on request
    assert L.locks_decode_step_launches(cache, summary, L.make_params(8, 512, flags=L.LOCKS_FLAG_UNFUSED)) == 3
