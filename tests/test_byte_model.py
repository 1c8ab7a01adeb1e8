"""The byte model in bench.py (resident summary bytes, per-step bytes, dense
bytes) checked against figures the LOCKS pages print.  The figures and their
citations live in tests/golden/pages_figures.json.  These pins need no GPU:
they check the arithmetic bench.py reports its effective bandwidth and KV-read
reduction with, in the pages' own quantised summary format (int4 basis, int8
coefficients and centroid, 16-token pages)."""
import json
import os

import pytest

import bench

HERE = os.path.dirname(os.path.abspath(__file__))
FIG = json.load(open(os.path.join(HERE, "golden", "pages_figures.json")))


def _close(got, want, rel):
    return abs(got - want) <= rel * abs(want)


def _residency(fmt):
    return bench.residency(fmt["rank"], page=fmt["page"], d=fmt["head_dim"], basis_bits=fmt["basis_bits"],
                           coef_bits=fmt["coef_bits"], centroid_bits=fmt["centroid_bits"])


@pytest.mark.parametrize("name", ["residency_r8", "residency_r2"])
def test_residency_matches_pages(name):
    f = FIG[name]
    assert _close(_residency(f["format"]), f["value"], f["rel_tol"])


@pytest.mark.parametrize("name", ["residency_r8", "residency_r2"])
def test_library_q4_block_matches_pages(name):
    # the library's LOCKS_DTYPE_Q4 block at the pages' page size, against the
    # page's own K + V bytes
    from sparse_kv_page_rank_gb300.locks import q4_page_head_bytes
    f = FIG[name]
    fmt = f["format"]
    kv = 2 * fmt["page"] * fmt["head_dim"] * 2
    assert _close(q4_page_head_bytes(fmt["rank"], fmt["page"]) / kv, f["value"], f["rel_tol"])


def _reduction(rank, context, budget):
    # per page-head: dense reads K+V of every token; the step reads every
    # summary (quantised format) plus K+V of the budget's tokens
    fmt = dict(FIG["residency_r8"]["format"], rank=rank)
    kv_per_token = 2 * fmt["head_dim"] * 2
    dense = context * kv_per_token
    step = _residency(fmt) * dense + budget * kv_per_token
    return dense / step


def test_kv_read_reduction_at_1m():
    f = FIG["kv_read_reduction_1m_r8"]
    w = f["workload"]
    assert _close(_reduction(w["rank"], w["context"], w["budget_tokens"]), f["value"], f["rel_tol"])


def test_kv_read_reduction_range():
    f = FIG["kv_read_reduction_range"]
    lo, hi = f["value"]
    r_hi, r_lo = f["ranks"]
    assert _close(_reduction(r_hi, 1 << 20, 2048), lo, f["rel_tol"])
    assert _close(_reduction(r_lo, 1 << 20, 2048), hi, f["rel_tol"])


def test_dense_bytes_llama_128k():
    f = FIG["llama31_8b_kv_128k_gib"]
    m = f["model"]
    # dense_bytes covers one layer (K+V of every token, q and o); q/o are tiny
    per_layer = bench.dense_bytes(1, m["kv_heads"], 4, m["context"])
    assert _close(m["layers"] * per_layer / 2**30, f["value"], f["rel_tol"])


def test_step_bytes_budget_fraction():
    f = FIG["attended_fraction"]
    w = f["workload"]
    P = bench.P
    k = w["budget_tokens"] // P
    sb = bench.step_bytes(1, 1, 1, w["context"] // P, k, 0, 8)
    dense_kv = bench.dense_bytes(1, 1, 1, w["context"]) - 2 * bench.D * 2
    assert _close(sb["selected_kv"] / dense_kv, f["value"], f["rel_tol"])
