"""Parity at the sizes the C ABI promises beyond the bench workloads (GPU).

include/locks.h accepts any group size G = num_q_heads / num_kv_heads in
1..16 and any even rank r in 2..16.  Group sizes that are not powers of two
take other code: the top-k scores fewer pages per CTA (1024) and loads the
scores head by head, and the scan runs its G <= 4 packed template at G = 3,
the 5..8 template at G = 6 and the two-row-half template at G = 9..15.  Ranks
above 8 use the scan's two-n-tile template.  This file also runs the
rank/batch-sweep shape at its full batch of 8 and the 1M-context workload at
16-token pages (65536 pages per KV head, whose top-k merges 64 chunks of 128
candidates each), on sampled problems.

Tolerances as in test_gpu_parity: page LSE 1e-3 relative, selection bit-exact
outside a 1e-4 band around the cut, output 1e-2 absolute, lse 1e-3 relative.
"""

import numpy as np
import pytest

import oracle as O
from synth import bf16_bits, bf16_to_f32, make_case, make_config_case
from tests.helpers import cut_band_ok, make_runtime, oracle_layout_from_abi, to_torch_bf16, torch_bf16_to_u16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

LSE_RTOL = 1e-3
OUT_ATOL = 1e-2
BAND = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_page_rank_gb300.build_lib import build
    build()


def _summaries(case, r, problems):
    """Oracle rank-r summaries (bf16, C-ABI layout) of every full page of the
    listed (sequence, KV head) problems; other page-heads stay zero (their
    results are not checked)."""
    pt, hkv, P, d = case.k_pool.shape
    basis_t = np.zeros((pt, hkv, r, d), dtype=np.uint16)
    coeffs = np.zeros((pt, hkv, P, r), dtype=np.uint16)
    for b, h in problems:
        for p in case.block_table[b, :case.n_full_pages(b)]:
            V, C, _, _ = O.page_summary(O.bf16_widen(case.k_pool[int(p), h]), r)
            basis_t[int(p), h] = bf16_bits(V.T.astype(np.float32))
            coeffs[int(p), h] = bf16_bits(C.astype(np.float32))
    return basis_t, coeffs


def _check_problems(case, r, budget, problems, nsum=None, dense=True):
    """Run select, decode_step (and the dense decode) on the whole case through
    the C ABI; check the listed problems one by one against the oracle."""
    P = case.page_size
    if nsum is None:
        nsum = [case.n_full_pages(b) for b in range(case.batch)]
    basis_t, coeffs = _summaries(case, r, problems)
    rt, q = make_runtime(case, r, budget, nsum)
    rt.set_summaries(to_torch_bf16(basis_t, "cuda"), to_torch_bf16(coeffs, "cuda"))
    page_lse = torch.full((case.batch, case.num_q_heads, case.max_pages), float("nan"), device="cuda")
    rt.select(q, page_lse)
    out, lse = rt.decode_step(q)
    out, lse = out.clone(), lse.clone()
    if dense:
        dout, dlse = rt.dense_decode(q)
    torch.cuda.synchronize()
    assert rt.device_error() == 0
    G = case.group
    pl = page_lse.cpu().numpy()
    sel = rt.sel_pages.cpu().numpy()
    cnt = rt.sel_count.cpu().numpy()
    go = bf16_to_f32(torch_bf16_to_u16(out)).astype(np.float64)
    gl = lse.cpu().numpy()
    if dense:
        gd = bf16_to_f32(torch_bf16_to_u16(dout)).astype(np.float64)
        gdl = dlse.cpu().numpy()
    kmax = min(budget // P, case.max_pages)
    for b, h in problems:
        hs = slice(h * G, (h + 1) * G)
        qh = case.q[b:b + 1, hs]
        kh, vh = case.k_pool[:, h:h + 1], case.v_pool[:, h:h + 1]
        ob, oc = oracle_layout_from_abi(basis_t[:, h:h + 1], coeffs[:, h:h + 1])
        bt, sl, ns = case.block_table[b:b + 1], case.seq_lens[b:b + 1], np.asarray(nsum[b:b + 1])
        ref = O.decode_step(qh, kh, vh, bt, sl, ns, ob, oc, 1, budget, page_size=P)
        shat = ref["shat"][(0, 0)]
        n = shat.shape[1]
        err = np.abs(pl[b, hs, :n] - shat) / np.maximum(1.0, np.abs(shat))
        assert err.size == 0 or err.max() <= LSE_RTOL, (b, h, err.max())
        k = min(kmax, n)
        assert cnt[b, h] == k
        chosen = sel[b, h, :k]
        assert list(chosen) == sorted(chosen)
        ok, detail = cut_band_ok(ref["sigma"][(0, 0)], chosen, ref["sel"][(0, 0)], k, BAND)
        assert ok, (b, h, detail)
        ro, rl = O.sparse_decode(qh, kh, vh, bt, sl, ns, {(0, 0): chosen}, 1, page_size=P)
        assert np.abs(go[b, hs] - ro[0]).max() <= OUT_ATOL, (b, h, np.abs(go[b, hs] - ro[0]).max())
        assert np.all(np.abs(gl[b, hs] - rl[0]) <= LSE_RTOL * np.maximum(1.0, np.abs(rl[0])))
        if dense:
            do, dl = O.dense_decode(qh, kh, vh, bt, sl, 1, page_size=P)
            assert np.abs(gd[b, hs] - do[0]).max() <= OUT_ATOL
            assert np.all(np.abs(gdl[b, hs] - dl[0]) <= LSE_RTOL * np.maximum(1.0, np.abs(dl[0])))


def _all(case):
    return [(b, h) for b in range(case.batch) for h in range(case.num_kv_heads)]


@pytest.mark.parametrize("G,Hkv,pages", [(3, 2, 2300), (6, 2, 700), (12, 1, 2100), (5, 3, 300), (9, 1, 1500),
                                         (15, 1, 400)])
def test_group_sizes_not_power_of_two(G, Hkv, pages):
    """G = 3, 5, 6, 9, 12, 15 with ragged lengths; at 2300 and 2100 pages the
    top-k of a non-power-of-two group (1024 pages per CTA) merges three
    chunks' candidates."""
    case = make_case(2, G * Hkv, Hkv, [64 * pages + 21, 64 * (pages // 2) + 40], true_rank=(2, 12),
                     n_carriers=4, seed=300 + G, spare_pages=5)
    _check_problems(case, 8, 64 * 24, _all(case))


@pytest.mark.parametrize("G,Hkv,r", [(4, 2, 6), (4, 2, 10), (2, 2, 14), (16, 1, 14), (6, 1, 12), (1, 3, 10)])
def test_bf16_ranks_between_the_powers_of_two(G, Hkv, r):
    """Even ranks 6, 10, 12, 14 in bf16 (ranks above 8 take the scan's
    two-n-tile path, whose second basis tile is partly empty here)."""
    case = make_case(2, G * Hkv, Hkv, [64 * 200 + 33, 64 * 150], true_rank=(2, 16), n_carriers=3, seed=400 + r + G)
    _check_problems(case, r, 64 * 12, _all(case))


@pytest.mark.slow
def test_sweep_shape_at_batch_8():
    """The rank/batch-sweep workload as the bench runs it: 8 sequences of 32768
    tokens, 32 query / 8 KV heads, true page ranks 2..16, r = 8, budget 1024;
    64 problems in one launch, four of them checked against the oracle."""
    case, cfg = make_config_case("sweep")
    assert case.batch == 8
    _check_problems(case, cfg["rank"], cfg["budget_tokens"], [(0, 0), (3, 5), (6, 2), (7, 7)])


@pytest.mark.slow
def test_ctx1m_at_16_token_pages():
    """1M context at 16-token pages: 65536 pages per KV head, k = 128, and the
    top-k's 64 chunks at G = 16 (1024 pages each) merged in one CTA through
    its radix select (64 x 128 candidates); one KV head checked."""
    case, cfg = make_config_case("ctx1m", page_size=16)
    assert case.max_pages == 65536
    _check_problems(case, cfg["rank"], cfg["budget_tokens"], [(0, 1)], dense=False)


@pytest.mark.parametrize("G,Hkv,r", [(3, 2, 8), (6, 1, 6), (12, 1, 4)])
def test_q4_group_sizes_not_power_of_two(G, Hkv, r):
    """The quantised format (int4 basis, int8 coefficients and centroid) at
    group sizes 3, 6 and 12, one per scan template."""
    from tests.test_gpu_q4 import _run_q4_case
    case = make_case(2, G * Hkv, Hkv, [64 * 300 + 7, 64 * 180], true_rank=(2, 12), n_carriers=2, seed=500 + G + r)
    _run_q4_case(case, r, 64 * 10)


@pytest.mark.parametrize("G,Hkv,r", [(3, 2, 8), (12, 1, 10)])
def test_page16_group_sizes_not_power_of_two(G, Hkv, r):
    """16-token pages at G = 3 (2 chunks of 1024 pages in the top-k) and at
    G = 12 with rank 10."""
    case = make_case(2, G * Hkv, Hkv, [16 * 1900 + 5, 16 * 700 + 16], true_rank=(2, 12), n_carriers=3,
                     seed=600 + G + r, page_size=16)
    _check_problems(case, r, 16 * 40, _all(case))
