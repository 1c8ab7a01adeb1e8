"""The decode step with the top-k inside the attention kernel (GPU).

With LOCKS_FLAG_FUSED, locks_decode_step runs as two kernels (the scan, then
attention whose thread-block clusters compute the group-shared top-k
themselves) for 64-token pages with k_max <= 32 and at most 128 pages per CTA
of a 16-CTA cluster; otherwise, and by default, as three kernels (scan, top-k,
attention).  Both forms are checked against the fp64 oracle with the
tolerances of test_gpu_parity (page LSE 1e-3 relative, selection bit-exact
outside a 1e-4 band around the cut, output 1e-2 absolute, lse 1e-3 relative),
and against each other: the same pages, and outputs within 1e-2.
"""

import numpy as np
import pytest

import oracle as O
from synth import bf16_to_f32, make_case, make_config_case
from tests.helpers import (cut_band_ok, make_runtime, oracle_layout_from_abi, oracle_summaries_bf16,
                           to_torch_bf16, torch_bf16_to_u16)

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

OUT_ATOL = 1e-2
LSE_RTOL = 1e-3
BAND = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_page_rank_gb300.build_lib import build
    build()


def _runtime(case, r, budget, nsum, basis_t, coeffs, form):
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime
    rt = LocksRuntime(to_torch_bf16(case.k_pool, "cuda"), to_torch_bf16(case.v_pool, "cuda"),
                      torch.from_numpy(case.block_table).cuda(), torch.from_numpy(case.seq_lens).cuda(),
                      torch.tensor(np.asarray(nsum, dtype=np.int32)).cuda(), case.num_q_heads, r, budget,
                      form=form)
    rt.set_summaries(to_torch_bf16(basis_t, "cuda"), to_torch_bf16(coeffs, "cuda"))
    return rt


def _step(rt, q):
    rt.sel_pages.fill_(-7)
    rt.sel_count.fill_(-7)
    out, lse = rt.decode_step(q)
    torch.cuda.synchronize()
    assert rt.device_error() == 0
    return (bf16_to_f32(torch_bf16_to_u16(out)).astype(np.float64), lse.cpu().numpy().astype(np.float64),
            rt.sel_pages.cpu().numpy(), rt.sel_count.cpu().numpy())


def _check(case, r, budget, nsum=None, expect_fused=True):
    if nsum is None:
        nsum = [case.n_full_pages(b) for b in range(case.batch)]
    basis_t, coeffs = oracle_summaries_bf16(case, r)
    q = to_torch_bf16(case.q, "cuda")
    rf = _runtime(case, r, budget, nsum, basis_t, coeffs, form="fused")
    ru = _runtime(case, r, budget, nsum, basis_t, coeffs, form="unfused")
    assert rf.decode_step_launches() == (2 if expect_fused else 3)
    assert ru.decode_step_launches() == 3
    fo, fl, fsel, fcnt = _step(rf, q)
    uo, ul, usel, ucnt = _step(ru, q)
    ob, oc = oracle_layout_from_abi(basis_t, coeffs)
    ref = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, ob, oc,
                        case.num_kv_heads, budget)
    P = case.page_size
    kmax = min(budget // P, case.max_pages)
    for b in range(case.batch):
        for h in range(case.num_kv_heads):
            n = min(int(nsum[b]), int(case.seq_lens[b]) // P)
            k = min(kmax, n)
            for sel, cnt in ((fsel, fcnt), (usel, ucnt)):
                assert cnt[b, h] == k, (b, h, cnt[b, h], k)
                chosen = sel[b, h, :k]
                assert list(chosen) == sorted(chosen)
                if k < n:
                    ok, detail = cut_band_ok(ref["sigma"][(b, h)], chosen, ref["sel"][(b, h)], k, BAND)
                    assert ok, (b, h, detail)
                else:
                    assert list(chosen) == list(range(n))
            assert list(fsel[b, h, :k]) == list(usel[b, h, :k]), (b, h)
    gsel = {(b, h): fsel[b, h, :fcnt[b, h]] for b in range(case.batch) for h in range(case.num_kv_heads)}
    ro, rl = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, gsel,
                             case.num_kv_heads, page_size=P)
    for go, gl in ((fo, fl), (uo, ul)):
        assert np.isfinite(go).all()
        assert np.abs(go - ro).max() <= OUT_ATOL, np.abs(go - ro).max()
        fin = np.isfinite(rl)
        assert np.all(np.isfinite(gl) == fin)
        assert np.all(np.abs(gl[fin] - rl[fin]) <= LSE_RTOL * np.maximum(1, np.abs(rl[fin])))
    assert np.abs(fo - uo).max() <= OUT_ATOL


@pytest.mark.parametrize("G,Hkv,r,pages,budget_pages", [
    (4, 2, 8, 2047, 32),    # 16 CTAs, 128 pages per CTA, partial last chunk, k = 32
    (4, 8, 8, 300, 16),     # many problems, smaller clusters
    (1, 1, 8, 64, 8),       # the tiny shape: 8 pages per CTA
    (2, 3, 4, 1000, 5),     # k not a power of two
    (16, 1, 8, 1500, 32),   # G = 16 (four s_hat loads per page)
    (3, 2, 6, 777, 7),      # G = 3 (scalar s_hat loads)
    (8, 1, 16, 129, 1),     # k = 1, two pages per list boundary
])
def test_fused_step_matches_oracle_and_unfused(G, Hkv, r, pages, budget_pages):
    case = make_case(2, G * Hkv, Hkv, [64 * pages + 37, 64 * (pages // 2)], true_rank=(2, 12), n_carriers=4,
                     seed=700 + G + pages, spare_pages=2)
    _check(case, r, 64 * budget_pages)


def test_fused_step_tail_and_unsummarised_pages():
    """Unsummarised full pages join the open tail, which the fused kernel
    orders first and loads before its dependency wait."""
    case = make_case(3, 8, 2, [64 * 400 + 9, 64 * 250 + 63, 64 * 90], true_rank=(4, 10), n_carriers=2, seed=71)
    _check(case, 8, 64 * 12, nsum=[397, 240, 90])


def test_fused_step_budget_covers_every_page():
    """No selection needed (k_max >= summarised pages): every page is
    attended, which is dense attention."""
    case = make_case(2, 8, 2, [64 * 20 + 5, 64 * 17], true_rank=(2, 8), n_carriers=2, seed=72)
    _check(case, 8, 64 * 32)


def test_fused_step_zero_budget_attends_only_the_tail():
    case = make_case(2, 4, 1, [64 * 50 + 30, 64 * 40], true_rank=(2, 8), n_carriers=1, seed=73)
    _check(case, 4, 32)  # budget below one page: k_max = 0


def test_fused_step_equal_keys_tie_to_lower_pages():
    """Every logical page maps to one physical page, so all scores are
    bit-identical: the first k pages must be chosen in both forms."""
    case = make_case(1, 4, 1, 64 * 700, true_rank=(4, 8), n_carriers=0, seed=74)
    case.block_table[0, :700] = case.block_table[0, 3]
    _check(case, 8, 64 * 20)


def test_fused_step_not_taken_beyond_its_envelope():
    """More than 2048 pages (128 per CTA of a 16-CTA cluster), or k above 32,
    runs the three-kernel form; the results still match the oracle."""
    case = make_case(1, 4, 1, 64 * 2100 + 3, true_rank=(2, 12), n_carriers=4, seed=75)
    _check(case, 8, 64 * 16, expect_fused=False)
    case = make_case(1, 4, 2, 64 * 300, true_rank=(2, 12), n_carriers=4, seed=76)
    _check(case, 8, 64 * 40, expect_fused=False)


@pytest.mark.slow
def test_fused_step_llama128k_sampled():
    """The 128K workload (8 KV heads x 2048 pages, k = 32) through both forms,
    with oracle summaries for two KV heads (the others stay zero)."""
    case, cfg = make_config_case("llama128k")
    from tests.test_gpu_shapes import _summaries
    heads = [(0, 2), (0, 6)]
    basis_t, coeffs = _summaries(case, cfg["rank"], heads)
    nsum = [case.n_full_pages(0)]
    q = to_torch_bf16(case.q, "cuda")
    rf = _runtime(case, cfg["rank"], cfg["budget_tokens"], nsum, basis_t, coeffs, form="fused")
    assert rf.decode_step_launches() == 2
    fo, fl, fsel, fcnt = _step(rf, q)
    del rf
    ru = _runtime(case, cfg["rank"], cfg["budget_tokens"], nsum, basis_t, coeffs, form="unfused")
    uo, ul, usel, ucnt = _step(ru, q)
    del ru
    G = case.group
    for b, h in heads:
        hs = slice(h * G, (h + 1) * G)
        ob, oc = oracle_layout_from_abi(basis_t[:, h:h + 1], coeffs[:, h:h + 1])
        bt, sl, ns = case.block_table[b:b + 1], case.seq_lens[b:b + 1], np.asarray(nsum)
        ref = O.decode_step(case.q[b:b + 1, hs], case.k_pool[:, h:h + 1], case.v_pool[:, h:h + 1], bt, sl, ns,
                            ob, oc, 1, cfg["budget_tokens"])
        k = 32
        assert fcnt[b, h] == k and ucnt[b, h] == k
        ok, detail = cut_band_ok(ref["sigma"][(0, 0)], fsel[b, h, :k], ref["sel"][(0, 0)], k, BAND)
        assert ok, detail
        assert list(fsel[b, h, :k]) == list(usel[b, h, :k])
        ro, rl = O.sparse_decode(case.q[b:b + 1, hs], case.k_pool[:, h:h + 1], case.v_pool[:, h:h + 1], bt, sl, ns,
                                 {(0, 0): fsel[b, h, :k]}, 1)
        assert np.abs(fo[b, hs] - ro[0]).max() <= OUT_ATOL
        assert np.abs(uo[b, hs] - ro[0]).max() <= OUT_ATOL
        assert np.all(np.abs(fl[b, hs] - rl[0]) <= LSE_RTOL * np.maximum(1.0, np.abs(rl[0])))


def test_default_form_is_three_kernels():
    """Without a flag the step takes the three-kernel form, whatever the
    number of (sequence, KV head) problems; LOCKS_FLAG_FUSED takes the
    two-kernel form within its limits."""
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for batch in (1, sms // 8 + 1):
        k = torch.zeros((4 * batch, 8, 64, 128), dtype=torch.bfloat16, device="cuda")
        bt = torch.arange(4 * batch, dtype=torch.int32, device="cuda").view(batch, 4)
        sl = torch.full((batch,), 256, dtype=torch.int32, device="cuda")
        ns = torch.full((batch,), 4, dtype=torch.int32, device="cuda")
        assert LocksRuntime(k, k, bt, sl, ns, 32, 8, 128).decode_step_launches() == 3, (batch, sms)
        assert LocksRuntime(k, k, bt, sl, ns, 32, 8, 128, form="fused").decode_step_launches() == 2, (batch, sms)
