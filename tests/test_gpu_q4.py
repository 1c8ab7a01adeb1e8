"""Parity of the quantised, centred summary format (LOCKS_DTYPE_Q4: int4
basis, int8 coefficients and centroid, as in the explainer's §2
"Kernmechanisme", Kwantisatie) with the fp64 oracle (GPU).

The oracle quantises its own centred SVD summaries; the same codes and
scales, packed in the ABI layout, go to the GPU, and both sides then compute
from the values the codes stand for.  Tolerances as for bf16 summaries: page
LSE 1e-3 relative, selection bit-exact outside a 1e-4 band around the cut,
output 1e-2 absolute, lse 1e-3 relative.  The builder's own quantised
summaries are checked by their reconstruction error against the oracle's
(within 1e-3) and by the planted carrier pages they keep.
"""

import numpy as np
import pytest

import oracle as O
from synth import bf16_to_f32, make_case
from tests.helpers import (cut_band_ok, make_runtime, oracle_summaries_q4, to_torch_bf16, torch_bf16_to_u16,
                           unpack_q4)

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


def _run_q4_case(case, r, budget):
    nsum = [case.n_full_pages(b) for b in range(case.batch)]
    packed, basis, coeffs, cent = oracle_summaries_q4(case, r)
    rt, q = make_runtime(case, r, budget, nsum, quantized=True)
    rt.set_summaries(torch.from_numpy(packed).to("cuda"), None)
    page_lse = torch.full((case.batch, case.num_q_heads, case.max_pages), float("nan"), device="cuda")
    rt.select(q, page_lse)
    out, lse = rt.decode_step(q)
    torch.cuda.synchronize()
    assert rt.device_error() == 0
    ref = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, basis, coeffs,
                        case.num_kv_heads, budget, centroid=cent)
    G = case.group
    pl = page_lse.cpu().numpy()
    sel = rt.sel_pages.cpu().numpy()
    cnt = rt.sel_count.cpu().numpy()
    kmax = min(budget // 64, case.max_pages)
    for b in range(case.batch):
        for h in range(case.num_kv_heads):
            shat = ref["shat"][(b, h)]
            n = shat.shape[1]
            got = pl[b, h * G:(h + 1) * G, :n]
            err = np.abs(got - shat) / np.maximum(1.0, np.abs(shat))
            assert err.size == 0 or err.max() <= LSE_RTOL, (b, h, err.max())
            k = min(kmax, n)
            assert cnt[b, h] == k
            chosen = sel[b, h, :k]
            assert list(chosen) == sorted(chosen)
            ok, detail = cut_band_ok(ref["sigma"][(b, h)], chosen, ref["sel"][(b, h)], k, BAND)
            assert ok, (b, h, detail)
    gsel = {(b, h): sel[b, h, :cnt[b, h]] for b in range(case.batch) for h in range(case.num_kv_heads)}
    ro, rl = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, gsel,
                             case.num_kv_heads)
    go = bf16_to_f32(torch_bf16_to_u16(out)).astype(np.float64)
    assert np.isfinite(go).all()
    assert np.abs(go - ro).max() <= OUT_ATOL
    gl = lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.all(np.abs(gl[fin] - rl[fin]) <= LSE_RTOL * np.maximum(1, np.abs(rl[fin])))


@pytest.mark.parametrize("G,Hkv,r", [(4, 2, 8), (16, 1, 8), (8, 1, 4), (1, 2, 2), (2, 3, 6)])
def test_q4_select_and_step_ragged(G, Hkv, r):
    case = make_case(2, G * Hkv, Hkv, [64 * 41 + 17, 64 * 37], true_rank=(2, 12), n_carriers=2, seed=40 + G + r)
    _run_q4_case(case, r, 640)


def test_q4_many_scan_chunks():
    case = make_case(1, 8, 2, 64 * 2600 + 5, true_rank=(4, 12), n_carriers=16, seed=47)
    _run_q4_case(case, 8, 2048)


@pytest.mark.parametrize("r", [2, 4, 8])
def test_q4_builder_reconstruction_and_carriers(r):
    case = make_case(1, 8, 2, 64 * 96, true_rank=(2, 12), n_carriers=4, seed=50 + r)
    rt, q = make_runtime(case, r, 64 * 8, quantized=True)
    pages = np.array([case.block_table[0, j] for j in range(case.n_full_pages(0))], dtype=np.int32)
    rt.build_summaries(torch.from_numpy(pages).to("cuda"))
    torch.cuda.synchronize()
    assert rt.device_error() == 0
    blocks = rt.basis_t.cpu().numpy()
    worst = 0.0
    for p in pages:
        for h in range(case.num_kv_heads):
            K = O.bf16_widen(case.k_pool[p, h])
            g = unpack_q4(blocks[p, h], r)
            assert np.abs(g["vq"]).max() <= 7 and np.abs(g["cq"]).max() <= 127 and np.abs(g["muq"]).max() <= 127
            Vg, Cg, mug = O.dequantize_summary(g)
            Vo, Co, muo = O.dequantize_summary(O.quantized_page_summary(K, r))
            de = abs(O.reconstruction_error(K, Vg, Cg, mug) - O.reconstruction_error(K, Vo, Co, muo))
            worst = max(worst, de)
    assert worst <= 1e-3, worst
    # the builder's own summaries still find the planted carrier pages
    rt.decode_step(q)
    torch.cuda.synchronize()
    sel = rt.sel_pages.cpu().numpy()
    cnt = rt.sel_count.cpu().numpy()
    for h in range(case.num_kv_heads):
        chosen = set(sel[0, h, :cnt[0, h]].tolist())
        carriers = [int(c) for c in case.carriers[0, h] if c >= 0]
        assert all(c in chosen for c in carriers), (h, carriers, sorted(chosen))


def test_q4_builder_is_deterministic():
    """Two builds of the same pages give the same bytes (a race inside the
    builder would show here first)."""
    case = make_case(1, 8, 2, 64 * 300, true_rank=(2, 12), n_carriers=4, seed=61)
    pages = torch.from_numpy(np.array([case.block_table[0, j] for j in range(case.n_full_pages(0))],
                                      dtype=np.int32)).to("cuda")
    blocks = []
    for _ in range(3):
        rt, _q = make_runtime(case, 8, 64 * 8, quantized=True)
        rt.build_summaries(pages)
        torch.cuda.synchronize()
        assert rt.device_error() == 0
        blocks.append(rt.basis_t.clone())
    assert torch.equal(blocks[0], blocks[1]) and torch.equal(blocks[0], blocks[2])
