"""Parity at the bench's full sizes, on sampled problems.

The two bench workloads, llama128k (1 sequence, 32 query / 8 KV heads, 131072
tokens, r = 8, budget 2048) and ctx1m (1 sequence, 32 / 2 heads, 1048576
tokens, r = 8, budget 2048), run through the C ABI in the launch configuration
bench.py times (the plan depends on the shapes only).  The oracle cannot do
every problem at this size in seconds, so it computes sampled (sequence, KV
head) problems one by one, on oracle-built summaries; the GPU runs the whole
workload.  Tolerances as in test_gpu_parity: page LSE 1e-3 relative,
selection bit-exact outside a 1e-4 band around the cut, output 1e-2 absolute,
lse 1e-3 relative.
"""

import numpy as np
import pytest

import oracle as O
from synth import bf16_bits, bf16_to_f32, make_config_case
from tests.helpers import cut_band_ok, make_runtime, oracle_layout_from_abi, to_torch_bf16, torch_bf16_to_u16

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LSE_RTOL = 1e-3
OUT_ATOL = 1e-2
BAND = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_page_rank_gb300.build_lib import build
    build()


def _summaries_for_heads(case, r, heads):
    """Oracle summaries (bf16, C-ABI layout) of every full page for the listed
    KV heads; other heads get zero summaries (their results are not checked)."""
    pt, hkv, P, d = case.k_pool.shape
    basis_t = np.zeros((pt, hkv, r, d), dtype=np.uint16)
    coeffs = np.zeros((pt, hkv, P, r), dtype=np.uint16)
    for b in range(case.batch):
        for p in case.block_table[b, :case.n_full_pages(b)]:
            for h in heads:
                V, C, _, _ = O.page_summary(O.bf16_widen(case.k_pool[int(p), h]), r)
                basis_t[int(p), h] = bf16_bits(V.T.astype(np.float32))
                coeffs[int(p), h] = bf16_bits(C.astype(np.float32))
    return basis_t, coeffs


@pytest.mark.parametrize("name,heads", [("llama128k", (0, 5)), ("ctx1m", (1,))])
def test_full_size_sampled_problems(name, heads):
    case, cfg = make_config_case(name)
    r, budget = cfg["rank"], cfg["budget_tokens"]
    G, b = case.group, 0
    nsum = [case.n_full_pages(x) for x in range(case.batch)]
    basis_t, coeffs = _summaries_for_heads(case, r, heads)
    rt, q = make_runtime(case, r, budget, nsum)
    rt.set_summaries(to_torch_bf16(basis_t, "cuda"), to_torch_bf16(coeffs, "cuda"))
    page_lse = torch.full((case.batch, case.num_q_heads, case.max_pages), float("nan"), device="cuda")
    rt.select(q, page_lse)
    out, lse = rt.decode_step(q)
    out, lse = out.clone(), lse.clone()
    dout, dlse = rt.dense_decode(q)
    torch.cuda.synchronize()
    assert rt.device_error() == 0
    pl = page_lse.cpu().numpy()
    sel = rt.sel_pages.cpu().numpy()
    cnt = rt.sel_count.cpu().numpy()
    go = bf16_to_f32(torch_bf16_to_u16(out)).astype(np.float64)
    gd = bf16_to_f32(torch_bf16_to_u16(dout)).astype(np.float64)
    gl, gdl = lse.cpu().numpy(), dlse.cpu().numpy()
    kmax = min(budget // 64, case.max_pages)

    for h in heads:
        # problem (b, h) alone: one sequence, one KV head and its G query heads
        hs = slice(h * G, (h + 1) * G)
        qh = case.q[b:b + 1, hs]
        kh, vh = case.k_pool[:, h:h + 1], case.v_pool[:, h:h + 1]
        ob, oc = oracle_layout_from_abi(basis_t[:, h:h + 1], coeffs[:, h:h + 1])
        bt, sl, ns = case.block_table[b:b + 1], case.seq_lens[b:b + 1], np.asarray(nsum[b:b + 1])
        ref = O.decode_step(qh, kh, vh, bt, sl, ns, ob, oc, 1, budget)

        shat = ref["shat"][(0, 0)]
        n = shat.shape[1]
        err = np.abs(pl[b, hs, :n] - shat) / np.maximum(1.0, np.abs(shat))
        assert err.max() <= LSE_RTOL, (name, h, err.max())

        k = min(kmax, n)
        assert cnt[b, h] == k
        chosen = sel[b, h, :k]
        assert list(chosen) == sorted(chosen)
        ok, detail = cut_band_ok(ref["sigma"][(0, 0)], chosen, ref["sel"][(0, 0)], k, BAND)
        assert ok, (name, h, detail)

        # output over the GPU's own selection (the selection is checked above)
        ro, rl = O.sparse_decode(qh, kh, vh, bt, sl, ns, {(0, 0): chosen}, 1)
        assert np.abs(go[b, hs] - ro[0]).max() <= OUT_ATOL
        assert np.all(np.abs(gl[b, hs] - rl[0]) <= LSE_RTOL * np.maximum(1.0, np.abs(rl[0])))

        do, dl = O.dense_decode(qh, kh, vh, bt, sl, 1)
        assert np.abs(gd[b, hs] - do[0]).max() <= OUT_ATOL
        assert np.all(np.abs(gdl[b, hs] - dl[0]) <= LSE_RTOL * np.maximum(1.0, np.abs(dl[0])))
