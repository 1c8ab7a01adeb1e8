"""The growing-cache loop (GPU): decode steps that append one token per
sequence, with the summary builder on a side stream.

The loop runs a few 64-step segments through its captured graph and keeps one
step of each segment aside.  Checked against the fp64 oracle:
  * the lengths and summarised-page counts each kept step saw (the counts
    advance two segments after a page fills, once its build is done);
  * every page built inside the loop, by reconstruction error against the
    oracle's SVD (|e_gpu - e_oracle| <= 1e-3, the builder tolerance of
    test_gpu_parity);
  * each kept step's selection and output, against the oracle's decode step
    on the GPU-built summaries at that step's lengths (selection bit-exact
    outside a 1e-4 band around the cut, output 1e-2, lse 1e-3 relative).
Before the loop, the summaries of the pages that will fill hold large
constant values: a step that read one before its build finished would pick
that page, which the oracle on the final summaries does not.
"""

import numpy as np
import pytest

import oracle as O
from synth import bf16_to_f32, make_case
from tests.helpers import cut_band_ok, oracle_layout_from_abi, to_torch_bf16, torch_bf16_to_u16

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


def _recon_err(K, V_rows, C):
    return np.linalg.norm(K - C @ V_rows) / np.linalg.norm(K)


@pytest.mark.parametrize("form,P", [("unfused", 64), ("fused", 64), ("unfused", 16)])
def test_growing_loop_matches_oracle(form, P):
    """A segment is P steps (one page per sequence fills per segment), at
    64-token pages in both forms of the step and at 16-token pages."""
    from sparse_kv_page_rank_gb300.growing import GrowingLoop
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime

    segments, r, budget = 5, 8, P * 8
    snap = 37 * P // 64
    start = np.array([P * 30, P * 45, P * 20], dtype=np.int32)
    final = start + P * segments
    case = make_case(3, 8, 2, final.tolist(), true_rank=(4, 12), n_carriers=6, seed=90 + P, page_size=P)
    B, Hkv, G = case.batch, case.num_kv_heads, case.group
    dev = "cuda"
    rt = LocksRuntime(to_torch_bf16(case.k_pool, dev), to_torch_bf16(case.v_pool, dev),
                      torch.from_numpy(case.block_table).to(dev), torch.from_numpy(start.copy()).to(dev),
                      torch.from_numpy(start // P).to(dev), case.num_q_heads, r, budget, form=form)
    first = np.concatenate([case.block_table[b, :start[b] // P] for b in range(B)])
    rt.build_summaries(torch.from_numpy(first).to(dev))
    filling = np.stack([case.block_table[b, start[b] // P:final[b] // P] for b in range(B)])  # [B][segments]
    qf = bf16_to_f32(case.q)
    for b in range(B):
        pages = torch.from_numpy(filling[b]).to(dev).long()
        for h in range(Hkv):
            # every basis row along sign(q) of the group's first head: a huge logit for it
            row = np.where(qf[b, h * G] >= 0, 0.5, -0.5).astype(np.float32)
            rt.basis_t[pages, h] = torch.from_numpy(row).to(dev, torch.bfloat16)
            rt.coeffs[pages, h] = 40.0
    q = to_torch_bf16(case.q, dev)

    loop = GrowingLoop(rt, q, snapshot_step=snap)
    res = loop.run(segments, build=True)
    assert rt.device_error() == 0
    assert len(res["build_ms"]) == segments - 1
    snaps = {k: v.cpu().numpy() for k, v in loop.snapshots.items() if k != "out"}
    outs = loop.snapshots["out"]

    # the state each kept step saw
    for s in range(segments):
        assert np.array_equal(snaps["seq_lens"][s], start + P * s + snap + 1), s
        assert np.array_equal(snaps["n_summarized"][s], start // P + max(0, s - 1)), s
    assert np.array_equal(rt.seq_lens.cpu().numpy(), final)
    assert np.array_equal(rt.n_summarized.cpu().numpy(), start // P + segments - 2)

    # the summaries built inside the loop; the last page to fill is not built
    basis_t, coeffs = torch_bf16_to_u16(rt.basis_t), torch_bf16_to_u16(rt.coeffs)
    bt_f, co_f = bf16_to_f32(basis_t).astype(np.float64), bf16_to_f32(coeffs).astype(np.float64)
    kf = O.bf16_widen(case.k_pool)
    for b in range(B):
        for p in filling[b, :segments - 1]:
            for h in range(Hkv):
                V, C, _, _ = O.page_summary(kf[p, h], r)
                e_or = _recon_err(kf[p, h], V.T, C)
                e_gpu = _recon_err(kf[p, h], bt_f[p, h], co_f[p, h])
                assert abs(e_gpu - e_or) <= 1e-3, (b, p, h, e_gpu, e_or)
        assert np.all(np.abs(bt_f[filling[b, -1]]) == 0.5) and np.all(co_f[filling[b, -1]] == 40.0)

    # each kept step against the oracle on the GPU-built summaries
    ob, oc = oracle_layout_from_abi(basis_t, coeffs)
    kmax = budget // P
    for s in range(segments):
        sl, ns = snaps["seq_lens"][s], snaps["n_summarized"][s]
        ref = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, sl, ns, ob, oc, Hkv, budget,
                            page_size=P)
        sel, cnt = snaps["sel_pages"][s], snaps["sel_count"][s]
        for b in range(B):
            for h in range(Hkv):
                k = min(kmax, int(ns[b]))
                assert cnt[b, h] == k, (s, b, h)
                chosen = sel[b, h, :k]
                assert list(chosen) == sorted(chosen)
                assert chosen.max() < ns[b]
                ok, detail = cut_band_ok(ref["sigma"][(b, h)], chosen, ref["sel"][(b, h)], k, BAND)
                assert ok, (s, b, h, detail)
        gsel = {(b, h): sel[b, h, :cnt[b, h]] for b in range(B) for h in range(Hkv)}
        ro, rl = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, sl, ns, gsel, Hkv,
                                 page_size=P)
        go = bf16_to_f32(torch_bf16_to_u16(outs[s])).astype(np.float64)
        gl = snaps["lse"][s].astype(np.float64)
        assert np.isfinite(go).all()
        assert np.abs(go - ro).max() <= OUT_ATOL, (s, np.abs(go - ro).max())
        assert np.all(np.abs(gl - rl) <= LSE_RTOL * np.maximum(1.0, np.abs(rl))), s


def test_growing_loop_rejects_unaligned_start():
    from sparse_kv_page_rank_gb300.growing import GrowingLoop
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime
    case = make_case(1, 4, 1, 64 * 12, true_rank=(4, 8), n_carriers=1, seed=91)
    dev = "cuda"
    for lens, nsum in (([64 * 5 + 3], [5]), ([64 * 5], [4])):
        rt = LocksRuntime(to_torch_bf16(case.k_pool, dev), to_torch_bf16(case.v_pool, dev),
                          torch.from_numpy(case.block_table).to(dev), torch.tensor(lens, dtype=torch.int32).to(dev),
                          torch.tensor(nsum, dtype=torch.int32).to(dev), 4, 8, 256)
        with pytest.raises(ValueError):
            GrowingLoop(rt, to_torch_bf16(case.q, dev))
