"""Parity of the CUDA path with the fp64 oracle (GPU).

Tolerances (fixed up front):
  * page LSE s_hat: |gpu - oracle| <= 1e-3 * max(1, |oracle|), given identical
    (bf16) summaries;
  * selection: bit-exact set equality, excluding pages whose GSA score lies
    within 1e-4 of the k-th largest oracle score; exactly k pages, ascending;
  * attention output: max |gpu - oracle| <= 1e-2 on bf16 inputs (the output
    itself is bf16, ~4e-3 relative rounding), lse within 1e-3 relative;
  * summaries: |e_gpu - e_oracle| <= 1e-3 for the relative reconstruction
    error e = ||K - C V^T||_F / ||K||_F.
Inputs: seeded synthetic page-local low-rank caches (synth), with ragged
lengths, partial tail pages, unsummarised full pages, several scan / top-k
chunks, G in {1, 2, 4, 16} and r in {2, 4, 8, 16}.  bf16 summaries are in the
runtime's packed layout (LOCKS_DTYPE_BF16_PACKED) unless a case asks for the
two-array layout (LOCKS_DTYPE_BF16).
"""

import math

import numpy as np
import pytest

import oracle as O
from synth import make_case, make_config_case, bf16_to_f32
from tests.helpers import (cut_band_ok, make_runtime, oracle_layout_from_abi, oracle_summaries_bf16,
                           to_torch_bf16, torch_bf16_to_u16)

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


def _upload_summaries(rt, basis_t, coeffs):
    rt.set_summaries(to_torch_bf16(basis_t, rt.device), to_torch_bf16(coeffs, rt.device))


def _run_case(case, r, budget, nsum=None, check_dense=True, split=False):
    """Identical-summary parity of select, decode_step and dense decode."""
    if nsum is None:
        nsum = [case.n_full_pages(b) for b in range(case.batch)]
    basis_t, coeffs = oracle_summaries_bf16(case, r)
    rt, q = make_runtime(case, r, budget, nsum, split=split)
    _upload_summaries(rt, basis_t, coeffs)
    page_lse = torch.full((case.batch, case.num_q_heads, case.max_pages), float("nan"), device="cuda")
    rt.select(q, page_lse)
    out, lse = rt.decode_step(q)
    torch.cuda.synchronize()
    assert rt.device_error() == 0

    ob, oc = oracle_layout_from_abi(basis_t, coeffs)
    ref = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, ob, oc,
                        case.num_kv_heads, budget)
    G = case.group
    pl = page_lse.cpu().numpy()
    sel = rt.sel_pages.cpu().numpy()
    cnt = rt.sel_count.cpu().numpy()
    kmax = min(budget // 64, case.max_pages)
    worst_lse = 0.0
    for b in range(case.batch):
        for h in range(case.num_kv_heads):
            shat = ref["shat"][(b, h)]
            n = shat.shape[1]
            got = pl[b, h * G:(h + 1) * G, :n]
            err = np.abs(got - shat) / np.maximum(1.0, np.abs(shat))
            worst_lse = max(worst_lse, float(err.max()) if err.size else 0.0)
            assert err.size == 0 or err.max() <= LSE_RTOL, (b, h, err.max())
            k = min(kmax, n)
            assert cnt[b, h] == k
            chosen = sel[b, h, :k]
            assert list(chosen) == sorted(chosen)
            ok, detail = cut_band_ok(ref["sigma"][(b, h)], chosen, ref["sel"][(b, h)], k, BAND)
            assert ok, (b, h, detail)
    # output over the GPU's own selection (selection verified above)
    gsel = {(b, h): sel[b, h, :cnt[b, h]] for b in range(case.batch) for h in range(case.num_kv_heads)}
    ro, rl = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, gsel,
                             case.num_kv_heads)
    go = bf16_to_f32(torch_bf16_to_u16(out)).astype(np.float64)
    assert np.isfinite(go).all()
    assert np.abs(go - ro).max() <= OUT_ATOL, np.abs(go - ro).max()
    gl = lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.all(np.isfinite(gl) == fin)
    assert np.all(np.abs(gl[fin] - rl[fin]) <= LSE_RTOL * np.maximum(1, np.abs(rl[fin])))
    if check_dense:
        dout, dlse = rt.dense_decode(q)
        do, dl = O.dense_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                case.num_kv_heads)
        gd = bf16_to_f32(torch_bf16_to_u16(dout)).astype(np.float64)
        assert np.abs(gd - do).max() <= OUT_ATOL, np.abs(gd - do).max()
        gdl = dlse.cpu().numpy()
        fin = np.isfinite(dl)
        assert np.all(np.abs(gdl[fin] - dl[fin]) <= LSE_RTOL * np.maximum(1, np.abs(dl[fin])))
    return rt, q, ref, worst_lse


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("G,Hkv,r", [(4, 2, 8), (1, 1, 8), (2, 3, 4), (16, 2, 8), (4, 2, 16), (8, 1, 2)])
def test_select_and_step_ragged(G, Hkv, r, split):
    case = make_case(2, G * Hkv, Hkv, [64 * 41 + 17, 64 * 37], true_rank=(2, 12), n_carriers=2,
                     seed=100 + G + r, spare_pages=3)
    _run_case(case, r, budget=64 * 6, split=split)


def test_unsummarised_full_pages_join_the_tail():
    case = make_case(2, 8, 2, [64 * 30 + 9, 64 * 25 + 63], true_rank=(4, 10), n_carriers=2, seed=7)
    _run_case(case, 8, budget=64 * 5, nsum=[27, 20])


@pytest.mark.parametrize("G,pages", [(16, 2600), (4, 4200)])
def test_many_chunks_scan_and_topk(G, pages):
    """More pages than one top-k CTA scores (1024 at G=16, 4096 at G=4):
    several chunks' candidates merged by the last CTA; many scan CTAs."""
    case = make_case(1, G, 1, 64 * pages + 3, true_rank=(4, 12), n_carriers=16, seed=8 + G)
    _run_case(case, 8, budget=64 * 40, check_dense=True)


def test_merge_of_more_candidates_than_registers_hold():
    """Three top-k chunks (G = 16: 1024 pages each) offering 400 candidates
    each: the 1200 candidates exceed the merge's register capacity (1024), so
    the last CTA merges them with the radix select in shared memory."""
    case = make_case(1, 16, 1, 64 * 3000 + 3, true_rank=(4, 12), n_carriers=16, seed=21)
    _run_case(case, 8, budget=64 * 400, check_dense=False)


def test_boundary_bin_of_many_equal_keys():
    """1500 logical pages share one physical page (the planted carrier), so
    their scores are bit-identical and larger than every other page's; with
    k = 600 the boundary bin holds 1500 keys, more than the histogram select
    ranks itself, and the radix select takes over.  Ties go to the lower
    page, so exactly logical pages 0..599 are chosen."""
    case = make_case(1, 1, 1, 64 * 2000, true_rank=(2, 8), n_carriers=1, seed=77)
    c = int(case.carriers[0, 0, 0])
    case.block_table[0, :1500] = case.block_table[0, c]
    nsum = [case.n_full_pages(0)]
    pages = sorted(set(int(x) for x in case.block_table[0, :nsum[0]]))
    basis_t, coeffs = oracle_summaries_bf16(case, 8, pages=pages)
    rt, q = make_runtime(case, 8, 64 * 600, nsum)
    _upload_summaries(rt, basis_t, coeffs)
    rt.select(q)
    torch.cuda.synchronize()
    assert rt.device_error() == 0
    ob, oc = oracle_layout_from_abi(basis_t, coeffs)
    ref = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, ob, oc,
                        case.num_kv_heads, 64 * 600)
    assert list(ref["sel"][(0, 0)]) == list(range(600))  # the oracle's own tie rule
    assert int(rt.sel_count[0, 0]) == 600
    assert rt.sel_pages[0, 0, :600].cpu().tolist() == list(range(600))


def test_tiny_workload_carrier_kept():
    case, cfg = make_config_case("tiny")
    rt, q, ref, _ = _run_case(case, cfg["rank"], cfg["budget_tokens"])
    carrier = int(case.carriers[0, 0, 0])
    assert carrier in set(rt.sel_pages[0, 0, :rt.sel_count[0, 0]].cpu().tolist())


def test_budget_covering_all_pages_equals_dense():
    case = make_case(2, 8, 2, [64 * 12 + 5, 64 * 9], seed=9)
    basis_t, coeffs = oracle_summaries_bf16(case, 8)
    rt, q = make_runtime(case, 8, budget_tokens=64 * 100)
    _upload_summaries(rt, basis_t, coeffs)
    out, lse = rt.decode_step(q)
    o1 = out.float().clone()
    l1 = lse.clone()
    dout, dlse = rt.dense_decode(q)
    torch.cuda.synchronize()
    assert (o1 - dout.float()).abs().max().item() <= 1e-2
    assert (l1 - dlse).abs().max().item() <= 1e-4


def test_zero_budget_and_no_summaries():
    case = make_case(2, 4, 2, [64 * 7 + 3, 64 * 5], seed=10)
    # budget below one page: only the tail (here every page, nothing summarised)
    basis_t, coeffs = oracle_summaries_bf16(case, 4)
    rt, q = make_runtime(case, 4, budget_tokens=63, n_summarized=[0, 0])
    _upload_summaries(rt, basis_t, coeffs)
    out, lse = rt.decode_step(q)
    do, dl = O.dense_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, 2)
    go = bf16_to_f32(torch_bf16_to_u16(out)).astype(np.float64)
    assert np.abs(go - do).max() <= OUT_ATOL
    assert rt.sel_count.sum().item() == 0
    # budget 0 with summaries: the step attends only the partial tail page
    rt2, q2 = make_runtime(case, 4, budget_tokens=0)
    _upload_summaries(rt2, basis_t, coeffs)
    out2, _ = rt2.decode_step(q2)
    gsel = {(b, h): [] for b in range(2) for h in range(2)}
    ro, _ = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                            [7, 5], gsel, 2)
    go2 = bf16_to_f32(torch_bf16_to_u16(out2)).astype(np.float64)
    assert np.abs(go2 - ro).max() <= OUT_ATOL


def test_empty_sequence_gives_zero_output():
    case = make_case(2, 4, 2, [0, 64 * 4 + 1], seed=11)
    rt, q = make_runtime(case, 8, budget_tokens=128)
    out, lse = rt.dense_decode(q)
    torch.cuda.synchronize()
    assert out[0].float().abs().max().item() == 0.0
    assert torch.isinf(lse[0]).all() and (lse[0] < 0).all()
    out, lse = rt.decode_step(q)
    torch.cuda.synchronize()
    assert out[0].float().abs().max().item() == 0.0
    assert rt.device_error() == 0


def test_exact_page_lse_matches_oracle():
    case = make_case(2, 8, 2, [64 * 20 + 11, 64 * 13], seed=12)
    rt, q = make_runtime(case, 8, 256)
    pl = rt.exact_page_lse(q).cpu().numpy()
    kf, qf = O.bf16_widen(case.k_pool), O.bf16_widen(case.q)
    G = case.group
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        for j in range(case.n_pages(b)):
            p = case.block_table[b, j]
            n = min(64, L - 64 * j)
            for hq in range(case.num_q_heads):
                want = O.exact_page_lse(qf[b, hq], kf[p, hq // G, :n])
                assert abs(pl[b, hq, j] - want) <= LSE_RTOL * max(1, abs(want)), (b, j, hq)


def test_graph_capture_replay_bit_identical():
    case = make_case(2, 8, 2, [64 * 33 + 7, 64 * 30], true_rank=(2, 10), seed=13)
    basis_t, coeffs = oracle_summaries_bf16(case, 8)
    rt, q = make_runtime(case, 8, budget_tokens=64 * 4)
    _upload_summaries(rt, basis_t, coeffs)
    out_e, lse_e = rt.decode_step(q)
    ref_o, ref_l = out_e.clone(), lse_e.clone()
    ref_sel = rt.sel_pages.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    out_g = torch.zeros_like(out_e)
    lse_g = torch.zeros_like(lse_e)
    with torch.cuda.stream(s):
        rt.decode_step(q, out_g, lse_g, stream=s)  # warm-up on the capture stream
        with torch.cuda.graph(g, stream=s):
            rt.decode_step(q, out_g, lse_g, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out_g.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, ref_o)
    assert torch.equal(lse_g, ref_l)
    assert torch.equal(rt.sel_pages, ref_sel)
    # the graph reads lengths on the device: drop the last token of sequence 0
    # (its partial tail page shrinks) and replay
    rt.seq_lens[0] -= 1
    g.replay()
    torch.cuda.synchronize()
    assert not torch.equal(out_g[0], ref_o[0])
    assert torch.equal(out_g[1], ref_o[1])
    assert rt.device_error() == 0


def test_device_error_on_bad_block_table():
    case = make_case(1, 4, 2, 64 * 10 + 5, seed=14)
    basis_t, coeffs = oracle_summaries_bf16(case, 8)
    rt, q = make_runtime(case, 8, budget_tokens=64 * 3)
    _upload_summaries(rt, basis_t, coeffs)
    good = rt.block_table.clone()
    rt.block_table[0, 2] = case.pages_total + 5   # out of range: skipped, flagged
    rt.decode_step(q)
    rt.dense_decode(q)
    err = rt.device_error()
    assert err & 0x1
    rt.block_table.copy_(good)
    out, _ = rt.decode_step(q)
    assert rt.device_error() == 0
    rt.seq_lens[0] = 64 * 11 + 1                   # longer than max_pages * P
    rt.decode_step(q)
    assert rt.device_error() & 0x4


# ---------------------------------------------------------------------------
# summary builder
# ---------------------------------------------------------------------------

def _recon_err(K, V_rows, C):
    R = C @ V_rows
    return np.linalg.norm(K - R) / np.linalg.norm(K)


@pytest.mark.parametrize("r,true_rank", [(8, (8, 8)), (4, (2, 16)), (16, (2, 16)), (2, (2, 6))])
def test_builder_reconstruction_error_matches_svd(r, true_rank):
    case = make_case(1, 4, 2, 64 * 24, true_rank=true_rank, n_carriers=2, seed=20 + r)
    device = "cuda"
    k = to_torch_bf16(case.k_pool, device)
    pages = torch.from_numpy(case.block_table[0, :24].copy()).to(device)
    from sparse_kv_page_rank_gb300 import locks as L
    pt, hkv = case.k_pool.shape[:2]
    kf = O.bf16_widen(case.k_pool)
    for dtype in (L.LOCKS_DTYPE_F32, L.LOCKS_DTYPE_BF16):
        tdt = torch.float32 if dtype == L.LOCKS_DTYPE_F32 else torch.bfloat16
        bt = torch.zeros((pt, hkv, r, 128), dtype=tdt, device=device)
        co = torch.zeros((pt, hkv, 64, r), dtype=tdt, device=device)
        cache = L.make_cache(k, k, torch.from_numpy(case.block_table).to(device),
                             torch.from_numpy(case.seq_lens).to(device))
        summ = L.make_summary(bt, co, r, dtype)
        L.locks_build_summaries(cache, summ, pages, 24)
        torch.cuda.synchronize()
        btn = bt.float().cpu().numpy().astype(np.float64)
        con = co.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(btn).all() and np.isfinite(con).all()
        for p in case.block_table[0, :24]:
            for h in range(hkv):
                K = kf[p, h]
                V, C, _, S = O.page_summary(K, r)
                e_or = _recon_err(K, V.T, C)
                e_gpu = _recon_err(K, btn[p, h], con[p, h])
                assert abs(e_gpu - e_or) <= 1e-3, (dtype, p, h, e_gpu, e_or)
                if dtype == L.LOCKS_DTYPE_F32:
                    Vg = btn[p, h]
                    nz = np.linalg.norm(Vg, axis=1) > 0
                    gram = Vg[nz] @ Vg[nz].T
                    assert np.abs(gram - np.eye(nz.sum())).max() <= 1e-3
                    # descending: row norms of C are the singular values
                    sv = np.linalg.norm(con[p, h], axis=0)
                    assert np.all(np.diff(sv[nz]) <= 1e-3 * sv[0])


def test_builder_rank_deficient_and_zero_pages():
    """A page of exact rank 2 (small integers, exact in bf16) is rebuilt to
    fp32 precision and its columns past rank 2 vanish; an all-zero page gives
    an all-zero summary (no NaN); a full-rank Gaussian page matches the SVD's
    reconstruction error."""
    rng = np.random.default_rng(0)
    from synth import bf16_bits
    from sparse_kv_page_rank_gb300 import locks as L
    pt, hkv, r = 3, 1, 8
    k = np.zeros((pt, hkv, 64, 128), dtype=np.float32)
    a, c = rng.choice([-1.0, 1.0], 64), rng.choice([-1.0, 1.0], 64)
    bvec, evec = rng.integers(-2, 3, 128).astype(np.float64), rng.integers(-2, 3, 128).astype(np.float64)
    k[0, 0] = np.outer(a, bvec) + np.outer(c, evec)
    k[1, 0] = rng.standard_normal((64, 128))
    kb = bf16_bits(k)
    dev = "cuda"
    kt = to_torch_bf16(kb, dev)
    bt = torch.full((pt, hkv, r, 128), 7.0, device=dev)
    co = torch.full((pt, hkv, 64, r), 7.0, device=dev)
    cache = L.make_cache(kt, kt, torch.zeros((1, 3), dtype=torch.int32, device=dev),
                         torch.zeros(1, dtype=torch.int32, device=dev))
    L.locks_build_summaries(cache, L.make_summary(bt, co, r, L.LOCKS_DTYPE_F32),
                            torch.tensor([0, 1, 2], dtype=torch.int32, device=dev), 3)
    torch.cuda.synchronize()
    btn, con = bt.cpu().numpy(), co.cpu().numpy()
    assert np.isfinite(btn).all() and np.isfinite(con).all()
    K0 = bf16_to_f32(kb[0, 0]).astype(np.float64)
    assert np.linalg.matrix_rank(K0) == 2
    assert _recon_err(K0, btn[0, 0].astype(np.float64), con[0, 0].astype(np.float64)) < 1e-5
    assert np.abs(con[0, 0][:, 2:]).max() <= 1e-5 * np.abs(con[0, 0][:, 0]).max()
    assert np.abs(btn[2, 0]).max() == 0 and np.abs(con[2, 0]).max() == 0
    K1 = bf16_to_f32(kb[1, 0]).astype(np.float64)
    V, C, _, _ = O.page_summary(K1, r)
    e_or = _recon_err(K1, V.T, C)
    assert abs(_recon_err(K1, btn[1, 0].astype(np.float64), con[1, 0].astype(np.float64)) - e_or) <= 1e-3


def test_builder_summaries_drive_selection():
    """End to end with GPU-built summaries: the planted carrier pages of the
    tiny workload and of a GQA-4 cache survive selection."""
    for name, ctx in (("tiny", None), ("llama128k", 64 * 512)):
        case, cfg = make_config_case(name, context=ctx)
        rt, q = make_runtime(case, cfg["rank"], cfg["budget_tokens"])
        pages = torch.from_numpy(np.concatenate([case.block_table[b, :case.n_full_pages(b)]
                                                 for b in range(case.batch)])).to("cuda")
        rt.build_summaries(pages)
        rt.select(q)
        torch.cuda.synchronize()
        sel = rt.sel_pages.cpu().numpy()
        cnt = rt.sel_count.cpu().numpy()
        kept, total = 0, 0
        for b in range(case.batch):
            for h in range(case.num_kv_heads):
                chosen = set(sel[b, h, :cnt[b, h]].tolist())
                for cpg in case.carriers[b, h]:
                    if cpg >= 0:
                        total += 1
                        kept += int(cpg) in chosen
        assert kept / total >= 0.9, (name, kept, total)


def test_decode_step_with_host_query_and_output():
    """q and out in page-locked host memory (read and written in place by the
    kernels) give bit-identical results to device buffers."""
    case = make_case(2, 8, 2, [64 * 30 + 9, 64 * 25 + 63], true_rank=(4, 10), n_carriers=2, seed=71)
    basis_t, coeffs = oracle_summaries_bf16(case, 8)
    rt, q = make_runtime(case, 8, 640)
    _upload_summaries(rt, basis_t, coeffs)
    out_dev, lse_dev = rt.decode_step(q)
    out_dev, lse_dev = out_dev.clone(), lse_dev.clone()
    q_host = q.cpu().pin_memory()
    out_host = torch.zeros(out_dev.shape, dtype=torch.bfloat16).pin_memory()
    lse_host = torch.zeros(lse_dev.shape, dtype=torch.float32).pin_memory()
    rt.decode_step(q_host, out=out_host, lse=lse_host)
    torch.cuda.synchronize()
    assert rt.device_error() == 0
    assert torch.equal(out_host.view(torch.int16), out_dev.cpu().view(torch.int16))
    assert torch.equal(lse_host, lse_dev.cpu())


@pytest.mark.parametrize("P", [64, 16])
def test_packed_layout_holds_the_two_array_values(P):
    """LOCKS_DTYPE_BF16_PACKED: the builder writes bit-for-bit the values of
    the two-array bf16 layout, basis rows then coefficients in one block per
    page-head, and the scan gives bit-identical page LSEs from either."""
    from sparse_kv_page_rank_gb300 import locks as L
    r = 8
    case = make_case(2, 8, 2, [P * 30 + 3, P * 22], true_rank=(2, 10), n_carriers=2, seed=61, page_size=P)
    dev = "cuda"
    split, q = make_runtime(case, r, P * 6, split=True)
    packed, _ = make_runtime(case, r, P * 6)
    assert packed.summary.dtype == L.LOCKS_DTYPE_BF16_PACKED and split.summary.dtype == L.LOCKS_DTYPE_BF16
    pages = torch.from_numpy(np.concatenate([case.block_table[b, :case.n_full_pages(b)]
                                             for b in range(case.batch)])).to(dev)
    split.build_summaries(pages)
    packed.build_summaries(pages)
    torch.cuda.synchronize()
    blocks = packed.blocks.view(torch.int16)
    pt, hkv = blocks.shape[:2]
    assert torch.equal(blocks[:, :, :r * 128], split.basis_t.view(torch.int16).reshape(pt, hkv, -1))
    assert torch.equal(blocks[:, :, r * 128:], split.coeffs.view(torch.int16).reshape(pt, hkv, -1))
    pls = []
    for rt in (split, packed):
        pl = torch.full((case.batch, case.num_q_heads, case.max_pages), float("nan"), device=dev)
        rt.select(q, pl)
        torch.cuda.synchronize()
        assert rt.device_error() == 0
        pls.append(pl)
    assert torch.equal(torch.nan_to_num(pls[0], nan=7.0), torch.nan_to_num(pls[1], nan=7.0))
    assert torch.equal(split.sel_pages, packed.sel_pages) and torch.equal(split.sel_count, packed.sel_count)
