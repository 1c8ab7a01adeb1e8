"""locks_decode_step_static, the decode step for callers that cannot allocate
device memory (hosts that hand every byte of the GPU to their own pool, or
thin C callers with nowhere to keep a workspace), checked against the
ordinary locks_decode_step with a caller-owned workspace.

The static entry point runs in one array the library keeps on each GPU, so
its calls share that memory; the test makes two calls in a row with
different queries, to show that the second does not see the first's
leftovers.  Tolerances are those of the other GPU tests: outputs within
1e-2 absolute, lse within 1e-3 relative, selections identical (both paths
run the same kernels on the same inputs).

This file is named so that pytest collects it last."""

import numpy as np
import pytest

from synth import make_case
from tests.helpers import make_runtime

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

OUT_ATOL = 1e-2
LSE_RTOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_page_rank_gb300.build_lib import build
    build()


def _bf16(arr):
    return torch.from_numpy(arr.astype(np.float32)).to(torch.bfloat16).cuda()


def test_static_step_matches_decode_step_on_two_calls_in_a_row():
    from sparse_kv_page_rank_gb300 import locks as L

    case = make_case(2, 8, 2, [64 * 30 + 9, 64 * 25 + 63], true_rank=(4, 10), n_carriers=2, seed=31)
    rt, q1 = make_runtime(case, 8, 640)
    pages = np.concatenate([case.block_table[b, :case.n_full_pages(b)] for b in range(case.batch)])
    rt.build_summaries(torch.from_numpy(pages.astype(np.int32)).cuda())
    rng = np.random.Generator(np.random.PCG64(32))
    q2 = _bf16(rng.standard_normal(tuple(q1.shape)))

    # reference: the ordinary entry point with the runtime's own workspace
    refs = []
    for q in (q1, q2):
        out, lse = rt.decode_step(q)
        refs.append((out.clone(), lse.clone(), rt.sel_pages.clone(), rt.sel_count.clone()))
    torch.cuda.synchronize()
    assert rt.device_error() == 0

    # the static entry point, twice in a row on one stream
    got = []
    for q in (q1, q2):
        out = torch.full_like(refs[0][0], float("nan"))
        lse = torch.full_like(refs[0][1], float("nan"))
        sel = torch.full_like(refs[0][2], -7)
        cnt = torch.full_like(refs[0][3], -7)
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        L.locks_decode_step_static(rt.cache, rt.summary, rt.params, q, out, lse, sel, cnt, err)
        got.append((out, lse, sel, cnt, err))
    torch.cuda.synchronize()

    for (r_out, r_lse, r_sel, r_cnt), (out, lse, sel, cnt, err) in zip(refs, got):
        assert int(err.item()) == 0
        assert torch.equal(cnt, r_cnt)
        for b in range(case.batch):
            for h in range(case.num_kv_heads):
                n = int(r_cnt[b, h])
                assert torch.equal(sel[b, h, :n], r_sel[b, h, :n])
        assert torch.isfinite(out.float()).all()
        assert float((out.float() - r_out.float()).abs().max()) <= OUT_ATOL
        assert bool(((lse - r_lse).abs() <= LSE_RTOL * r_lse.abs().clamp(min=1.0)).all())


def test_static_step_rejects_shapes_beyond_its_workspace():
    from sparse_kv_page_rank_gb300 import locks as L

    # a valid one-page cache whose block table is very wide: the per-page
    # scores alone (8 heads x 65536 pages x 4 query heads x 4 B) fill 8 MiB
    hkv, G, r, max_pages = 8, 4, 8, 65536
    k = torch.zeros((1, hkv, 64, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    bt = torch.zeros((1, max_pages), dtype=torch.int32, device="cuda")
    sl = torch.tensor([64], dtype=torch.int32, device="cuda")
    ns = torch.tensor([1], dtype=torch.int32, device="cuda")
    basis = torch.zeros((1, hkv, r, 128), dtype=torch.bfloat16, device="cuda")
    coef = torch.zeros((1, hkv, 64, r), dtype=torch.bfloat16, device="cuda")
    cache = L.make_cache(k, v, bt, sl, ns)
    summ = L.make_summary(basis, coef, r)
    params = L.make_params(hkv * G, 2048)
    assert L.locks_workspace_size(cache, summ, params) > L.LOCKS_STATIC_WS_BYTES
    q = torch.zeros((1, hkv * G, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(L.LocksError) as e:
        L.locks_decode_step_static(cache, summ, params, q, out, None)
    assert e.value.status == L.LOCKS_ERR_WORKSPACE


def test_static_step_allocates_nothing_and_replays_in_a_graph():
    """Device free memory (cudaMemGetInfo) is unchanged over several static
    calls after the first, and a call captured in a CUDA graph (after an
    uncaptured one on the device) gives the uncaptured call's results."""
    from sparse_kv_page_rank_gb300 import locks as L

    case = make_case(2, 8, 2, [64 * 40 + 3, 64 * 33], true_rank=(4, 10), n_carriers=2, seed=33)
    rt, q = make_runtime(case, 8, 512)
    pages = np.concatenate([case.block_table[b, :case.n_full_pages(b)] for b in range(case.batch)])
    rt.build_summaries(torch.from_numpy(pages.astype(np.int32)).cuda())
    outs = [(torch.empty_like(rt.out), torch.empty_like(rt.lse), torch.empty_like(rt.sel_pages),
             torch.empty_like(rt.sel_count), torch.empty((1,), dtype=torch.int32, device="cuda")) for _ in range(2)]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def call(o):
        L.locks_decode_step_static(rt.cache, rt.summary, rt.params, q, o[0], o[1], o[2], o[3], o[4], stream=stream)

    call(outs[0])
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(6):
        call(outs[0])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(outs[0][4].item()) == 0

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            call(outs[1])
        g.replay()
    torch.cuda.synchronize()
    assert int(outs[1][4].item()) == 0
    for a, b in zip(outs[0][:4], outs[1][:4]):
        assert torch.equal(a, b)
