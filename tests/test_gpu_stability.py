"""Repeatability of the decode step under back-to-back launches (GPU).

The 128K workload (1 sequence, 32 query / 8 KV heads, r = 8, budget 2048) is
stepped many times in a row on one stream, the kernels overlapping through
programmatic dependent launch as in the bench.  Every step has the same
inputs, so every step must give bit-identical outputs and selections, and no
bounded wait may run out (the device error word stays 0).  This guards the
producer / consumer ring protocols of the scan and attention kernels against
ordering races that only show under load.
"""

import numpy as np
import pytest

from synth import make_config_case
from tests.helpers import make_runtime

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

STEPS = 600


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_page_rank_gb300.build_lib import build
    build()


def test_back_to_back_steps_bit_identical():
    from sparse_kv_page_rank_gb300 import locks as L

    case, cfg = make_config_case("llama128k")
    rt, q = make_runtime(case, cfg["rank"], cfg["budget_tokens"])
    pages = np.concatenate([case.block_table[b, :case.n_full_pages(b)] for b in range(case.batch)])
    rt.build_summaries(torch.from_numpy(pages.astype(np.int32)).cuda())
    torch.cuda.synchronize()
    assert rt.device_error() == 0
    B, Hq, d = q.shape
    outs = torch.empty((STEPS, B, Hq, d), dtype=torch.bfloat16, device="cuda")
    lses = torch.empty((STEPS, B, Hq), dtype=torch.float32, device="cuda")
    sels = torch.empty((STEPS,) + tuple(rt.sel_pages.shape), dtype=torch.int32, device="cuda")
    cnts = torch.empty((STEPS,) + tuple(rt.sel_count.shape), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    sels.fill_(-1)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(STEPS):
            L.locks_decode_step(rt.cache, rt.summary, rt.params, q, outs[i], lses[i], sels[i], cnts[i], rt.ws,
                                rt.ws_bytes, stream)
    stream.synchronize()
    assert rt.device_error() == 0
    ref = outs[0].view(torch.int16)
    for i in range(1, STEPS):
        assert torch.equal(outs[i].view(torch.int16), ref), i
        assert torch.equal(lses[i], lses[0]), i
        assert torch.equal(cnts[i], cnts[0]), i
        assert torch.equal(sels[i], sels[0]), i
