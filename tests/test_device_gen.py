"""The device-side cache generator, run on the CPU: the layout and the
page-local structure it promises (ranks, carrier direction, NaN tail,
block table a permutation, seeded)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth.device_gen import make_device_cache  # noqa: E402


def _case(seed=5):
    return make_device_cache(2, 8, 2, 64 * 40 + 10, true_rank=(3, 6), n_carriers=4, seed=seed, device="cpu",
                             chunk_pages=16)


def test_layout_and_seeding():
    c = _case()
    k, v, bt = c["k_pool"], c["v_pool"], c["block_table"]
    assert k.shape == v.shape == (82, 2, 64, 128) and k.dtype == torch.bfloat16
    assert bt.dtype == torch.int32 and sorted(bt.reshape(-1).tolist()) == list(range(82))
    assert c["seq_lens"].tolist() == [2570, 2570] and c["n_full"].tolist() == [40, 40]
    last = bt[:, -1].long()
    assert torch.isnan(k[last, :, 10:].float()).all() and not torch.isnan(k[last, :, :10].float()).any()
    assert torch.isnan(v[last, :, 10:].float()).all()
    full = torch.ones(82, dtype=torch.bool)
    full[last] = False
    assert not torch.isnan(k[full].float()).any()
    d = _case()
    assert torch.equal(d["k_pool"].view(torch.int16), k.view(torch.int16))
    assert not torch.equal(_case(seed=6)["k_pool"].view(torch.int16), k.view(torch.int16))


def test_page_local_low_rank_and_carriers():
    c = _case()
    k, bt, q = c["k_pool"].double(), c["block_table"], c["q"].double()
    qh = q / q.norm(dim=-1, keepdim=True)
    car = c["carriers"]
    G = 4
    for b in range(2):
        for h in range(2):
            cp = car[b, h].tolist()
            assert cp == sorted(set(cp)) and all(0 <= p < 40 for p in cp)
            for j in range(40):
                K = k[bt[b, j].long(), h]
                s = torch.linalg.svdvals(K).numpy()
                # true rank 2..6 (a carrier's basis is one lower, plus the q_hat
                # shift): a clear gap at the rank, noise (0.05 x sqrt(64)) below
                gaps = s[:7] / s[1:8]
                assert gaps.max() > 5 and s[7] < 1.5, (b, h, j, s[:8])
                if j in cp:
                    head = h * G + cp.index(j) % G
                    assert abs(float((K @ qh[b, head]).mean()) - 3.0) < 0.3, (b, h, j)
