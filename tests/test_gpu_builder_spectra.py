"""The summary builder on spectra that slow its subspace iteration (GPU).

The builder takes the top-r eigenvectors of the page's Gram matrix K K^T by
subspace iteration on l = r + 8 vectors (8 steps) and a Jacobi
Rayleigh-Ritz step.  Its convergence for the r-th vector goes as
(sigma_{l+1} / sigma_r)^16, so pages whose singular values barely fall past
the cut converge least.  Pages here are built with exact singular values
(K = U diag(sigma) W^T, random orthonormal U and W, then rounded to bf16):

  * near tie at the cut: sigma_{r+1} = 0.999 sigma_r;
  * flat beyond the cut: sigma_{r+1} .. sigma_{r+16} all 0.99 sigma_r, so
    even the iteration's extra vectors sit inside the flat stretch;
  * slow decay: sigma_i = 0.97^i, no gap anywhere;
  * a dominant direction: sigma_1 = 300 sigma_2, the rest decaying slowly (the
    fp32 Gram matrix holds the rest within 1/300^2 of its largest entry).

On all of them the builder's reconstruction error ||K - C V^T||_F / ||K||_F
must be within 1e-3 of the oracle's truncated SVD of the same bf16 keys (the
builder tolerance of test_gpu_parity); with fp32 output the basis must also
be orthonormal within 1e-3.  A basis that mixes nearly tied directions is as
good a rank-r summary as the SVD's (the residual differs by a second-order
amount), which is what the error comparison measures.
"""

import numpy as np
import pytest

import oracle as O
from synth import bf16_bits, bf16_to_f32
from tests.helpers import to_torch_bf16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

P, D = 64, 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_page_rank_gb300.build_lib import build
    build()


def _spectrum(kind, r):
    i = np.arange(P, dtype=np.float64)
    if kind == "near_tie":
        s = 0.9 ** i
        s[r:] = s[r - 1] * 0.999 * 0.9 ** (i[r:] - r)
    elif kind == "flat_beyond":
        s = 0.9 ** i
        s[r:r + 16] = s[r - 1] * 0.99
        s[r + 16:] = s[r - 1] * 0.99 * 0.8 ** (i[r + 16:] - r - 15)
    elif kind == "slow_decay":
        s = 0.97 ** i
    elif kind == "dominant":
        s = 0.97 ** i
        s[0] = 300.0 * s[1]
    else:
        raise ValueError(kind)
    return 4.0 * s / s[r - 1]


def _pages(kind, r, n, seed):
    rng = np.random.default_rng(seed)
    k = np.zeros((n, 1, P, D), dtype=np.float32)
    for p in range(n):
        u, _ = np.linalg.qr(rng.standard_normal((P, P)))
        w, _ = np.linalg.qr(rng.standard_normal((D, P)))
        k[p, 0] = (u * _spectrum(kind, r)) @ w.T
    return bf16_bits(k)


def _recon_err(K, V_rows, C):
    return np.linalg.norm(K - C @ V_rows) / np.linalg.norm(K)


@pytest.mark.parametrize("kind", ["near_tie", "flat_beyond", "slow_decay", "dominant"])
@pytest.mark.parametrize("r", [2, 4, 8, 16])
def test_builder_matches_svd_on_slow_spectra(kind, r):
    from sparse_kv_page_rank_gb300 import locks as L
    n = 6
    kb = _pages(kind, r, n, seed=100 + r)
    dev = "cuda"
    kt = to_torch_bf16(kb, dev)
    ids = torch.arange(n, dtype=torch.int32, device=dev)
    cache = L.make_cache(kt, kt, torch.zeros((1, n), dtype=torch.int32, device=dev),
                         torch.zeros(1, dtype=torch.int32, device=dev))
    for dtype in (L.LOCKS_DTYPE_F32, L.LOCKS_DTYPE_BF16):
        tdt = torch.float32 if dtype == L.LOCKS_DTYPE_F32 else torch.bfloat16
        bt = torch.zeros((n, 1, r, D), dtype=tdt, device=dev)
        co = torch.zeros((n, 1, P, r), dtype=tdt, device=dev)
        L.locks_build_summaries(cache, L.make_summary(bt, co, r, dtype), ids, n)
        torch.cuda.synchronize()
        btn = bt.float().cpu().numpy().astype(np.float64)
        con = co.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(btn).all() and np.isfinite(con).all()
        for p in range(n):
            K = bf16_to_f32(kb[p, 0]).astype(np.float64)
            V, C, _, _ = O.page_summary(K, r)
            e_or = _recon_err(K, V.T, C)
            e_gpu = _recon_err(K, btn[p, 0], con[p, 0])
            assert abs(e_gpu - e_or) <= 1e-3, (kind, r, dtype, p, e_gpu, e_or)
            if dtype == L.LOCKS_DTYPE_F32:
                Vg = btn[p, 0]
                assert np.abs(Vg @ Vg.T - np.eye(r)).max() <= 1e-3, (kind, r, p)
