"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test names the passage it follows and the independent fact it checks:
closed forms, textbook routines (LAPACK SVD vs a pure-Python Jacobi), the
Eckart-Young optimality that Theorem 1 relies on, brute-force sums, and the
limits the pages fix (full rank => exact LSE; budget covering every page =>
dense attention).  A plausible slip in the oracle (dropped 1/sqrt(d), missing
GSA normalisation, wrong tie order, transposed summary) fails at least one.
"""

import math
import random

import numpy as np
import pytest

import oracle as O
from synth import make_case, bf16_to_f32


def _orth(rng, d, t):
    q, _ = np.linalg.qr(rng.standard_normal((d, t)))
    return q


# --- log-sum-exp ------------------------------------------------------------

def test_lse_brute_force_tiny_pages():
    """Page mass by log-sum-exp (LOCKS abstract; explainer §2 'Reconstructie en
    Selectie'): on 4-token pages the oracle's LSE equals ln(fsum(exp)) computed
    term by term, and a shifted copy does not overflow."""
    rng = random.Random(5)
    for _ in range(200):
        xs = [rng.uniform(-30, 30) for _ in range(4)]
        want = math.log(math.fsum(math.exp(x) for x in xs))
        assert abs(O.logsumexp(np.array(xs)) - want) < 1e-12 * max(1, abs(want))
    big = np.array([1000.0, 1000.0, 1000.0, 1000.0])
    assert abs(O.logsumexp(big) - (1000.0 + math.log(4))) < 1e-12
    assert O.logsumexp(np.zeros(0)) == -np.inf


def test_scale_closed_form_ln10():
    """1/sqrt(d) scaling of the equation for s_hat_j(q) (explainer §2): with
    q = sqrt(d) e_1 and keys ln(i) e_1, i = 1..4, the logits are ln 1..ln 4, so
    both the exact and the reconstructed page mass are ln 10."""
    d, P = 128, 4
    q = np.zeros(d)
    q[0] = math.sqrt(d)
    K = np.zeros((P, d))
    K[:, 0] = [math.log(i) for i in range(1, P + 1)]
    assert abs(O.exact_page_lse(q, K) - math.log(10)) < 1e-13
    V, C, mu, S = O.page_summary(K, 1)
    assert abs(O.reconstructed_page_lse(q, V, C) - math.log(10)) < 1e-13
    # rank 0 of signal: a zero basis gives ln P (all logits 0)
    assert abs(O.reconstructed_page_lse(q, np.zeros((d, 1)), np.zeros((P, 1))) - math.log(P)) < 1e-15


# --- summary (truncated SVD / eigendecomposition) ----------------------------

def test_summary_exact_low_rank_and_truncation():
    """Rank-r summary (explainer §2 'Kernmechanisme'): a page of exact rank 2
    with known singular values (5, 2) is reproduced exactly at r = 2; at r = 1
    the residual is the dropped singular value (2)."""
    rng = np.random.default_rng(0)
    P, d = 16, 32
    U = _orth(rng, P, 2)
    W = _orth(rng, d, 2)
    K = 5.0 * np.outer(U[:, 0], W[:, 0]) + 2.0 * np.outer(U[:, 1], W[:, 1])
    V, C, mu, S = O.page_summary(K, 2)
    assert np.allclose(S[:2], [5.0, 2.0], atol=1e-12)
    assert np.allclose(C @ V.T, K, atol=1e-12)
    assert np.allclose(V.T @ V, np.eye(2), atol=1e-12)
    V1, C1, _, _ = O.page_summary(K, 1)
    assert abs(np.linalg.norm(K - C1 @ V1.T) - 2.0) < 1e-12
    # columns past the rank are zero (rank-deficit reading)
    V4, C4, _, _ = O.page_summary(K, 4)
    assert np.all(V4[:, 2:] == 0) and np.all(C4[:, 2:] == 0)


def test_summary_matches_pure_python_jacobi():
    """The eigendecomposition of the page Gram matrix (explainer §2) computed by
    a textbook cyclic Jacobi in pure Python gives the same sigma^2 and the same
    rank-r reconstruction as the oracle's LAPACK SVD (signs are irrelevant)."""
    rng = np.random.default_rng(1)
    P, d, r = 8, 16, 3
    K = rng.standard_normal((P, d)) @ np.diag(np.linspace(3, 0.2, d))
    V, C, _, S = O.page_summary(K, r)
    w, U = O.jacobi_eigh(K @ K.T)
    assert np.allclose(w, S ** 2, rtol=1e-10, atol=1e-10)
    sig = np.sqrt(w[:r])
    Cj = U[:, :r] * sig
    Vj = K.T @ U[:, :r] / sig
    assert np.allclose(Cj @ Vj.T, C @ V.T, atol=1e-10)


def test_eckart_young_residual_optimal():
    """Theorem 1's premise (explainer §3): the page-local basis is
    residual-optimal among orthogonal rank-r reconstructions.  Residual^2 equals
    the spectral tail sum_{i>r} sigma_i^2 and no random orthonormal basis does
    better."""
    rng = np.random.default_rng(2)
    P, d, r = 64, 128, 8
    K = rng.standard_normal((P, 12)) @ rng.standard_normal((12, d)) + 0.05 * rng.standard_normal((P, d))
    V, C, _, S = O.page_summary(K, r)
    res2 = np.linalg.norm(K - C @ V.T) ** 2
    assert abs(res2 - np.sum(S[r:] ** 2)) < 1e-9 * np.sum(S ** 2)
    for _ in range(50):
        Q = _orth(rng, d, r)
        assert np.linalg.norm(K - (K @ Q) @ Q.T) ** 2 >= res2 - 1e-9


def test_summary_transpose_slip_detected():
    """V is d x r and C is P x r: the logit of token i uses (V^T q).c_i.  A
    page whose rows are identical shows the roles are not swapped: every logit
    equals q.k/sqrt(d)."""
    rng = np.random.default_rng(3)
    P, d = 64, 128
    k = rng.standard_normal(d)
    K = np.tile(k, (P, 1))
    q = rng.standard_normal(d)
    V, C, _, _ = O.page_summary(K, 2)
    logits = O.reconstructed_logits(q, V, C)
    assert np.allclose(logits, q @ k / math.sqrt(d), atol=1e-12)


def test_centered_summary_identical_keys_closed_form():
    """Centred variant (explainer §2: eigendecomposition of key deviations plus
    the q.mu_j term): a page of identical keys has zero deviation, so at any
    rank s_hat = ln P + q.mu/sqrt(d) exactly."""
    rng = np.random.default_rng(4)
    P, d = 64, 128
    k = rng.standard_normal(d)
    K = np.tile(k, (P, 1))
    q = rng.standard_normal(d)
    V, C, mu, _ = O.page_summary(K, 4, centered=True)
    assert np.allclose(C, 0) and np.allclose(mu, k)
    assert abs(O.reconstructed_page_lse(q, V, C, mu) - (math.log(P) + q @ k / math.sqrt(d))) < 1e-12


@pytest.mark.parametrize("P", [64, 16])
@pytest.mark.parametrize("centered", [False, True])
def test_full_rank_reconstruction_equals_exact_lse(centered, P):
    """At r = min(P, d) the reconstructed page LSE equals the exact LSE that
    reads every key (equation for s_hat_j(q), explainer §2), to 1e-12."""
    rng = np.random.default_rng(5)
    d = 128
    K = rng.standard_normal((P, d)) * 2
    for _ in range(5):
        q = rng.standard_normal(d) * 3
        V, C, mu, _ = O.page_summary(K, min(P, d), centered)
        a = O.reconstructed_page_lse(q, V, C, mu if centered else None)
        b = O.exact_page_lse(q, K)
        assert abs(a - b) < 1e-12 * max(1.0, abs(b))


def test_error_nonincreasing_in_rank():
    """Theorem 1 (explainer §3) bounds the error by the spectral tail energy of
    the page-local reconstruction; its constants are not printed, so only the
    monotone consequence is pinned: the mean |s_hat - s*| over pages does not
    grow with r and vanishes at full rank."""
    case = make_case(1, 1, 1, 64 * 24, true_rank=(2, 16), n_carriers=0, seed=11)
    kf = O.bf16_widen(case.k_pool)
    q = O.bf16_widen(case.q)[0, 0]
    errs = []
    for r in (1, 2, 4, 8, 16, 64):
        e = []
        for j in range(24):
            K = kf[case.block_table[0, j], 0]
            V, C, _, _ = O.page_summary(K, r)
            e.append(abs(O.reconstructed_page_lse(q, V, C) - O.exact_page_lse(q, K)))
        errs.append(np.mean(e))
    assert all(errs[i + 1] <= errs[i] + 1e-12 for i in range(len(errs) - 1)), errs
    assert errs[-1] < 1e-12


# --- GSA and selection -------------------------------------------------------

def test_gsa_closed_form():
    """GSA (explainer §2 'Group-Shared Selection'): head 0 masses (1, 3), head 1
    masses (2, 2) give shares (1/4, 3/4) and (1/2, 1/2); their means are 3/8
    and 5/8."""
    shat = np.log(np.array([[1.0, 3.0], [2.0, 2.0]]))
    sig = O.gsa_scores(shat)
    assert np.allclose(sig, np.log([3 / 8, 5 / 8]), atol=1e-14)


def test_gsa_normalisation_changes_ranking():
    """Averaging shares (not raw masses): head 0 carries a huge total mass on
    pages it spreads evenly; head 1 concentrates on page 2.  Raw-mass averaging
    would rank page 0 first; share averaging ranks page 2 first."""
    shat = np.log(np.array([[1000.0, 900.0, 900.0], [1.0, 1.0, 50.0]]))
    sig = O.gsa_scores(shat)
    assert int(np.argmax(sig)) == 2
    raw = np.log(np.exp(shat).mean(axis=0))
    assert int(np.argmax(raw)) == 0


def test_gsa_single_head_is_lse_ranking():
    """G = 1: sigma_j = s_hat_j - Z, so selection follows s_hat exactly."""
    rng = np.random.default_rng(6)
    s = rng.standard_normal(50) * 4
    sig = O.gsa_scores(s[None, :])
    assert np.allclose(sig, s - O.logsumexp(s), atol=1e-12)
    assert list(O.select_top_pages(sig, 7)) == sorted(np.argsort(-s, kind="stable")[:7])


def test_gsa_head_permutation_invariance():
    rng = np.random.default_rng(7)
    shat = rng.standard_normal((4, 40)) * 3
    a = O.select_top_pages(O.gsa_scores(shat), 9)
    b = O.select_top_pages(O.gsa_scores(shat[[2, 0, 3, 1]]), 9)
    assert list(a) == list(b)


def test_topk_ties_go_to_lower_index_and_sorted():
    sig = np.array([0.5, 2.0, 2.0, 1.0, 2.0, -1.0, 1.0])
    assert list(O.select_top_pages(sig, 2)) == [1, 2]
    assert list(O.select_top_pages(sig, 4)) == [1, 2, 3, 4]
    assert list(O.select_top_pages(sig, 5)) == [1, 2, 3, 4, 6]
    assert list(O.select_top_pages(sig, 100)) == list(range(7))
    assert list(O.select_top_pages(sig, 0)) == []


# --- attention -----------------------------------------------------------------

def test_attention_closed_form_weights():
    """Two tokens whose scaled logits are ln 3 and 0 get weights 3/4 and 1/4."""
    d = 128
    q = np.zeros((1, d))
    q[0, 0] = math.sqrt(d) * math.log(3.0)
    K = np.zeros((2, d))
    K[0, 0] = 1.0
    V = np.zeros((2, d))
    V[0, :] = 4.0
    V[1, :] = -8.0
    o, lse = O.attention(q, K, V)
    assert np.allclose(o, 0.75 * 4.0 + 0.25 * -8.0, atol=1e-13)
    assert abs(lse[0] - math.log(4.0)) < 1e-13


def test_attention_uniform_keys_mean_value():
    rng = np.random.default_rng(8)
    k = rng.standard_normal(128)
    K = np.tile(k, (10, 1))
    V = rng.standard_normal((10, 128))
    o, _ = O.attention(rng.standard_normal((3, 128)), K, V)
    assert np.allclose(o, V.mean(axis=0)[None, :], atol=1e-13)


def _small_case(seed=9, G=2, Hkv=2, L=64 * 21 + 17, B=2, P=64):
    return make_case(B, G * Hkv, Hkv, [L, L - 64 * 3 - 5][:B], true_rank=(2, 8), n_carriers=2, seed=seed,
                     page_size=P)


def _oracle_summaries(case, r):
    kf = O.bf16_widen(case.k_pool)
    basis = np.zeros((case.pages_total, case.num_kv_heads, 128, r))
    coeffs = np.zeros((case.pages_total, case.num_kv_heads, case.page_size, r))
    for b in range(case.batch):
        for j in range(case.n_full_pages(b)):
            p = case.block_table[b, j]
            for h in range(case.num_kv_heads):
                V, C, _, _ = O.page_summary(kf[p, h], r)
                basis[p, h], coeffs[p, h] = V, C
    return basis, coeffs


@pytest.mark.parametrize("P", [64, 16])
def test_budget_covering_all_pages_equals_dense(P):
    """Selecting every page reads the whole cache: the output is dense attention."""
    case = _small_case(P=P)
    basis, coeffs = _oracle_summaries(case, 4)
    nsum = np.array([case.n_full_pages(b) for b in range(case.batch)])
    r = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum,
                      basis, coeffs, case.num_kv_heads, budget_tokens=10 ** 6, page_size=P)
    od, ld = O.dense_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                            case.num_kv_heads, page_size=P)
    assert np.allclose(r["out"], od, atol=1e-12)
    assert np.allclose(r["lse"], ld, atol=1e-12)
    assert np.isfinite(r["out"]).all()  # NaN-poisoned slots past seq_len never read


@pytest.mark.parametrize("P", [64, 16])
def test_sparse_equals_dense_over_chosen_tokens(P):
    """Attention over selected pages + tail equals attention over exactly those
    tokens gathered by hand; the open tail is always included."""
    case = _small_case(seed=10, P=P)
    basis, coeffs = _oracle_summaries(case, 8)
    nsum = np.array([case.n_full_pages(b) - 1 for b in range(case.batch)])  # last full page unsummarised
    r = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum,
                      basis, coeffs, case.num_kv_heads, budget_tokens=P * 5, page_size=P)
    kf, vf, qf = O.bf16_widen(case.k_pool), O.bf16_widen(case.v_pool), O.bf16_widen(case.q)
    G = case.group
    for (b, h), pages in r["sel"].items():
        L = int(case.seq_lens[b])
        assert len(pages) == 5 and list(pages) == sorted(pages)
        toks_k, toks_v = [], []
        allp = list(pages) + list(range(int(nsum[b]), case.n_pages(b)))
        for j in allp:
            p = case.block_table[b, j]
            n = min(P, L - P * j)
            toks_k.append(kf[p, h, :n])
            toks_v.append(vf[p, h, :n])
        o, l = O.attention(qf[b, h * G:(h + 1) * G], np.concatenate(toks_k), np.concatenate(toks_v))
        assert np.allclose(r["out"][b, h * G:(h + 1) * G], o, atol=1e-12)


def test_exact_selection_maximises_mass_recall_g1():
    """With G = 1 the exact LSE-oracle selection (read every key) has the
    largest attention-mass recall of any k-page set; recall of all pages is 1."""
    case = make_case(1, 1, 1, 64 * 30, true_rank=(2, 8), n_carriers=1, seed=12)
    nsum = np.array([30])
    r = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum,
                      None, None, 1, budget_tokens=64 * 6, exact_selection=True)
    s_star = r["shat"][(0, 0)]
    best = O.mass_recall(s_star, r["sel"][(0, 0)])
    rng = np.random.default_rng(0)
    for _ in range(200):
        other = rng.choice(30, 6, replace=False)
        assert O.mass_recall(s_star, other) <= best + 1e-12
    assert abs(O.mass_recall(s_star, range(30)) - 1.0) < 1e-12


# --- Proposition 1: a shared sketch is blind to page-specific directions ------

def test_proposition1_shared_sketch_misses_carrier_page_local_keeps_it():
    """Propositie 1 (explainer §3; LOCKS abstract): a fixed shared rank-rho
    projection is blind to within-page directions in its orthogonal complement.
    On the tiny workload, a shared sketch whose span excludes the carrier
    direction estimates the carrier page like any other page, while the
    page-local rank-8 summary ranks it first.  rho = r (1 + d/P) = 24 gives both
    the same summary bytes."""
    case = make_case(1, 1, 1, 4096, true_rank=(8, 8), n_carriers=1, seed=0)
    kf = O.bf16_widen(case.k_pool)
    q = O.bf16_widen(case.q)[0, 0]
    carrier = int(case.carriers[0, 0, 0])
    n = 64
    qhat = q / np.linalg.norm(q)
    rng = np.random.default_rng(1)
    rho = 8 * (1 + 128 // 64)
    draw = rng.standard_normal((128, rho))
    draw -= np.outer(qhat, qhat @ draw)          # span(S_sh) orthogonal to q_hat
    S_sh, _ = np.linalg.qr(draw)
    local, shared = np.zeros(n), np.zeros(n)
    for j in range(n):
        K = kf[case.block_table[0, j], 0]
        V, C, _, _ = O.page_summary(K, 8)
        local[j] = O.reconstructed_page_lse(q, V, C)
        shared[j] = O.shared_sketch_page_lse(q, S_sh, K)
    assert int(np.argmax(local)) == carrier
    others = np.delete(shared, carrier)
    # the carrier's shared-sketch estimate sits inside the spread of the others
    assert others.min() - 1e-9 <= shared[carrier] <= others.max() + 1e-9
    assert carrier not in set(O.select_top_pages(shared, 8))
    assert carrier in set(O.select_top_pages(local, 8))


def test_generator_poison_never_read():
    """Slots past seq_len are NaN in the generator; the oracle's dense output is
    finite, so it cuts every page at the sequence length."""
    case = make_case(2, 4, 2, [64 * 3 + 5, 64 * 2], seed=3)
    assert np.isnan(bf16_to_f32(case.k_pool)).any()
    od, _ = O.dense_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, 2)
    assert np.isfinite(od).all()


# --- quantised summary ------------------------------------------------------

def test_quantize_roundtrip_within_half_step():
    """Quantised storage (explainer §2 'Kernmechanisme', Kwantisatie: int4 basis, int8
    coefficients and centroid), symmetric per-vector scales: every value is
    recovered to within half a quantisation step, the largest magnitude maps
    to +-qmax, and every code lies in [-qmax, qmax]."""
    rng = np.random.default_rng(11)
    for qmax in (O.INT4_MAX, O.INT8_MAX):
        for n in (8, 64, 128):
            x = rng.standard_normal(n) * rng.uniform(0.01, 20.0)
            q, s = O.quantize_symmetric(x, qmax)
            assert s > 0 and np.all(np.abs(q) <= qmax)
            assert np.all(np.abs(q * s - x) <= s / 2 * (1 + 1e-9))
            i = int(np.argmax(np.abs(x)))
            assert abs(q[i]) == qmax and np.sign(q[i]) == np.sign(x[i])


def test_quantize_exact_on_its_grid():
    """Values already on a scale's grid (integers times a float32 scale, one of
    them at +-qmax) come back unchanged, with that scale."""
    rng = np.random.default_rng(12)
    for qmax in (O.INT4_MAX, O.INT8_MAX):
        ints = rng.integers(-qmax, qmax + 1, size=64)
        ints[5] = -qmax
        s0 = float(np.float32(0.0371))
        q, s = O.quantize_symmetric(ints * s0, qmax)
        assert s == s0 and np.array_equal(q, ints)
    q, s = O.quantize_symmetric(np.zeros(16), O.INT4_MAX)
    assert s == 0.0 and not q.any()


def test_quantized_summary_dequantizes_to_the_summary():
    """dequantize(quantize(V, C, mu)) is (V, C, mu) to within half a step of
    each vector's scale, column by column (a transposed layout or a scale
    applied to the wrong axis breaks this), and its page LSE follows the
    centred equation for s_hat_j(q)."""
    rng = np.random.default_rng(13)
    K = rng.standard_normal((64, 128)) + 0.5
    V, C, mu, _ = O.page_summary(K, 6, centered=True)
    qs = O.quantize_summary(V, C, mu)
    V2, C2, mu2 = O.dequantize_summary(qs)
    assert V2.shape == V.shape and C2.shape == C.shape
    assert np.all(np.abs(V2 - V) <= qs["sv"][None, :] / 2 * (1 + 1e-9))
    assert np.all(np.abs(C2 - C) <= qs["sc"][None, :] / 2 * (1 + 1e-9))
    assert np.all(np.abs(mu2 - mu) <= qs["smu"] / 2 * (1 + 1e-9))
    q = rng.standard_normal(128)
    direct = math.log(math.fsum(math.exp(v) for v in (C2 @ V2.T @ q + q @ mu2) / math.sqrt(128)))
    assert abs(O.reconstructed_page_lse(q, V2, C2, mu2) - direct) < 1e-12


# --- reconstruction error (the builder's parity measure) ----------------------

def test_reconstruction_error_closed_forms():
    """Relative reconstruction error ||K - (1 mu^T + C V^T)||_F / ||K||_F, the
    measure by which a summary is compared with the truncated SVD (explainer
    §2 'Kernmechanisme'; Theorem 1, explainer §3, bounds the output error by
    this residual).  Hand-built cases, no SVD involved:
      * K has entries 3 at (0, 0) and 4 at (1, 1); the summary keeps the first
        (V = e_0, C = 3 e_0): residual 4, ||K|| = 5, error 4/5 (dividing by
        the reconstruction's norm 3 would give 4/3);
      * a summary of all zeros reconstructs nothing: error 1;
      * K = 1 mu^T + c v^T exactly, with mu given: error 0; the same summary
        without mu leaves the centroid part: error ||1 mu^T|| / ||K||."""
    P, d = 16, 32
    K = np.zeros((P, d))
    K[0, 0], K[1, 1] = 3.0, 4.0
    V = np.zeros((d, 1))
    V[0, 0] = 1.0
    C = np.zeros((P, 1))
    C[0, 0] = 3.0
    assert abs(O.reconstruction_error(K, V, C) - 0.8) < 1e-15
    assert O.reconstruction_error(K, np.zeros((d, 2)), np.zeros((P, 2))) == 1.0
    rng = np.random.default_rng(21)
    mu = rng.standard_normal(d)
    v = _orth(rng, d, 1)
    c = rng.standard_normal((P, 1))
    K2 = np.tile(mu, (P, 1)) + c @ v.T
    assert O.reconstruction_error(K2, v, c, mu) < 1e-14
    want = math.sqrt(P) * np.linalg.norm(mu) / np.linalg.norm(K2)
    assert abs(O.reconstruction_error(K2, v, c) - want) < 1e-12


def test_reconstruction_error_equals_spectral_tail():
    """For the rank-r truncated SVD the error is sqrt(sum_{i>r} sigma_i^2 /
    sum_i sigma_i^2) (Eckart-Young): a page of exact rank 2 with singular
    values (5, 2) has error 2/sqrt(29) at r = 1 and 0 at r = 2; a centred page
    of identical keys has error 0 at any rank."""
    rng = np.random.default_rng(22)
    P, d = 16, 32
    U = _orth(rng, P, 2)
    W = _orth(rng, d, 2)
    K = 5.0 * np.outer(U[:, 0], W[:, 0]) + 2.0 * np.outer(U[:, 1], W[:, 1])
    V1, C1, _, _ = O.page_summary(K, 1)
    assert abs(O.reconstruction_error(K, V1, C1) - 2.0 / math.sqrt(29.0)) < 1e-12
    V2, C2, _, _ = O.page_summary(K, 2)
    assert O.reconstruction_error(K, V2, C2) < 1e-13
    k = rng.standard_normal(d)
    Ki = np.tile(k, (P, 1))
    Vc, Cc, muc, _ = O.page_summary(Ki, 3, centered=True)
    assert O.reconstruction_error(Ki, Vc, Cc, muc) < 1e-14


# --- sparse decode over a given page list --------------------------------------

def _gather_by_token(pool_f64, block_table, b, h, pages, L, P):
    """Rows of the listed logical pages' tokens, one token at a time: token t
    of the sequence lives in physical page block_table[b, t // P], slot t % P,
    and exists only for t < L."""
    rows = []
    for j in pages:
        for t in range(j * P, (j + 1) * P):
            if t < L:
                rows.append(pool_f64[int(block_table[b, t // P]), h, t % P])
    return np.array(rows).reshape(-1, pool_f64.shape[-1])


@pytest.mark.parametrize("P", [64, 16])
def test_sparse_decode_equals_attention_over_listed_tokens(P):
    """Attention over the selected pages plus the open tail (LOCKS abstract:
    only the top pages are attended; the open tail is read densely): for a
    hand-chosen page list, with the last full page left unsummarised and a
    partial last page, sparse_decode equals attention over exactly the tokens
    of those pages and of every page from n_summarized to ceil(L / P) - 1,
    gathered token by token."""
    case = _small_case(seed=14, P=P)
    nsum = np.array([case.n_full_pages(b) - 1 for b in range(case.batch)])
    rng = np.random.default_rng(23)
    sel = {(b, h): np.sort(rng.choice(int(nsum[b]), 4, replace=False))
           for b in range(case.batch) for h in range(case.num_kv_heads)}
    out, lse = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, sel,
                               case.num_kv_heads, page_size=P)
    kf, vf, qf = O.bf16_widen(case.k_pool), O.bf16_widen(case.v_pool), O.bf16_widen(case.q)
    G = case.group
    for (b, h), pages in sel.items():
        L = int(case.seq_lens[b])
        assert L % P, "the case must end in a partial page"
        tail = list(range(int(nsum[b]), -(-L // P)))
        assert len(tail) == 2
        Kt = _gather_by_token(kf, case.block_table, b, h, list(pages) + tail, L, P)
        Vt = _gather_by_token(vf, case.block_table, b, h, list(pages) + tail, L, P)
        assert Kt.shape[0] == 4 * P + P + L % P
        o, l = O.attention(qf[b, h * G:(h + 1) * G], Kt, Vt)
        assert np.allclose(out[b, h * G:(h + 1) * G], o, atol=1e-12)
        assert np.allclose(lse[b, h * G:(h + 1) * G], l, atol=1e-12)


@pytest.mark.parametrize("P", [64, 16])
def test_sparse_decode_every_page_equals_dense(P):
    """Listing every summarised page leaves nothing out: with the tail added
    the token set is the whole sequence, so sparse_decode equals dense
    attention (and an empty list with nothing summarised does too)."""
    case = _small_case(seed=15, P=P)
    nsum = np.array([case.n_full_pages(b) - 2 for b in range(case.batch)])
    allsel = {(b, h): np.arange(int(nsum[b])) for b in range(case.batch) for h in range(case.num_kv_heads)}
    out, lse = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum, allsel,
                               case.num_kv_heads, page_size=P)
    od, ld = O.dense_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                            case.num_kv_heads, page_size=P)
    assert np.allclose(out, od, atol=1e-12) and np.allclose(lse, ld, atol=1e-12)
    none = {k: np.zeros(0, int) for k in allsel}
    out0, lse0 = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                 np.zeros(case.batch, int), none, case.num_kv_heads, page_size=P)
    assert np.allclose(out0, od, atol=1e-12) and np.allclose(lse0, ld, atol=1e-12)


def test_sparse_decode_on_decode_step_selection_equals_decode_step():
    """sparse_decode on the page lists that decode_step selected gives
    decode_step's own output: the two restate one page-list rule."""
    case = _small_case(seed=16)
    basis, coeffs = _oracle_summaries(case, 4)
    nsum = np.array([case.n_full_pages(b) - 1 for b in range(case.batch)])
    r = O.decode_step(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum,
                      basis, coeffs, case.num_kv_heads, budget_tokens=64 * 6)
    out, lse = O.sparse_decode(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, nsum,
                               r["sel"], case.num_kv_heads)
    assert np.allclose(out, r["out"], atol=1e-13) and np.allclose(lse, r["lse"], atol=1e-13)
