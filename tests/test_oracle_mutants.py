"""Plant plausible mistakes in the oracle (on the CPU) and check that at least
one pin in test_oracle_pins.py fails for each: evidence that the pins would
catch a dropped term, a wrong sign or index, or a transposed operand."""

import functools
import math

import numpy as np
import pytest

import oracle
import oracle.locks_oracle as L
import tests.test_oracle_pins as pins


def _lse_no_shift(x, axis=-1):
    x = np.asarray(x, dtype=np.float64)
    if x.shape[axis] == 0:
        return np.full(np.delete(x.shape, axis if axis >= 0 else x.ndim + axis), -np.inf)
    with np.errstate(over="ignore", divide="ignore"):
        return np.log(np.sum(np.exp(x), axis=axis))


def _logits_no_scale(q, V, C, mu=None, scale=None):
    out = C @ (V.T @ np.asarray(q, dtype=np.float64))
    if mu is not None:
        out = out + float(np.asarray(q) @ mu)
    return out


def _logits_minus_mu(q, V, C, mu=None, scale=None):
    d = np.asarray(q).shape[-1]
    out = C @ (V.T @ np.asarray(q, dtype=np.float64))
    if mu is not None:
        out = out - float(np.asarray(q) @ mu)
    return out / math.sqrt(d)


def _gsa_raw_mean(shat):
    shat = np.asarray(shat, dtype=np.float64)
    return np.log(np.exp(shat).mean(axis=0))


def _gsa_max(shat):
    return np.max(np.asarray(shat, dtype=np.float64), axis=0)


def _topk_ties_high(sigma, k):
    sigma = np.asarray(sigma, dtype=np.float64)
    n = sigma.size
    k = max(0, min(int(k), n))
    order = sorted(range(n), key=lambda j: (-sigma[j], -j))
    return np.array(sorted(order[:k]), dtype=np.int64)


def _summary_no_sigma(K, r, centered=False):
    V, C, mu, S = ORIG["page_summary"](K, r, centered)
    nz = np.linalg.norm(C, axis=0) > 0
    C = C.copy()
    C[:, nz] /= np.linalg.norm(C[:, nz], axis=0)
    return V, C, mu, S


def _summary_smallest(K, r, centered=False):
    K = np.asarray(K, dtype=np.float64)
    P, d = K.shape
    mu = K.mean(axis=0) if centered else np.zeros(d)
    U, S, Wt = np.linalg.svd(K - mu, full_matrices=False)
    idx = np.argsort(S)[:r]
    V = np.zeros((d, r))
    C = np.zeros((P, r))
    for c, i in enumerate(idx):
        V[:, c] = Wt[i]
        C[:, c] = U[:, i] * S[i]
    return V, C, mu, S


def _attention_no_scale(q, K, V, scale=None):
    return ORIG["attention"](q, K, V, 1.0)


def _quant_floor(x, qmax):
    x = np.asarray(x, dtype=np.float64)
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    s = float(np.float32(amax / qmax)) if amax > 0 else 0.0
    if s == 0.0:
        return np.zeros(x.shape, dtype=np.int64), 0.0
    return np.clip(np.floor(x / s), -qmax, qmax).astype(np.int64), s


def _quant_wide_scale(x, qmax):
    return ORIG["quantize_symmetric"](x, qmax + 1)


def _page_tokens_fixed_64(pool_f64, block_table, b, h, pages, seq_len, P):
    return ORIG["_page_tokens"](pool_f64, block_table, b, h, pages, seq_len, 64)


def _recon_error_over_reconstruction_norm(K, V, C, mu=None):
    K = np.asarray(K, dtype=np.float64)
    R = C @ V.T
    if mu is not None:
        R = R + np.asarray(mu, dtype=np.float64)[None, :]
    nr = np.linalg.norm(R)
    return float(np.linalg.norm(K - R) / nr) if nr > 0 else 1.0


def _recon_error_without_centroid(K, V, C, mu=None):
    return ORIG["reconstruction_error"](K, V, C, None)


def _sparse_decode_variant(drop_tail=False, floor_pages=False):
    def f(q, k_pool, v_pool, block_table, seq_lens, n_summarized, sel, num_kv_heads, page_size=64, scale=None):
        qf, kf, vf = L._widen(q), L._widen(k_pool), L._widen(v_pool)
        B, Hq, d = qf.shape
        G = Hq // num_kv_heads
        P = page_size
        out = np.zeros((B, Hq, d))
        lse = np.full((B, Hq), -np.inf)
        for b in range(B):
            n = int(seq_lens[b])
            n_pages = n // P if floor_pages else -(-n // P)
            n_sum = min(int(n_summarized[b]), n // P)
            for h in range(num_kv_heads):
                pages = [int(j) for j in sel[(b, h)]] + ([] if drop_tail else list(range(n_sum, n_pages)))
                Kt = L._page_tokens(kf, block_table, b, h, pages, n, P)
                Vt = L._page_tokens(vf, block_table, b, h, pages, n, P)
                o, l = L.attention(qf[b, h * G:(h + 1) * G], Kt, Vt, scale)
                out[b, h * G:(h + 1) * G] = o
                lse[b, h * G:(h + 1) * G] = l
        return out, lse
    return f


ORIG = {n: getattr(L, n) for n in ("page_summary", "attention", "quantize_symmetric", "_page_tokens",
                                   "reconstruction_error")}

MUTANTS = {
    "lse_without_max_shift": ("logsumexp", _lse_no_shift),
    "logits_without_1_over_sqrt_d": ("reconstructed_logits", _logits_no_scale),
    "centroid_term_sign": ("reconstructed_logits", _logits_minus_mu),
    "gsa_raw_mass_mean": ("gsa_scores", _gsa_raw_mean),
    "gsa_max_instead_of_mean": ("gsa_scores", _gsa_max),
    "topk_ties_to_higher_index": ("select_top_pages", _topk_ties_high),
    "summary_coefficients_without_sigma": ("page_summary", _summary_no_sigma),
    "summary_smallest_singular_vectors": ("page_summary", _summary_smallest),
    "attention_without_scale": ("attention", _attention_no_scale),
    "quantize_truncates": ("quantize_symmetric", _quant_floor),
    "quantize_scale_one_code_too_wide": ("quantize_symmetric", _quant_wide_scale),
    "page_tokens_assume_64_token_pages": ("_page_tokens", _page_tokens_fixed_64),
    "reconstruction_error_over_reconstruction_norm": ("reconstruction_error", _recon_error_over_reconstruction_norm),
    "reconstruction_error_ignores_centroid": ("reconstruction_error", _recon_error_without_centroid),
    "sparse_decode_drops_the_tail": ("sparse_decode", _sparse_decode_variant(drop_tail=True)),
    "sparse_decode_floor_page_count": ("sparse_decode", _sparse_decode_variant(floor_pages=True)),
}


def _at_page_size(test, P):
    f = functools.partial(test, P=P)
    f.__name__ = f"{test.__name__}[P={P}]"
    return f


PIN_TESTS = [
    pins.test_lse_brute_force_tiny_pages,
    pins.test_scale_closed_form_ln10,
    pins.test_summary_exact_low_rank_and_truncation,
    pins.test_eckart_young_residual_optimal,
    pins.test_centered_summary_identical_keys_closed_form,
    pins.test_gsa_closed_form,
    pins.test_gsa_normalisation_changes_ranking,
    pins.test_topk_ties_go_to_lower_index_and_sorted,
    pins.test_attention_closed_form_weights,
    pins.test_summary_transpose_slip_detected,
    pins.test_quantize_roundtrip_within_half_step,
    pins.test_quantize_exact_on_its_grid,
    pins.test_quantized_summary_dequantizes_to_the_summary,
    _at_page_size(pins.test_sparse_equals_dense_over_chosen_tokens, 64),
    _at_page_size(pins.test_sparse_equals_dense_over_chosen_tokens, 16),
    pins.test_reconstruction_error_closed_forms,
    pins.test_reconstruction_error_equals_spectral_tail,
    _at_page_size(pins.test_sparse_decode_equals_attention_over_listed_tokens, 64),
    _at_page_size(pins.test_sparse_decode_every_page_equals_dense, 16),
    pins.test_sparse_decode_on_decode_step_selection_equals_decode_step,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(L, attr, fn)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, fn)
    failed = []
    for t in PIN_TESTS:
        try:
            with np.errstate(all="ignore"):
                t()
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failed.append(t.__name__)
    assert failed, f"no pin caught mutant {name}"
