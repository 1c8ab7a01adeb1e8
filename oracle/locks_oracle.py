"""Plain, slow, obviously-correct fp64 implementation of the LOCKS decode step.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference legs may use this module.  It shares no code with the
CUDA path.

Sources (web pages about arXiv:2607.24555, "LOCKS: Page-Local Compact Key
Summaries for Efficient Long-Context Decoding"):
  [expl]  gist.science explainer (Dutch), "Technische Samenvatting":
          §2 Methodologie — "Kernmechanisme", "Reconstructie en Selectie"
          (the equation for s_hat_j(q)), "Group-Shared Selection (GSA)";
          §3 — Propositie 1, Theorem 1.
  [abs]   insight.aitobox.com page, "Abstract" (English paragraphs).
  [blog]  brainszone.ai blog, "Ringkasan spektral per halaman" and
          "Seleksi blok tanpa membaca key".

Notation follows the pages: a page j holds P tokens with keys k_i (i in P_j),
its summary is a basis V_j (d x r) and coefficients c_i (r-vectors, stacked into
C_j, P x r), optionally a centroid mu_j; d is the head dimension.

Readings where the pages are silent:
  * the summary is the rank-r truncated SVD of the raw P x d key block
    (V_r = right singular vectors, C = U_r Sigma_r); the centred variant of the
    explainer subtracts the page mean first and adds the q.mu_j term;
  * singular values <= 1e-6 * sigma_1 give an all-zero column (rank deficit);
  * logits are scaled by 1/sqrt(d); logs and exps are natural;
  * GSA normalises each head's page masses into shares (divide by the head's
    total estimated mass exp(Z_h)) and averages the shares over the group;
  * k = min(floor(budget / P), number of summarised full pages); ties in the
    GSA score go to the lower logical page index; the list is returned sorted
    ascending;
  * the open tail (every page of the sequence past the summarised ones,
    including the partial last page) is always attended, outside the budget.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "logsumexp", "page_summary", "reconstructed_logits", "reconstructed_page_lse",
    "exact_page_lse", "gsa_scores", "select_top_pages", "attention",
    "sparse_decode", "dense_decode", "decode_step", "build_summaries",
    "mass_recall", "carrier_retention", "shared_sketch_page_lse", "jacobi_eigh",
    "reconstruction_error", "bf16_widen", "INT4_MAX", "INT8_MAX", "quantize_symmetric",
    "quantize_summary", "dequantize_summary", "quantized_page_summary",
]

RANK_DEFICIT_RTOL = 1e-6


def bf16_widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def logsumexp(x: np.ndarray, axis=-1) -> np.ndarray:
    """ln sum exp(x) along ``axis`` with the maximum factored out; an empty or
    all -inf slice gives -inf."""
    x = np.asarray(x, dtype=np.float64)
    if x.shape[axis] == 0:
        return np.full(np.delete(x.shape, axis if axis >= 0 else x.ndim + axis), -np.inf)
    m = np.max(x, axis=axis, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    s = np.sum(np.exp(x - m_safe), axis=axis, keepdims=True)
    with np.errstate(divide="ignore"):
        out = np.log(s) + m_safe
    return np.squeeze(out, axis=axis)


# ---------------------------------------------------------------------------
# Summary construction ([expl] §2 "Kernmechanisme": a small eigendecomposition
# of the page's keys when the page is finalised; the top-r eigenvectors are the
# basis and every token keeps its coefficients).
# ---------------------------------------------------------------------------

def page_summary(K: np.ndarray, r: int, centered: bool = False):
    """Rank-r spectral summary of one page's key block K (P x d).

    Returns (V, C, mu, sing): V is d x r with orthonormal columns (the top-r
    right singular vectors of K - 1 mu^T), C = U_r Sigma_r is P x r (row i is
    c_i), mu is the centroid (zeros unless ``centered``), sing holds all
    singular values in descending order.  Columns past min(P, d) or whose
    singular value is <= 1e-6 sigma_1 are zero.
    """
    K = np.asarray(K, dtype=np.float64)
    P, d = K.shape
    mu = K.mean(axis=0) if centered else np.zeros(d)
    X = K - mu[None, :]
    U, S, Wt = np.linalg.svd(X, full_matrices=False)
    V = np.zeros((d, r))
    C = np.zeros((P, r))
    top = S[0] if S.size else 0.0
    for i in range(min(r, S.size)):
        if top > 0 and S[i] > RANK_DEFICIT_RTOL * top:
            V[:, i] = Wt[i, :]
            C[:, i] = U[:, i] * S[i]
    return V, C, mu, S


def reconstruction_error(K: np.ndarray, V: np.ndarray, C: np.ndarray, mu=None) -> float:
    """Relative Frobenius error ||K - (1 mu^T + C V^T)||_F / ||K||_F."""
    K = np.asarray(K, dtype=np.float64)
    R = C @ V.T
    if mu is not None:
        R = R + np.asarray(mu, dtype=np.float64)[None, :]
    nk = np.linalg.norm(K)
    return float(np.linalg.norm(K - R) / nk) if nk > 0 else float(np.linalg.norm(R))


def build_summaries(k_pool: np.ndarray, page_ids, r: int, centered: bool = False):
    """Summaries of the listed physical pages for every KV head.

    k_pool: float64 [pages_total][Hkv][P][d].  Returns dicts keyed by physical
    page id: basis [Hkv][d][r], coeffs [Hkv][P][r], centroid [Hkv][d].
    """
    basis, coeffs, cent = {}, {}, {}
    for p in page_ids:
        p = int(p)
        vs, cs, ms = [], [], []
        for h in range(k_pool.shape[1]):
            V, C, mu, _ = page_summary(k_pool[p, h], r, centered)
            vs.append(V)
            cs.append(C)
            ms.append(mu)
        basis[p] = np.stack(vs)
        coeffs[p] = np.stack(cs)
        cent[p] = np.stack(ms)
    return basis, coeffs, cent


# ---------------------------------------------------------------------------
# Quantised summary ([expl] §2 "Kernmechanisme", Kwantisatie bullet: the basis is
# stored in int4, the coefficients and the centroid in int8).  The pages give
# no scale layout; the reading taken here: symmetric scales, one per basis
# vector, one per coefficient column and one for the centroid, stored as
# float32; s = max|x| / qmax with qmax = 7 (int4) or 127 (int8), and
# q = round-half-to-even(x / s) clamped to [-qmax, qmax].  A zero vector has
# s = 0 and q = 0.  The value a quantised summary stands for is q * s.
# ---------------------------------------------------------------------------

INT4_MAX = 7
INT8_MAX = 127


def quantize_symmetric(x: np.ndarray, qmax: int):
    """One scale for the whole vector x: returns (q int64 array, s float)."""
    x = np.asarray(x, dtype=np.float64)
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    s = float(np.float32(amax / qmax)) if amax > 0 else 0.0
    if s == 0.0:
        return np.zeros(x.shape, dtype=np.int64), 0.0
    q = np.clip(np.rint(x / s), -qmax, qmax).astype(np.int64)
    return q, s


def quantize_summary(V: np.ndarray, C: np.ndarray, mu: np.ndarray) -> dict:
    """Quantise one page-head summary (V d x r, C P x r, centroid mu d).

    Returns vq [r][d] (int4 values), sv [r], cq [P][r] (int8 values), sc [r],
    muq [d] (int8 values), smu."""
    d, r = V.shape
    P = C.shape[0]
    vq = np.zeros((r, d), dtype=np.int64)
    cq = np.zeros((P, r), dtype=np.int64)
    sv = np.zeros(r)
    sc = np.zeros(r)
    for j in range(r):
        vq[j], sv[j] = quantize_symmetric(V[:, j], INT4_MAX)
        cq[:, j], sc[j] = quantize_symmetric(C[:, j], INT8_MAX)
    muq, smu = quantize_symmetric(mu, INT8_MAX)
    return dict(vq=vq, sv=sv, cq=cq, sc=sc, muq=muq, smu=smu)


def dequantize_summary(qs: dict):
    """The summary a quantised one stands for: (V d x r, C P x r, mu d)."""
    V = (qs["vq"] * qs["sv"][:, None]).T.astype(np.float64)
    C = (qs["cq"] * qs["sc"][None, :]).astype(np.float64)
    mu = (qs["muq"] * qs["smu"]).astype(np.float64)
    return V, C, mu


def quantized_page_summary(K: np.ndarray, r: int) -> dict:
    """Centred rank-r summary of a page-head, quantised ([expl] §2: centred
    keys, then int4 basis and int8 coefficients / centroid)."""
    V, C, mu, _ = page_summary(K, r, centered=True)
    return quantize_summary(V, C, mu)


# ---------------------------------------------------------------------------
# Reconstruction and page-mass estimate ([expl] §2 "Reconstructie en Selectie",
# the equation s_hat_j(q) = log sum_{i in P_j} exp((q.mu_j + (V_j^T q).c_i)/sqrt d);
# [abs] "reconstructs within-page logits, estimates each page's attention mass
# by log-sum-exp").
# ---------------------------------------------------------------------------

def reconstructed_logits(q: np.ndarray, V: np.ndarray, C: np.ndarray, mu=None, scale=None) -> np.ndarray:
    """l_i = (q.mu + (V^T q).c_i) * scale for every token i of the page."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    w = V.T @ q                       # V_j^T q  (r,)
    logits = C @ w                    # (V_j^T q)^T c_i for all i  (P,)
    if mu is not None:
        logits = logits + float(q @ np.asarray(mu, dtype=np.float64))
    return logits * scale


def reconstructed_page_lse(q, V, C, mu=None, scale=None) -> float:
    """s_hat_j(q): log-sum-exp of the reconstructed within-page logits."""
    return float(logsumexp(reconstructed_logits(q, V, C, mu, scale)))


def exact_page_lse(q: np.ndarray, K: np.ndarray, scale=None) -> float:
    """s*_j(q) = log sum_i exp(q.k_i * scale): the read-every-key page mass used
    by the exact LSE-oracle selector ([abs]; [expl] §3 "Retrieval en QA")."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return float(logsumexp((K @ q) * scale))


# ---------------------------------------------------------------------------
# Group-Shared Selection ([expl] §2 "Group-Shared Selection (GSA)": average the
# estimated mass share over the query heads of a GQA group into one table).
# ---------------------------------------------------------------------------

def gsa_scores(shat: np.ndarray) -> np.ndarray:
    """shat: (G, n) page masses (log domain) of the G heads of one KV group.

    Z_h = ln sum_j exp(shat[h, j]) (head h's total estimated mass);
    share[h, j] = exp(shat[h, j] - Z_h); sigma_j = ln( (1/G) sum_h share[h, j] ).
    """
    shat = np.asarray(shat, dtype=np.float64)
    G, n = shat.shape
    if n == 0:
        return np.zeros(0)
    Z = logsumexp(shat, axis=1)                          # (G,)
    shares = np.exp(shat - Z[:, None])                   # each row sums to 1
    with np.errstate(divide="ignore"):
        return np.log(shares.sum(axis=0) / G)


def select_top_pages(sigma: np.ndarray, k: int) -> np.ndarray:
    """The k pages with the largest sigma ([expl] §2: pages are ranked by their
    estimated mass); equal sigma -> lower index first; returned ascending."""
    sigma = np.asarray(sigma, dtype=np.float64)
    n = sigma.size
    k = max(0, min(int(k), n))
    order = sorted(range(n), key=lambda j: (-sigma[j], j))
    return np.array(sorted(order[:k]), dtype=np.int64)


# ---------------------------------------------------------------------------
# Attention (softmax over the chosen tokens; [blog] "only the top pages are
# processed"; the dense case reads every token).
# ---------------------------------------------------------------------------

def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale=None):
    """q (G, d), K (T, d), V (T, d) -> o (G, d), lse (G,) natural log.

    o_h = sum_t softmax_t(q_h.k_t * scale) v_t.  T = 0 gives o = 0, lse = -inf.
    """
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[-1] if V.ndim == 2 else d)), np.full(q.shape[0], -np.inf)
    s = (q @ K.T) * scale                    # (G, T)
    lse = logsumexp(s, axis=1)
    p = np.exp(s - lse[:, None])
    return p @ V, lse


def _page_tokens(pool_f64, block_table, b, h, pages, seq_len, P):
    """Gather keys (or values) of the listed logical pages of sequence b, head h,
    cut at the sequence length."""
    rows = []
    for j in pages:
        phys = int(block_table[b, j])
        n = min(P, seq_len - j * P)
        if n > 0:
            rows.append(pool_f64[phys, h, :n])
    if not rows:
        return np.zeros((0, pool_f64.shape[-1]))
    return np.concatenate(rows, axis=0)


def _widen(x):
    x = np.asarray(x)
    return bf16_widen(x) if x.dtype == np.uint16 else x.astype(np.float64)


def decode_step(q, k_pool, v_pool, block_table, seq_lens, n_summarized, basis, coeffs,
                num_kv_heads: int, budget_tokens: int, page_size: int = 64, scale=None,
                centroid=None, dense: bool = False, exact_selection: bool = False,
                want=("out",)):
    """One LOCKS decode step for every (sequence, KV head).

    q: [B][Hq][d]; k_pool, v_pool: [pages_total][Hkv][P][d] (bf16 bits or
    floats); block_table: [B][max_pages]; seq_lens, n_summarized: [B];
    basis: [pages_total][Hkv][d][r] (V_j) or None; coeffs: [pages_total][Hkv][P][r];
    centroid: optional [pages_total][Hkv][d].

    For each (b, h_kv): s_hat for every summarised page and every head of the
    group (or s* when ``exact_selection``), GSA score sigma, top-k pages, then
    attention over selected pages + open tail (or every page when ``dense``).
    Returns a dict with 'out' [B][Hq][d], 'lse' [B][Hq], 'sel' {(b,h): pages},
    'shat' {(b,h): (G, n_sum)}, 'sigma' {(b,h): (n_sum,)}.
    """
    qf = _widen(q)
    kf = _widen(k_pool)
    vf = _widen(v_pool)
    B, Hq, d = qf.shape
    G = Hq // num_kv_heads
    P = page_size
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, Hq, d))
    lse = np.full((B, Hq), -np.inf)
    sel, shats, sigmas = {}, {}, {}
    bas = None if basis is None else _widen(basis)
    coe = None if coeffs is None else _widen(coeffs)
    cen = None if centroid is None else _widen(centroid)
    for b in range(B):
        L = int(seq_lens[b])
        n_pages = -(-L // P)
        n_sum = min(int(n_summarized[b]), L // P)
        k = min(budget_tokens // P, n_sum)
        for h in range(num_kv_heads):
            qg = qf[b, h * G:(h + 1) * G]
            if dense:
                pages = list(range(n_pages))
            else:
                shat = np.zeros((G, n_sum))
                for j in range(n_sum):
                    phys = int(block_table[b, j])
                    for g in range(G):
                        if exact_selection:
                            shat[g, j] = exact_page_lse(qg[g], kf[phys, h], scale)
                        else:
                            mu = None if cen is None else cen[phys, h]
                            shat[g, j] = reconstructed_page_lse(qg[g], bas[phys, h], coe[phys, h], mu, scale)
                sigma = gsa_scores(shat)
                chosen = select_top_pages(sigma, k)
                sel[(b, h)] = chosen
                shats[(b, h)] = shat
                sigmas[(b, h)] = sigma
                pages = list(chosen) + list(range(n_sum, n_pages))
            Kt = _page_tokens(kf, block_table, b, h, pages, L, P)
            Vt = _page_tokens(vf, block_table, b, h, pages, L, P)
            o, l = attention(qg, Kt, Vt, scale)
            out[b, h * G:(h + 1) * G] = o
            lse[b, h * G:(h + 1) * G] = l
    return dict(out=out, lse=lse, sel=sel, shat=shats, sigma=sigmas)


def sparse_decode(q, k_pool, v_pool, block_table, seq_lens, n_summarized, sel, num_kv_heads,
                  page_size=64, scale=None):
    """Attention over given page lists ``sel[(b, h)]`` plus the open tail."""
    qf, kf, vf = _widen(q), _widen(k_pool), _widen(v_pool)
    B, Hq, d = qf.shape
    G = Hq // num_kv_heads
    P = page_size
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, Hq, d))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        L = int(seq_lens[b])
        n_pages = -(-L // P)
        n_sum = min(int(n_summarized[b]), L // P)
        for h in range(num_kv_heads):
            pages = [int(j) for j in sel[(b, h)]] + list(range(n_sum, n_pages))
            Kt = _page_tokens(kf, block_table, b, h, pages, L, P)
            Vt = _page_tokens(vf, block_table, b, h, pages, L, P)
            o, l = attention(qf[b, h * G:(h + 1) * G], Kt, Vt, scale)
            out[b, h * G:(h + 1) * G] = o
            lse[b, h * G:(h + 1) * G] = l
    return out, lse


def dense_decode(q, k_pool, v_pool, block_table, seq_lens, num_kv_heads, page_size=64, scale=None):
    """Attention over every token of every sequence (the dense baseline)."""
    r = decode_step(q, k_pool, v_pool, block_table, seq_lens, np.zeros(len(seq_lens), int),
                    None, None, num_kv_heads, 0, page_size, scale, dense=True)
    return r["out"], r["lse"]


# ---------------------------------------------------------------------------
# Measurement helpers ([abs]: "tracks the read-every-key exact-LSE oracle";
# [expl] §3 "carrier retention").
# ---------------------------------------------------------------------------

def mass_recall(s_star: np.ndarray, selected) -> float:
    """Mean over heads of sum_{j in S} exp(s*_hj) / sum_j exp(s*_hj), s_star (G, n)."""
    s_star = np.atleast_2d(np.asarray(s_star, dtype=np.float64))
    sel = np.asarray(list(selected), dtype=np.int64)
    tot = logsumexp(s_star, axis=1)
    if sel.size == 0:
        return 0.0
    part = logsumexp(s_star[:, sel], axis=1)
    return float(np.mean(np.exp(part - tot)))


def carrier_retention(carriers, selected) -> float:
    """Fraction of planted carrier pages that the selection kept."""
    c = [int(x) for x in np.asarray(carriers).ravel() if int(x) >= 0]
    if not c:
        return 1.0
    s = set(int(x) for x in selected)
    return sum(1 for x in c if x in s) / len(c)


def shared_sketch_page_lse(q: np.ndarray, S_sh: np.ndarray, K: np.ndarray, scale=None) -> float:
    """Page mass through a fixed query-independent shared projection S_sh
    (d x rho, orthonormal columns), the alternative the pages reject
    ([expl] §3 Propositie 1): logits (S_sh^T q).(S_sh^T k_i) * scale."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return float(logsumexp(((K @ S_sh) @ (S_sh.T @ q)) * scale))


def jacobi_eigh(A, sweeps: int = 60, tol: float = 1e-15):
    """Cyclic Jacobi eigensolver in pure Python for small symmetric matrices
    (a textbook method, used to cross-check the LAPACK SVD on tiny pages).
    Returns (eigenvalues descending, eigenvectors as columns)."""
    n = len(A)
    a = [[float(A[i][j]) for j in range(n)] for i in range(n)]
    v = [[1.0 if i == j else 0.0 for j in range(n)] for i in range(n)]
    for _ in range(sweeps):
        off = math.fsum(a[i][j] ** 2 for i in range(n) for j in range(n) if i != j)
        if off < tol * tol:
            break
        for p in range(n - 1):
            for q in range(p + 1, n):
                if abs(a[p][q]) < 1e-300:
                    continue
                theta = (a[q][q] - a[p][p]) / (2.0 * a[p][q])
                t = (1.0 if theta >= 0 else -1.0) / (abs(theta) + math.sqrt(theta * theta + 1.0))
                c = 1.0 / math.sqrt(t * t + 1.0)
                s = t * c
                for k in range(n):
                    akp, akq = a[k][p], a[k][q]
                    a[k][p] = c * akp - s * akq
                    a[k][q] = s * akp + c * akq
                for k in range(n):
                    apk, aqk = a[p][k], a[q][k]
                    a[p][k] = c * apk - s * aqk
                    a[q][k] = s * apk + c * aqk
                for k in range(n):
                    vkp, vkq = v[k][p], v[k][q]
                    v[k][p] = c * vkp - s * vkq
                    v[k][q] = s * vkp + c * vkq
    evals = [a[i][i] for i in range(n)]
    order = sorted(range(n), key=lambda i: -evals[i])
    w = np.array([evals[i] for i in order])
    vecs = np.array([[v[k][i] for i in order] for k in range(n)])
    return w, vecs
