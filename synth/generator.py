"""Seeded generator of page-local low-rank KV caches (inputs only).

Every array is drawn with numpy's PCG64 from one seed, in float32, and rounded
to bf16 (round-to-nearest-even) once.  Both sides of every parity test read the
same bf16 bit patterns: the oracle widens them to float64, the CUDA path uses
them as they are.

Key recipe, per (sequence b, KV head h, page p) with true rank t_p:

    K_p = (A_p B_p^T) D + E_p
    A_p ~ N(0, 1)              (P x t_p)
    B_p  orthonormal           (d x t_p)   QR of a Gaussian draw
    D    = diag(10 on 4 shared outlier channels, 1 elsewhere)
    E_p ~ N(0, 0.05^2)         (P x d)

With ``drift=True`` the bases of consecutive pages mix: B_p is the orthonormal
factor of 0.9 B_{p-1} + 0.1 G_p.  A carrier page assigned to query head g of
the group gets keys (A'_p B'_p^T D) + 3 q_hat + E_p, where q_hat = q_g/|q_g| and
B'_p has rank t_p - 1 and is orthogonal to q_hat, so the page's key subspace
contains the direction 3 q_hat.  Values and queries are N(0, 1).

Token slots past a sequence's length (inside its last page) and physical pages
that no sequence owns are filled with NaN, so that a kernel which reads them
by mistake poisons its output.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE_SIZE = 64
HEAD_DIM = 128

# The five workloads of the benchmark, by name.  Shapes follow Llama-3.1-8B
# (32 query / 8 KV heads) and GLM-4-9B-Chat-1M style GQA-16 attention.
CONFIGS = {
    "tiny": dict(batch=1, num_q_heads=1, num_kv_heads=1, context=4096, rank=8,
                 budget_tokens=512, true_rank=(8, 8), n_carriers=1, drift=False, seed=0),
    "llama128k": dict(batch=1, num_q_heads=32, num_kv_heads=8, context=131072, rank=8,
                      budget_tokens=2048, true_rank=(8, 8), n_carriers=16, drift=False, seed=1),
    "sweep": dict(batch=8, num_q_heads=32, num_kv_heads=8, context=32768, rank=8,
                  budget_tokens=1024, true_rank=(2, 16), n_carriers=16, drift=False, seed=2),
    "ctx1m": dict(batch=1, num_q_heads=32, num_kv_heads=2, context=1048576, rank=8,
                  budget_tokens=2048, true_rank=(8, 8), n_carriers=16, drift=True, seed=3),
    "growing": dict(batch=32, num_q_heads=32, num_kv_heads=8, context=8192, rank=4,
                    budget_tokens=1024, true_rank=(8, 8), n_carriers=16, drift=False, seed=4,
                    decode_steps=1024),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    nan = np.isnan(x)
    r = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class LocksCase:
    """One synthetic paged KV cache plus the decode-step query.

    Layouts (all C-contiguous):
      k_pool, v_pool  uint16 bf16 bits [pages_total][num_kv_heads][page_size][head_dim]
      block_table     int32 [batch][max_pages], physical page id or -1
      seq_lens        int32 [batch], tokens in the cache including the current one
      q               uint16 bf16 bits [batch][num_q_heads][head_dim]
      carriers        int32 [batch][num_kv_heads][n_carriers] logical page, -1 = none
      carrier_heads   int32 same shape, query head within the GQA group
    """

    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    seq_lens: np.ndarray
    block_table: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    q: np.ndarray
    carriers: np.ndarray
    carrier_heads: np.ndarray
    outlier_channels: np.ndarray
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def pages_total(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def n_pages(self, b: int) -> int:
        return -(-int(self.seq_lens[b]) // self.page_size)

    def n_full_pages(self, b: int) -> int:
        return int(self.seq_lens[b]) // self.page_size


def _orthonormal(rng: np.random.Generator, n: int, d: int, t: int) -> np.ndarray:
    g = rng.standard_normal((n, d, t), dtype=np.float32).astype(np.float64)
    qf, _ = np.linalg.qr(g)
    return qf


def make_case(batch: int, num_q_heads: int, num_kv_heads: int, seq_lens, *,
              true_rank=(8, 8), n_carriers: int = 1, drift: bool = False, seed: int = 0,
              head_dim: int = HEAD_DIM, page_size: int = PAGE_SIZE, spare_pages: int = 0,
              max_pages: int | None = None, noise: float = 0.05, outlier_scale: float = 10.0,
              n_outliers: int = 4, carrier_gain: float = 3.0, chunk_pages: int = 2048) -> LocksCase:
    """Draw one cache.  ``seq_lens`` is an int or a list of per-sequence lengths."""
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    if isinstance(seq_lens, (int, np.integer)):
        seq_lens = [int(seq_lens)] * batch
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (batch,)
    G = num_q_heads // num_kv_heads
    P, d = page_size, head_dim
    rng = np.random.Generator(np.random.PCG64(seed))

    n_pages = [-(-int(s) // P) for s in seq_lens]
    need = max(n_pages) if n_pages else 0
    if max_pages is None:
        max_pages = max(need, 1)
    if max_pages < need:
        raise ValueError("max_pages smaller than the longest sequence")
    pages_total = int(sum(n_pages)) + int(spare_pages)
    pages_total = max(pages_total, 1)

    outliers = np.sort(rng.choice(d, size=n_outliers, replace=False)).astype(np.int32)
    dscale = np.ones(d, dtype=np.float32)
    dscale[outliers] = outlier_scale

    q_f = rng.standard_normal((batch, num_q_heads, d), dtype=np.float32)
    q_bits = bf16_bits(q_f)
    q_used = bf16_to_f32(q_bits).astype(np.float64)

    perm = rng.permutation(pages_total).astype(np.int32)
    block_table = np.full((batch, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(batch):
        block_table[b, :n_pages[b]] = perm[off:off + n_pages[b]]
        off += n_pages[b]

    nan16 = np.uint16(0x7FC0)
    k_pool = np.full((pages_total, num_kv_heads, P, d), nan16, dtype=np.uint16)
    v_pool = np.full((pages_total, num_kv_heads, P, d), nan16, dtype=np.uint16)

    carriers = np.full((batch, num_kv_heads, max(n_carriers, 1)), -1, dtype=np.int32)
    carrier_heads = np.full_like(carriers, -1)

    lo, hi = true_rank
    tmax = hi
    for b in range(batch):
        npg = n_pages[b]
        nfull = int(seq_lens[b]) // P
        for h in range(num_kv_heads):
            nc = min(n_carriers, nfull)
            cpages = np.sort(rng.choice(nfull, size=nc, replace=False)) if nc > 0 else np.zeros(0, int)
            carriers[b, h, :nc] = cpages
            carrier_heads[b, h, :nc] = np.arange(nc) % G
            cmap = {int(p): int(i) for i, p in enumerate(cpages)}
            prev_basis = None
            for p0 in range(0, npg, chunk_pages):
                p1 = min(npg, p0 + chunk_pages)
                n = p1 - p0
                tr = rng.integers(lo, hi + 1, size=n) if hi > lo else np.full(n, lo)
                if drift:
                    basis = np.empty((n, d, tmax))
                    fresh = rng.standard_normal((n, d, tmax), dtype=np.float32).astype(np.float64)
                    for i in range(n):
                        if prev_basis is None:
                            mixed = fresh[i]
                        else:
                            mixed = 0.9 * prev_basis + 0.1 * fresh[i]
                        prev_basis, _ = np.linalg.qr(mixed)
                        basis[i] = prev_basis
                else:
                    basis = _orthonormal(rng, n, d, tmax)
                coef = rng.standard_normal((n, P, tmax), dtype=np.float32).astype(np.float64)
                colmask = (np.arange(tmax)[None, :] < tr[:, None]).astype(np.float64)
                coef *= colmask[:, None, :]
                # carrier pages: replace the basis by a rank t-1 one orthogonal to
                # q_hat and add carrier_gain * q_hat to every key of the page.
                shift = np.zeros((n, d))
                for i in range(n):
                    p = p0 + i
                    if p in cmap:
                        g = int(carrier_heads[b, h, cmap[p]])
                        qh = q_used[b, h * G + g]
                        qh = qh / np.linalg.norm(qh)
                        t = int(tr[i])
                        draw = rng.standard_normal((d, max(t - 1, 1)), dtype=np.float32).astype(np.float64)
                        draw -= np.outer(qh, qh @ draw)
                        bq, _ = np.linalg.qr(draw)
                        basis[i] = 0.0
                        if t - 1 > 0:
                            basis[i, :, :t - 1] = bq[:, :t - 1]
                        coef[i, :, t - 1:] = 0.0
                        shift[i] = carrier_gain * qh
                keys = np.einsum("npt,ndt->npd", coef, basis) * dscale[None, None, :]
                keys += shift[:, None, :]
                keys += noise * rng.standard_normal((n, P, d), dtype=np.float32)
                vals = rng.standard_normal((n, P, d), dtype=np.float32)
                phys = block_table[b, p0:p1]
                kb = bf16_bits(keys.astype(np.float32))
                vb = bf16_bits(vals)
                if p1 == npg and int(seq_lens[b]) % P:
                    used = int(seq_lens[b]) - (npg - 1) * P
                    kb[-1, used:] = nan16
                    vb[-1, used:] = nan16
                k_pool[phys, h] = kb
                v_pool[phys, h] = vb
    return LocksCase(batch=batch, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                     head_dim=d, page_size=P, seq_lens=seq_lens, block_table=block_table,
                     k_pool=k_pool, v_pool=v_pool, q=q_bits, carriers=carriers,
                     carrier_heads=carrier_heads, outlier_channels=outliers, seed=seed,
                     meta=dict(true_rank=tuple(true_rank), drift=drift, n_carriers=n_carriers))


def make_config_case(name: str, *, context: int | None = None, batch: int | None = None,
                     seed: int | None = None, **overrides) -> tuple[LocksCase, dict]:
    """Draw the named workload (optionally shrunk).  Returns (case, settings)."""
    cfg = dict(CONFIGS[name])
    if context is not None:
        cfg["context"] = context
    if batch is not None:
        cfg["batch"] = batch
    if seed is not None:
        cfg["seed"] = seed
    cfg.update(overrides)
    case = make_case(cfg["batch"], cfg["num_q_heads"], cfg["num_kv_heads"], cfg["context"],
                     true_rank=cfg["true_rank"], n_carriers=cfg["n_carriers"], drift=cfg["drift"],
                     seed=cfg["seed"], spare_pages=cfg.get("spare_pages", 0),
                     max_pages=cfg.get("max_pages"), page_size=cfg.get("page_size", PAGE_SIZE))
    return case, cfg


def logical_pages(case: LocksCase, b: int) -> int:
    return int(math.ceil(int(case.seq_lens[b]) / case.page_size))
