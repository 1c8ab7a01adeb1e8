"""Seeded page-local KV caches drawn on the GPU (inputs only).

For workloads too large to draw on the host: at 256K context a batch of 64
sequences holds 69 GB of keys and values.  The recipe is the one of
``synth.generator`` —

    K_p = (A_p B_p^T) D + E_p,  A_p ~ N(0, 1) (P x t),  B_p orthonormal (d x t),
    D = 10 on four outlier channels shared by the cache and 1 elsewhere,
    E_p ~ N(0, 0.05^2);  values and queries N(0, 1);

carrier pages (``n_carriers`` per sequence and KV head, at distinct seeded
full pages, carrier c assigned query head c mod G of the group) take a rank
t - 1 basis orthogonal to q_hat and 3 q_hat added to every key — but every
number comes from torch's device generator, so the values are not the host
generator's for the same seed, and no oracle reads them.  B_p is the
Gram-Schmidt orthonormalisation of a Gaussian draw.  Token slots past a
sequence's length are NaN.  Nothing here computes any part of the method.
"""

from __future__ import annotations

import math


def make_device_cache(batch: int, num_q_heads: int, num_kv_heads: int, context: int, *, true_rank=(8, 8),
                      n_carriers: int = 16, seed: int = 0, device="cuda", page_size: int = 64,
                      head_dim: int = 128, chunk_pages: int = 2048, noise: float = 0.05,
                      outlier_scale: float = 10.0, n_outliers: int = 4, carrier_gain: float = 3.0) -> dict:
    """Returns torch tensors on ``device``: k_pool, v_pool (bf16
    [pages_total][Hkv][P][d]), block_table (int32 [B][pages]), seq_lens and
    n_full (int32 [B]), q (bf16 [B][Hq][d]), carriers (int32 [B][Hkv][n_carriers],
    logical pages)."""
    import torch

    P, d = page_size, head_dim
    Hq, Hkv = num_q_heads, num_kv_heads
    if Hq % Hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    G = Hq // Hkv
    npg = math.ceil(context / P)
    nfull = context // P
    pt = batch * npg
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    outliers = torch.randperm(d, generator=gen, device=device)[:n_outliers]
    dscale = torch.ones(d, device=device)
    dscale[outliers] = outlier_scale
    q = torch.randn((batch, Hq, d), generator=gen, device=device).to(torch.bfloat16)
    qhat = q.float()
    qhat = (qhat / qhat.norm(dim=-1, keepdim=True)).view(batch * Hq, d)

    block_table = torch.randperm(pt, generator=gen, device=device).to(torch.int32).view(batch, npg)

    # carriers: distinct full pages per (sequence, KV head); carrier_row = the
    # query row (b * Hq + head) whose direction the page carries, -1 elsewhere
    nc = min(n_carriers, nfull)
    carriers = torch.full((batch, Hkv, max(n_carriers, 1)), -1, dtype=torch.int32, device=device)
    carrier_row = torch.full((pt, Hkv), -1, dtype=torch.long, device=device)
    if nc > 0:
        pick = torch.rand((batch, Hkv, nfull), generator=gen, device=device).argsort(dim=-1)[..., :nc]
        pick = pick.sort(dim=-1).values
        carriers[..., :nc] = pick.to(torch.int32)
        b_idx = torch.arange(batch, device=device)[:, None, None].expand(batch, Hkv, nc)
        h_idx = torch.arange(Hkv, device=device)[None, :, None].expand(batch, Hkv, nc)
        c_idx = torch.arange(nc, device=device)[None, None, :].expand(batch, Hkv, nc)
        phys = block_table.long()[b_idx, pick]
        carrier_row[phys, h_idx] = b_idx * Hq + h_idx * G + (c_idx % G)

    k_pool = torch.empty((pt, Hkv, P, d), dtype=torch.bfloat16, device=device)
    v_pool = torch.empty_like(k_pool)
    lo, hi = true_rank
    tmax = hi
    cols = torch.arange(tmax, device=device)
    for p0 in range(0, pt, chunk_pages):
        p1 = min(pt, p0 + chunk_pages)
        n = (p1 - p0) * Hkv
        rows = carrier_row[p0:p1].reshape(n)
        is_c = rows >= 0
        t = torch.randint(lo, hi + 1, (n,), generator=gen, device=device)
        t_used = torch.where(is_c, t - 1, t)
        g = torch.randn((n, d, tmax), generator=gen, device=device)
        qh = qhat[rows.clamp(min=0)] * is_c[:, None]
        g -= qh[:, :, None] * (qh[:, None, :] @ g)          # carriers: orthogonal to q_hat
        basis = torch.empty_like(g)
        for j in range(tmax):                                # modified Gram-Schmidt
            v = g[:, :, j]
            for i in range(j):
                v = v - (basis[:, :, i] * v).sum(-1, keepdim=True) * basis[:, :, i]
            basis[:, :, j] = v / v.norm(dim=-1, keepdim=True).clamp(min=1e-30)
        coef = torch.randn((n, P, tmax), generator=gen, device=device)
        coef *= (cols[None, :] < t_used[:, None]).float()[:, None, :]
        keys = coef @ basis.transpose(1, 2)
        keys *= dscale
        keys += carrier_gain * qh[:, None, :]
        keys += noise * torch.randn((n, P, d), generator=gen, device=device)
        vals = torch.randn((n, P, d), generator=gen, device=device)
        k_pool[p0:p1] = keys.view(p1 - p0, Hkv, P, d).to(torch.bfloat16)
        v_pool[p0:p1] = vals.view(p1 - p0, Hkv, P, d).to(torch.bfloat16)
        del g, basis, coef, keys, vals
    if context % P:
        last = block_table[:, -1].long()
        k_pool[last, :, context % P:] = float("nan")
        v_pool[last, :, context % P:] = float("nan")
    seq_lens = torch.full((batch,), context, dtype=torch.int32, device=device)
    n_full = torch.full((batch,), nfull, dtype=torch.int32, device=device)
    return dict(k_pool=k_pool, v_pool=v_pool, block_table=block_table, seq_lens=seq_lens, n_full=n_full, q=q,
                carriers=carriers)
