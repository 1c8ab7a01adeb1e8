"""Shared helpers of the test suite: moving synthetic cases to the GPU and
computing oracle summaries in the library's storage layout (test-side
marshalling only; no method arithmetic beyond calling the oracle)."""

from __future__ import annotations

import numpy as np

import oracle as O
from synth import bf16_bits, bf16_to_f32


def oracle_summaries_bf16(case, r: int, pages=None):
    """Oracle rank-r summaries of every full page (or the listed physical
    pages), rounded to bf16, in the C-ABI layouts:
    basis_t uint16 [pages_total][Hkv][r][d], coeffs uint16 [pages_total][Hkv][P][r]."""
    kf = O.bf16_widen(case.k_pool)
    pt, hkv, P, d = case.k_pool.shape
    basis_t = np.zeros((pt, hkv, r, d), dtype=np.uint16)
    coeffs = np.zeros((pt, hkv, P, r), dtype=np.uint16)
    if pages is None:
        pages = []
        for b in range(case.batch):
            pages.extend(int(x) for x in case.block_table[b, :case.n_full_pages(b)])
    for p in pages:
        for h in range(hkv):
            V, C, _, _ = O.page_summary(kf[p, h], r)
            basis_t[p, h] = bf16_bits(V.T.astype(np.float32))
            coeffs[p, h] = bf16_bits(C.astype(np.float32))
    return basis_t, coeffs


def q4_block_bytes(r: int, P: int = 64) -> int:
    """LOCKS_Q4_BLOCK_BYTES(r, P): 64r basis + 128 centroid + P r coefficients
    + 4 (2r + 1) scales, rounded up to 16."""
    return (64 * r + 128 + P * r + 4 * (2 * r + 1) + 15) // 16 * 16


def _q4_word_position(m):
    """Word m of a basis row sits at word 4(m%4) + m/4 of the row."""
    return 4 * (m % 4) + m // 4


def _q4_coef_position(i, j, r, P):
    """Byte of the code of token i, column j in the coefficient block."""
    return (((i % 8) * (r // 2) + j // 2) * (P // 8) + i // 8) * 2 + j % 2


def _q4_scale_order(r):
    """Float index -> (which, column): per column pair t, s_v[2t], s_v[2t+1],
    s_c[2t], s_c[2t+1]; then s_mu."""
    order = []
    for t in range(r // 2):
        order += [("sv", 2 * t), ("sv", 2 * t + 1), ("sc", 2 * t), ("sc", 2 * t + 1)]
    return order + [("smu", 0)]


def pack_q4(qs: dict, r: int) -> np.ndarray:
    """One oracle-quantised page-head summary in the LOCKS_DTYPE_Q4 byte layout
    of include/locks.h (the page size is the coefficient block's row count)."""
    P = np.asarray(qs["cq"]).shape[0]
    buf = np.zeros(q4_block_bytes(r, P), dtype=np.uint8)
    u = (np.asarray(qs["vq"]) + 8).astype(np.uint32).reshape(r, 16, 8)  # [row][word][element], code + 8
    words = np.zeros((r, 16), dtype=np.uint32)
    for i in range(8):
        words |= u[:, :, i] << np.uint32(4 * (i // 2) + 16 * (i % 2))
    placed = np.zeros_like(words)
    for m in range(16):
        placed[:, _q4_word_position(m)] = words[:, m]
    buf[:64 * r] = placed.astype("<u4").view(np.uint8).reshape(-1)
    buf[64 * r:64 * r + 128] = (np.asarray(qs["muq"]) + 128).astype(np.uint8)
    c0 = 64 * r + 128
    cq = np.asarray(qs["cq"])
    for i in range(P):
        for j in range(r):
            buf[c0 + _q4_coef_position(i, j, r, P)] = cq[i, j] + 128
    vals = {"sv": np.asarray(qs["sv"]), "sc": np.asarray(qs["sc"]), "smu": np.asarray([qs["smu"]])}
    scales = np.array([vals[w][c] for w, c in _q4_scale_order(r)], dtype=np.float32)
    buf[c0 + P * r:c0 + P * r + 4 * (2 * r + 1)] = scales.view(np.uint8)
    return buf


def unpack_q4(buf: np.ndarray, r: int, P: int = 64, d: int = 128) -> dict:
    """Inverse of pack_q4 (reads the ABI layout back into codes and scales)."""
    buf = np.asarray(buf, dtype=np.uint8)
    placed = buf[:64 * r].copy().view("<u4").reshape(r, d // 8).astype(np.int64)
    words = np.stack([placed[:, _q4_word_position(m)] for m in range(d // 8)], axis=1)
    vq = np.empty((r, d // 8, 8), dtype=np.int64)
    for i in range(8):
        vq[:, :, i] = ((words >> (4 * (i // 2) + 16 * (i % 2))) & 15) - 8
    vq = vq.reshape(r, d)
    muq = buf[64 * r:64 * r + 128].astype(np.int64) - 128
    c0 = 64 * r + 128
    cq = np.empty((P, r), dtype=np.int64)
    for i in range(P):
        for j in range(r):
            cq[i, j] = int(buf[c0 + _q4_coef_position(i, j, r, P)]) - 128
    flat = buf[c0 + P * r:c0 + P * r + 4 * (2 * r + 1)].view(np.float32).astype(np.float64)
    out = {"sv": np.zeros(r), "sc": np.zeros(r), "smu": 0.0}
    for f, (w, c) in zip(flat, _q4_scale_order(r)):
        if w == "smu":
            out["smu"] = float(f)
        else:
            out[w][c] = f
    return dict(vq=vq, sv=out["sv"], cq=cq, sc=out["sc"], muq=muq, smu=out["smu"])


def oracle_summaries_q4(case, r: int, heads=None, pages=None):
    """Oracle quantised centred summaries of every full page (or the listed
    physical pages) for the listed KV heads (default all): the packed ABI
    array uint8 [pages_total][Hkv][bytes] and the values it stands for in the
    oracle layout (basis [..][d][r], coeffs [..][P][r], centroid [..][d])."""
    pt, hkv, P, d = case.k_pool.shape
    packed = np.zeros((pt, hkv, q4_block_bytes(r, P)), dtype=np.uint8)
    basis = np.zeros((pt, hkv, d, r))
    coeffs = np.zeros((pt, hkv, P, r))
    cent = np.zeros((pt, hkv, d))
    if pages is None:
        pages = []
        for b in range(case.batch):
            pages.extend(int(x) for x in case.block_table[b, :case.n_full_pages(b)])
    for p in pages:
        for h in (range(hkv) if heads is None else heads):
            qs = O.quantized_page_summary(O.bf16_widen(case.k_pool[p, h]), r)
            packed[p, h] = pack_q4(qs, r)
            basis[p, h], coeffs[p, h], cent[p, h] = O.dequantize_summary(qs)
    return packed, basis, coeffs, cent


def oracle_layout_from_abi(basis_t_u16, coeffs_u16):
    """ABI layout (bf16 bits) -> oracle layout float64: basis [..][d][r], coeffs [..][P][r]."""
    basis = np.swapaxes(bf16_to_f32(basis_t_u16).astype(np.float64), -1, -2)
    coeffs = bf16_to_f32(coeffs_u16).astype(np.float64)
    return basis, coeffs


def to_torch_bf16(arr_u16, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr_u16).view(np.int16)).view(torch.bfloat16).to(device)


def torch_bf16_to_u16(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_runtime(case, rank: int, budget_tokens: int, n_summarized=None, device="cuda", quantized=False,
                 split=False):
    import torch
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime
    if n_summarized is None:
        n_summarized = [case.n_full_pages(b) for b in range(case.batch)]
    rt = LocksRuntime(to_torch_bf16(case.k_pool, device), to_torch_bf16(case.v_pool, device),
                      torch.from_numpy(case.block_table).to(device),
                      torch.from_numpy(case.seq_lens).to(device),
                      torch.tensor(np.asarray(n_summarized, dtype=np.int32)).to(device),
                      case.num_q_heads, rank, budget_tokens, quantized=quantized, split=split)
    q = to_torch_bf16(case.q, device)
    return rt, q


def cut_band_ok(sigma_oracle: np.ndarray, sel_gpu, sel_oracle, k: int, band: float = 1e-4):
    """Selection comparison outside the band |sigma - sigma_(k)| <= band around
    the cut.  Returns (ok, detail)."""
    n = sigma_oracle.size
    k = min(k, n)
    if k == 0:
        return len(sel_gpu) == 0, "k=0"
    if k >= n:
        return sorted(sel_gpu) == list(range(n)), "all"
    kth = np.sort(sigma_oracle)[::-1][k - 1]
    near = set(np.nonzero(np.abs(sigma_oracle - kth) <= band)[0].tolist())
    a = set(int(x) for x in sel_gpu) - near
    b = set(int(x) for x in sel_oracle) - near
    return a == b and len(sel_gpu) == k, f"gpu-only={sorted(a - b)} oracle-only={sorted(b - a)} near={len(near)}"
