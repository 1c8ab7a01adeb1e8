"""Device-side state of one paged cache for PyTorch callers.

``LocksRuntime`` owns the torch tensors the C ABI reads (pools, block table,
lengths, summaries, workspace), the C structs that point at them, and thin
methods that call the entry points of ``locks``.  It computes nothing itself.
"""

from __future__ import annotations

import torch

from . import locks as L


class LocksRuntime:
    """Holds a paged cache on ``device`` and calls liblocks.so on it.

    k_pool, v_pool: bf16 [pages_total][Hkv][P][128] with P = 64 or 16;
    block_table int32 [B][max_pages]; seq_lens, n_summarized int32 [B].
    Summaries are allocated here.  bf16: one LOCKS_DTYPE_BF16_PACKED block per
    page-head (basis rows, then coefficients), with ``basis_t`` [pages_total]
    [Hkv][rank][128] and ``coeffs`` [..][P][rank] as views into it; with
    ``split`` two separate LOCKS_DTYPE_BF16 arrays of those shapes instead.
    With ``quantized``: one LOCKS_DTYPE_Q4 block per page-head (uint8
    [pages_total][Hkv][q4_page_head_bytes(rank, P)]).
    ``form``: "auto" (the library's choice: three kernels), or "unfused" /
    "fused" for LOCKS_FLAG_UNFUSED / LOCKS_FLAG_FUSED (the decode step as three
    kernels, or as two wherever the size limits allow).
    """

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, n_summarized: torch.Tensor, num_q_heads: int, rank: int,
                 budget_tokens: int, scale: float = 0.0, quantized: bool = False, form: str = "auto",
                 split: bool = False):
        assert k_pool.dtype == torch.bfloat16 and v_pool.dtype == torch.bfloat16
        assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32
        self.device = k_pool.device
        self.k_pool, self.v_pool = k_pool, v_pool
        self.block_table, self.seq_lens = block_table, seq_lens
        self.n_summarized = n_summarized.to(torch.int32)
        pt, hkv, P, d = k_pool.shape
        self.batch = block_table.shape[0]
        self.num_kv_heads, self.num_q_heads = hkv, num_q_heads
        self.rank = rank
        self.quantized = quantized
        if quantized:
            self.basis_t = torch.zeros((pt, hkv, L.q4_page_head_bytes(rank, P)), dtype=torch.uint8,
                                       device=self.device)
            self.coeffs = None
            self.summary = L.make_summary(self.basis_t, None, rank, L.LOCKS_DTYPE_Q4)
        elif split:
            self.basis_t = torch.zeros((pt, hkv, rank, d), dtype=torch.bfloat16, device=self.device)
            self.coeffs = torch.zeros((pt, hkv, P, rank), dtype=torch.bfloat16, device=self.device)
            self.summary = L.make_summary(self.basis_t, self.coeffs, rank, L.LOCKS_DTYPE_BF16)
        else:
            self.blocks = torch.zeros((pt, hkv, rank * d + P * rank), dtype=torch.bfloat16, device=self.device)
            self.basis_t = self.blocks[:, :, :rank * d].unflatten(-1, (rank, d))
            self.coeffs = self.blocks[:, :, rank * d:].unflatten(-1, (P, rank))
            self.summary = L.make_summary(self.blocks, None, rank, L.LOCKS_DTYPE_BF16_PACKED)
        self.cache = L.make_cache(k_pool, v_pool, block_table, seq_lens, self.n_summarized)
        flags = {"auto": 0, "unfused": L.LOCKS_FLAG_UNFUSED, "fused": L.LOCKS_FLAG_FUSED}[form]
        self.params = L.make_params(num_q_heads, budget_tokens, scale, flags)
        self.k_max = min(budget_tokens // P, block_table.shape[1])
        self.ws_bytes = L.locks_workspace_size(self.cache, self.summary, self.params)
        self.ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.ws.data_ptr()) % 256
        self.ws = self.ws[off:off + self.ws_bytes]
        L.locks_workspace_init(self.ws, self.ws_bytes)
        # the builder's own error word, so that builds may run on another
        # stream beside calls that use the main workspace
        self.build_ws = torch.zeros(512, dtype=torch.uint8, device=self.device)
        off = (-self.build_ws.data_ptr()) % 256
        self.build_ws = self.build_ws[off:off + 256]
        B = self.batch
        self.sel_pages = torch.zeros((B, hkv, max(self.k_max, 1)), dtype=torch.int32, device=self.device)
        self.sel_count = torch.zeros((B, hkv), dtype=torch.int32, device=self.device)
        self.out = torch.zeros((B, num_q_heads, d), dtype=torch.bfloat16, device=self.device)
        self.lse = torch.zeros((B, num_q_heads), dtype=torch.float32, device=self.device)

    def set_summaries(self, basis_t: torch.Tensor, coeffs: torch.Tensor | None):
        """Install externally computed summaries (same layouts; coeffs is
        None for the quantised format)."""
        self.basis_t.copy_(basis_t)
        if self.coeffs is not None:
            self.coeffs.copy_(coeffs)

    def build_summaries(self, page_ids: torch.Tensor, stream=None):
        ids = page_ids.to(device=self.device, dtype=torch.int32).contiguous()
        L.locks_build_summaries(self.cache, self.summary, ids, ids.numel(), self.build_ws, 256, stream)

    def select(self, q: torch.Tensor, page_lse: torch.Tensor | None = None, stream=None):
        L.locks_select(self.cache, self.summary, self.params, q, self.sel_pages, self.sel_count, page_lse,
                       self.ws, self.ws_bytes, stream)
        return self.sel_pages, self.sel_count

    def page_scores(self, q: torch.Tensor, page_lse: torch.Tensor, stream=None):
        L.locks_page_scores(self.cache, self.summary, self.params, q, page_lse, self.ws, self.ws_bytes, stream)
        return page_lse

    def sparse_attend(self, q: torch.Tensor, stream=None):
        L.locks_sparse_attend(self.cache, self.params, q, self.sel_pages, self.sel_count, self.out, self.lse,
                              self.ws, self.ws_bytes, stream)
        return self.out, self.lse

    def decode_step(self, q: torch.Tensor, out=None, lse=None, keep_selection: bool = True, stream=None):
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        sp, sc = (self.sel_pages, self.sel_count) if keep_selection else (None, None)
        L.locks_decode_step(self.cache, self.summary, self.params, q, out, lse, sp, sc, self.ws,
                            self.ws_bytes, stream)
        return out, lse

    def decode_step_launches(self) -> int:
        """Kernels one decode_step launches for this cache's shapes (2 or 3)."""
        return L.locks_decode_step_launches(self.cache, self.summary, self.params)

    def dense_decode(self, q: torch.Tensor, out=None, lse=None, stream=None):
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        L.locks_dense_decode(self.cache, self.params, q, out, lse, self.ws, self.ws_bytes, stream)
        return out, lse

    def exact_page_lse(self, q: torch.Tensor, stream=None) -> torch.Tensor:
        pl = torch.full((self.batch, self.num_q_heads, self.block_table.shape[1]), float("nan"),
                        dtype=torch.float32, device=self.device)
        L.locks_exact_page_lse(self.cache, self.params, q, pl, stream)
        return pl

    def device_error(self, stream=None) -> int:
        """LOCKS_DEVERR_* bits set since the last read, by the calls on the
        main workspace and by the builder (both words are cleared)."""
        return L.locks_get_device_error(self.ws, stream) | L.locks_get_device_error(self.build_ws, stream)
