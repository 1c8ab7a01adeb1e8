"""The growing-cache decode loop: every decode step appends one token to every
sequence, and pages that fill are summarised by the builder on a second
stream while later steps run.

Summaries are made when a page is finalised and kept off the decode step's
critical path (LOCKS explainer, §2 "Implementatie"; the summary of a page
depends only on that page's keys, so each one is built once).  Until its
summary exists a full page is part of the open tail and is attended in full,
so the step's result is defined at every point of the loop.

``GrowingLoop`` holds the streams, the captured segment graph and the events;
every kernel it runs is one of liblocks.so's (decode step, builder) apart from
torch's few per-segment updates of the length table and counts.
"""

from __future__ import annotations

import torch

from . import locks as L
from .runtime import LocksRuntime


class GrowingLoop:
    """Decode steps over caches that grow by one token per sequence per step.

    ``rt``'s seq_lens and n_summarized give the start: every sequence must
    start on a page boundary with all its full pages summarised (n_summarized
    == seq_lens // P).  One segment is P steps, captured once as a CUDA graph
    on ``main``: step i reads its lengths from row i of a device table
    [P][B] (through its own cache struct), so the P decode steps run back to
    back with nothing between them; after each segment the table advances by
    P and rt.seq_lens takes the segment's last row.  At the end of segment s every sequence's
    last page is full; when ``build`` is set the builder summarises those B
    pages on ``side`` beside segment s + 1, and n_summarized advances by one
    on ``main`` after an event wait on that build, before segment s + 2.  So
    no step reads a summary while it is being written, and the main stream
    waits for the builder only if one build outlasts a whole segment.

    ``snapshot_step``: when set (0 <= step < P), the segment graph also copies
    that step's output, lse, selection and lengths aside, and ``run`` keeps
    one copy per segment (``snapshots``); for checking, not for timing.
    """

    def __init__(self, rt: LocksRuntime, q: torch.Tensor, snapshot_step: int | None = None):
        self.rt, self.q = rt, q
        self.P = rt.k_pool.shape[2]
        dev = rt.device
        self.main = torch.cuda.Stream(device=dev)
        self.side = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize(dev)
        lens = rt.seq_lens.cpu()
        nsum = rt.n_summarized.cpu()
        if bool((lens % self.P != 0).any()) or not torch.equal(nsum, lens // self.P):
            raise ValueError("every sequence must start on a page boundary with its full pages summarised")
        self.start_lens = rt.seq_lens.clone()
        self.start_nsum = rt.n_summarized.clone()
        self.start_pages = (lens // self.P).to(dev)
        self.room = int(rt.block_table.shape[1] - int((lens // self.P).max()))
        self._one = torch.ones_like(rt.seq_lens)
        steps = torch.arange(1, self.P + 1, dtype=torch.int32, device=dev)[:, None]
        self._table0 = (rt.seq_lens[None, :] + steps).contiguous()
        self.lens_table = self._table0.clone()
        self.caches = [L.make_cache(rt.k_pool, rt.v_pool, rt.block_table, self.lens_table[i], rt.n_summarized)
                       for i in range(self.P)]
        self.snapshot_step = snapshot_step
        if snapshot_step is not None:
            if not 0 <= snapshot_step < self.P:
                raise ValueError("snapshot_step must lie in [0, page_size)")
            self._stage = self._snapshot_buffers(1)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.main):
            self._segment()  # warm-up
            with torch.cuda.graph(self.graph, stream=self.main):
                self._segment()
        torch.cuda.synchronize(dev)
        self.reset()
        if rt.device_error() != 0:
            raise RuntimeError(f"device error word {rt.device_error():#x} after the warm-up segment")
        self.snapshots = None

    def _snapshot_buffers(self, n: int) -> dict:
        rt = self.rt
        return {"out": torch.empty((n,) + tuple(rt.out.shape), dtype=rt.out.dtype, device=rt.device),
                "lse": torch.empty((n,) + tuple(rt.lse.shape), dtype=rt.lse.dtype, device=rt.device),
                "sel_pages": torch.empty((n,) + tuple(rt.sel_pages.shape), dtype=torch.int32, device=rt.device),
                "sel_count": torch.empty((n,) + tuple(rt.sel_count.shape), dtype=torch.int32, device=rt.device),
                "seq_lens": torch.empty((n,) + tuple(rt.seq_lens.shape), dtype=torch.int32, device=rt.device),
                "n_summarized": torch.empty((n,) + tuple(rt.n_summarized.shape), dtype=torch.int32,
                                            device=rt.device)}

    def _segment(self):
        rt = self.rt
        for i in range(self.P):
            L.locks_decode_step(self.caches[i], rt.summary, rt.params, self.q, rt.out, rt.lse, rt.sel_pages,
                                rt.sel_count, rt.ws, rt.ws_bytes, self.main)
            if self.snapshot_step == i:
                for name, src in (("out", rt.out), ("lse", rt.lse), ("sel_pages", rt.sel_pages),
                                  ("sel_count", rt.sel_count), ("seq_lens", self.lens_table[i]),
                                  ("n_summarized", rt.n_summarized)):
                    self._stage[name][0].copy_(src)

    def reset(self):
        """Put the lengths and summarised-page counts back to the start."""
        with torch.cuda.stream(self.main):
            self.rt.seq_lens.copy_(self.start_lens)
            self.rt.n_summarized.copy_(self.start_nsum)
            self.lens_table.copy_(self._table0)
        torch.cuda.synchronize(self.rt.device)

    def fill_pages(self, segments: int) -> torch.Tensor:
        """int32 [segments][B]: the physical page of each sequence that fills
        at the end of each segment."""
        if segments > self.room:
            raise ValueError(f"{segments} segments need more block-table columns than the {self.room} left")
        cols = self.start_pages[:, None] + torch.arange(segments, device=self.rt.device, dtype=torch.int32)[None, :]
        return self.rt.block_table.gather(1, cols.long()).t().contiguous()

    def run(self, segments: int, build: bool = True) -> dict:
        """Replays ``segments`` segments from the current state.  With
        ``build`` false the summarised-page counts advance at the same points
        but nothing is built (the summaries must already be in place), which
        times the same steps without the builder beside them.  Returns the
        mean step time and each build's duration on the side stream."""
        rt, main, side = self.rt, self.main, self.side
        fill = self.fill_pages(segments)
        if bool((fill < 0).any()) or bool((fill >= rt.k_pool.shape[0]).any()):
            raise ValueError("a page that fills during the loop has no physical page in the block table")
        if self.snapshot_step is not None:
            self.snapshots = self._snapshot_buffers(segments)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        seg_done = [torch.cuda.Event() for _ in range(segments)]
        built = [torch.cuda.Event() for _ in range(segments)]
        build_events = []
        torch.cuda.synchronize(rt.device)
        with torch.cuda.stream(main):
            e0.record(main)
            for s in range(segments):
                if s >= 2:
                    if build:
                        main.wait_event(built[s - 2])
                    rt.n_summarized.add_(self._one)
                self.graph.replay()
                seg_done[s].record(main)
                rt.seq_lens.copy_(self.lens_table[-1])
                self.lens_table.add_(self.P)
                if self.snapshot_step is not None:
                    for name, buf in self.snapshots.items():
                        buf[s].copy_(self._stage[name][0])
                if build and s + 1 < segments:
                    side.wait_event(seg_done[s])
                    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    b0.record(side)
                    rt.build_summaries(fill[s], stream=side)
                    b1.record(side)
                    built[s].record(side)
                    build_events.append((b0, b1))
            e1.record(main)
        torch.cuda.synchronize(rt.device)
        total_ms = e0.elapsed_time(e1)
        return {"step_us": total_ms * 1e3 / (segments * self.P),
                "build_ms": [a.elapsed_time(b) for a, b in build_events]}
