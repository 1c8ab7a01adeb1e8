"""Benchmark of the LOCKS decode step on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config llama128k]
                    [--impl reference] [--no-cpu-baseline]

One step = the whole hot path on one batch: summary scan of every summarised
page, group-shared top-k selection, sparse attention over the selected pages
plus the tail (locks_decode_step), replayed from a CUDA graph.  Inputs are
seeded synthetic page-local low-rank caches shaped like the named workload;
summaries are built by the library's own GPU builder before timing.  L2 is
defeated by rotating R independent copies of the cache and summaries whose
total is several times the 129 MB L2.  Prints ONE JSON line.

The in-library dense paged decode is timed the same way for the speedup, the
summary-scan kernel alone for the roofline, and the fp64 CPU oracle on a
bounded sample for the CPU baseline (the only place, with --impl reference,
where this file runs the oracle).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import CONFIGS, make_config_case  # noqa: E402

METRIC = "decode-step µs & effective HBM GB/s (select+attend) at 128K/1M ctx vs dense"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
P, D = 64, 128

# DRAM traffic (bytes read + written) of one summary-scan launch per
# summarised page-head, keyed by (workload, page size), from ncu captures of
# the scan kernel at each workload; valid only while scan.cu is unchanged
# since those captures.
SCAN_TRAFFIC_PER_PAGE_HEAD = {
    ("llama128k", 64): (50365952 + 2816) / 16384,
    ("ctx1m", 64): (100761088 + 3253760) / 32768,
    ("llama128k", 16): (151064832 + 3976448) / 65536,
}
# the same for the quantised summary format
SCAN_Q4_TRAFFIC_PER_PAGE_HEAD = {
    ("llama128k", 64): (20229632 + 0) / 16384,
}
SCAN_TRAFFIC_SOURCE_SHA = "8ef72a34c0a70c64"


# ---------------------------------------------------------------------------
# byte model (algorithmic bytes; the pages' figures in tests/golden pin it)
# ---------------------------------------------------------------------------

def summary_bytes_per_page_head(rank: int, page: int = P, d: int = D, bytes_per=2) -> int:
    return (rank * d + page * rank) * bytes_per


def step_bytes(batch, hkv, G, n_sum, k, tail_tokens, rank, page: int = P) -> dict:
    """Algorithmic bytes of one decode step: every summary once, s_hat written
    and read once, K+V of the selected pages and the tail once, q and o."""
    summ = batch * hkv * n_sum * summary_bytes_per_page_head(rank, page)
    shat = 2 * batch * hkv * n_sum * G * 4
    sel = batch * hkv * (k * page + tail_tokens) * D * 2 * 2
    qo = 2 * batch * hkv * G * D * 2
    return dict(summaries=summ, shat=shat, selected_kv=sel, qo=qo, total=summ + shat + sel + qo)


def dense_bytes(batch, hkv, G, tokens) -> int:
    return batch * hkv * tokens * D * 2 * 2 + 2 * batch * hkv * G * D * 2


def residency(rank: int, page: int = P, d: int = D, basis_bits=16, coef_bits=16, centroid_bits=0) -> float:
    """Resident summary bytes as a fraction of the page's K+V bytes (bf16 cache)."""
    summ = (rank * d * basis_bits + page * rank * coef_bits + d * centroid_bits) / 8
    return summ / (2 * page * d * 2)


def max_over_ranks(value: float, world: int) -> float:
    """The largest of every rank's value (the job's time is its slowest
    replica's); the process group must be initialised when world > 1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _scan_source_sha() -> str:
    with open(os.path.join(ROOT, "sparse_kv_page_rank_gb300", "csrc", "scan.cu"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"locks_clocks_{os.getpid()}.csv")

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# reference arm / CPU baseline: the fp64 oracle on a bounded sample
# ---------------------------------------------------------------------------

def _oracle_sample(case, cfg, kv_heads, budget_seconds: float, steps: int | None = None,
                   max_pages: int | None = None):
    """Time the oracle's decode step (summaries precomputed, not timed) on a
    sample of KV heads of sequence 0, optionally cut to its first
    ``max_pages`` pages.  The time per (sequence, KV head) problem is scaled
    by the page ratio (the oracle's cost is linear in the pages it scans) and
    by the number of problems.  Returns (us per full step, detail)."""
    import oracle as O
    from synth.generator import LocksCase
    r = cfg["rank"]
    G = case.group
    P = case.page_size
    b = 0
    nfull_all = case.n_full_pages(b)
    nfull = nfull_all if max_pages is None else min(nfull_all, max_pages)
    seq_sample = np.array([nfull * P if nfull < nfull_all else int(case.seq_lens[b])], dtype=np.int32)
    n_pages = -(-int(seq_sample[0]) // P)
    phys = case.block_table[b, :n_pages]
    bt = np.arange(n_pages, dtype=np.int32)[None, :]
    subs = []
    for h in kv_heads:
        # one-sequence, one-KV-head slice of the cache on a compact pool, same bf16 inputs
        kp = np.ascontiguousarray(case.k_pool[phys, h:h + 1])
        vp = np.ascontiguousarray(case.v_pool[phys, h:h + 1])
        sub = LocksCase(batch=1, num_q_heads=G, num_kv_heads=1, head_dim=D, page_size=P,
                        seq_lens=seq_sample, block_table=bt, k_pool=kp, v_pool=vp,
                        q=case.q[b:b + 1, h * G:(h + 1) * G], carriers=case.carriers[b:b + 1, h:h + 1],
                        carrier_heads=case.carrier_heads[b:b + 1, h:h + 1],
                        outlier_channels=case.outlier_channels, seed=case.seed)
        basis = np.zeros((n_pages, 1, D, r))
        coeffs = np.zeros((n_pages, 1, P, r))
        for j in range(nfull):
            V, C, _, _ = O.page_summary(O.bf16_widen(kp[j, 0]), r)
            basis[j, 0], coeffs[j, 0] = V, C
        subs.append((sub, basis, coeffs))
    times = []
    t_end = time.perf_counter() + budget_seconds
    i = 0
    while True:
        sub, basis, coeffs = subs[i % len(subs)]
        t0 = time.perf_counter()
        O.decode_step(sub.q, sub.k_pool, sub.v_pool, sub.block_table, sub.seq_lens, [nfull], basis, coeffs,
                      1, cfg["budget_tokens"], page_size=P)
        times.append(time.perf_counter() - t0)
        i += 1
        if steps is not None:
            if i >= steps:
                break
        elif time.perf_counter() > t_end and i >= len(subs):
            break
    per_problem = statistics.median(times) * (nfull_all / max(nfull, 1))
    full = per_problem * case.batch * case.num_kv_heads
    return full * 1e6, dict(problems_timed=i, per_problem_s=per_problem, times=times, pages=nfull,
                            pages_full=nfull_all)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    case, cfg = make_config_case(args.config, page_size=args.page_size)
    W, K = args.warmup, args.steps
    # each step: one (sequence, KV head) problem of the workload on a page
    # window sized so that K + W steps take about two minutes, scaled to a full step
    t0 = time.perf_counter()
    _, probe = _oracle_sample(case, cfg, [0], 0.0, steps=1, max_pages=256)
    per_page = probe["times"][0] / max(probe["pages"], 1)
    window = int(max(16, min(case.n_full_pages(0), 120.0 / (K + W) / max(per_page, 1e-9))))
    _oracle_sample(case, cfg, [0], 0.0, steps=max(W, 1), max_pages=window)
    us_full, det = _oracle_sample(case, cfg, range(case.num_kv_heads), 0.0, steps=K, max_pages=window)
    wall = time.perf_counter() - t0
    line = {
        "impl": "reference", "metric": METRIC, "value": us_full, "unit": "us", "n_gpus": args.gpus,
        "steps": K, "warmup": W, "ms_per_step": us_full / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config_dict(args.config, case, cfg),
        "cpu_baseline": {"value": us_full, "unit": "us", "cores": 1, "kind": "oracle",
                         "sample": f"each step = one (sequence, KV head) problem of {args.config} on its first "
                                   f"{det['pages']} of {det['pages_full']} pages (summaries precomputed), "
                                   f"median scaled by pages and x {case.batch * case.num_kv_heads} problems; "
                                   f"{det['problems_timed']} steps, {wall:.1f} s"},
        "e2e": {"value": us_full, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def _config_dict(name, case, cfg, extra=None):
    d = {"workload": f"{name}: batch {case.batch}, {case.num_q_heads} q heads / {case.num_kv_heads} kv heads, "
                     f"head_dim {D}, page {case.page_size}, context {int(case.seq_lens[0])}, rank {cfg['rank']}, "
                     f"budget {cfg['budget_tokens']} tokens, bf16",
         "batch": case.batch, "num_q_heads": case.num_q_heads, "num_kv_heads": case.num_kv_heads,
         "context": int(case.seq_lens[0]), "page_size": case.page_size, "rank": cfg["rank"],
         "budget_tokens": cfg["budget_tokens"]}
    if extra:
        d.update(extra)
    return d


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from sparse_kv_page_rank_gb300.build_lib import build
    build()
    from sparse_kv_page_rank_gb300 import locks as L
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime

    case, cfg = make_config_case(args.config, page_size=args.page_size)
    r, budget = cfg["rank"], cfg["budget_tokens"]
    B, Hq, Hkv, G = case.batch, case.num_q_heads, case.num_kv_heads, case.group
    P = case.page_size

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    k0, v0 = to_dev(case.k_pool), to_dev(case.v_pool)
    bt = torch.from_numpy(case.block_table).to(dev)
    sl = torch.from_numpy(case.seq_lens).to(dev)
    nsum_host = np.array([case.n_full_pages(b) for b in range(B)], dtype=np.int32)
    ns = torch.from_numpy(nsum_host).to(dev)
    q = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).to(dev)
    pages = torch.from_numpy(np.concatenate([case.block_table[b, :nsum_host[b]] for b in range(B)])).to(dev)

    per_copy = k0.numel() * 4 + (r * D + P * r) * 2 * case.pages_total * Hkv
    # bytes one step touches (summaries + selected pages); rotate enough copies
    # that consecutive replays of the same copy are > 4x L2 apart
    touched = Hkv * int(nsum_host.sum()) * summary_bytes_per_page_head(r, P) + \
        B * Hkv * min(budget // P, case.max_pages) * P * D * 4
    R = max(2, min(16, math.ceil(4 * 129e6 / max(touched, 1))))
    if args.copies:
        R = args.copies
    rts = []
    for i in range(R):
        kk = k0 if i == 0 else k0.clone()
        vv = v0 if i == 0 else v0.clone()
        rt = LocksRuntime(kk, vv, bt, sl, ns, Hq, r, budget)
        rts.append(rt)
    del case.k_pool, case.v_pool
    # summaries by the library's builder (timed once, outside the step)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    rts[0].build_summaries(pages)
    e1.record()
    torch.cuda.synchronize()
    build_ms = e0.elapsed_time(e1)
    build_pages_per_s = pages.numel() * Hkv / (build_ms / 1e3)
    for rt in rts[1:]:
        rt.set_summaries(rts[0].basis_t, rts[0].coeffs)
    torch.cuda.synchronize()
    assert rts[0].device_error() == 0

    stream = torch.cuda.Stream(device=dev)
    page_lse_bufs = [torch.empty((B, Hq, case.max_pages), dtype=torch.float32, device=dev) for _ in rts]

    def capture(fn, nsteps):
        """One CUDA graph holding `nsteps` consecutive calls, step i on copy
        i mod R: the steps run back to back on the device (as the layers of a
        model would), kernels chained by programmatic dependent launch."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(min(R, nsteps)):
                fn(i % R, rts[i % R])
            with torch.cuda.graph(g, stream=stream):
                for i in range(nsteps):
                    fn(i % R, rts[i % R])
        torch.cuda.synchronize()
        return g

    replay_ms = []

    def timed(fn, K, W, extra_replays=0):
        """Device time per call over exactly K calls (one graph of K calls),
        after a graph of W warm-up calls.  extra_replays further replays of
        the same graph are timed one by one into replay_ms (for percentiles;
        the returned value is the first replay's)."""
        gw, gk = capture(fn, W), capture(fn, K)
        with torch.cuda.stream(stream):
            gw.replay()
        stream.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s0.record(stream)
            gk.replay()
            s1.record(stream)
        s1.synchronize()
        torch.cuda.synchronize()
        ms = max_over_ranks(s0.elapsed_time(s1), world)
        replay_ms.clear()
        for _ in range(extra_replays):
            with torch.cuda.stream(stream):
                s0.record(stream)
                gk.replay()
                s1.record(stream)
            s1.synchronize()
            replay_ms.append(max_over_ranks(s0.elapsed_time(s1), world) / K)
        del gw, gk
        return ms / K

    step_fn = lambda i, rt: rt.decode_step(q, stream=stream)  # noqa: E731
    dense_fn = lambda i, rt: rt.dense_decode(q, rt.out, rt.lse, stream=stream)  # noqa: E731
    scan_fn = lambda i, rt: rt.page_scores(q, page_lse_bufs[i], stream=stream)  # noqa: E731

    K, W = args.steps, max(3, args.warmup)
    if args.profile:
        # a few replays of the step and of the dense decode, nothing else
        # (the command ncu captures)
        timed(step_fn, K, W)
        timed(dense_fn, K, W)
        timed(scan_fn, K, W)
        if r <= 8 and not args.no_q4:
            # the quantised format's step and scan, after the bf16 ones
            qrts = [LocksRuntime(rt_.k_pool, rt_.v_pool, bt, sl, ns, Hq, r, budget, quantized=True) for rt_ in rts]
            qrts[0].build_summaries(pages)
            for qrt in qrts[1:]:
                qrt.set_summaries(qrts[0].basis_t, None)
            timed(lambda i, rt_: qrts[i].decode_step(q, stream=stream), K, W)
            timed(lambda i, rt_: qrts[i].page_scores(q, page_lse_bufs[i], stream=stream), K, W)
        print(json.dumps({"profile": args.config, "copies": R, "steps": K, "warmup": W}))
        return
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    step_ms = timed(step_fn, K, W, extra_replays=9)
    step_pct = {f"p{p}": float(np.percentile(np.array([step_ms] + replay_ms) * 1e3, p)) for p in (10, 50, 90)}
    clk = clocks.stop()
    dense_ms = timed(dense_fn, max(20, K // 4), W)
    scan_ms = timed(scan_fn, K, W)

    # e2e through the public API: pinned host q -> device, decode step, out -> pinned host
    q_host = q.cpu().pin_memory()
    out_host = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    q_dev = torch.empty_like(q)

    def e2e_zero_copy_fn(i, rt):
        # the kernels read q from, and write out to, page-locked host memory
        rt.decode_step(q_host, out=out_host, stream=stream)

    def e2e_fn(i, rt):
        q_dev.copy_(q_host, non_blocking=True)
        rt.decode_step(q_dev, stream=stream)
        out_host.copy_(rt.out, non_blocking=True)

    e2e_ms_copy = timed(e2e_fn, K, W)
    e2e_ms_dev = timed(e2e_zero_copy_fn, K, W)
    # every timed call must have finished without a device-side error
    # (a bounded wait that ran out, or a bad block-table entry)
    errs = [rt_.device_error() for rt_ in rts]
    if any(errs):
        raise SystemExit(f"device error bits {errs} after the timed steps: this run is invalid")

    # quality: mass recall of the selected pages against the exact page LSE
    # (read-every-key, on the GPU), and carrier retention
    rt = rts[0]
    rt.decode_step(q)
    exact = rt.exact_page_lse(q)
    torch.cuda.synchronize()
    sel = rt.sel_pages.cpu().numpy()
    cnt = rt.sel_count.cpu().numpy()
    ex = exact.double().cpu().numpy()
    recalls, oracle_recalls, kept, total = [], [], 0, 0
    for b in range(B):
        n = int(nsum_host[b])
        for h in range(Hkv):
            k = int(cnt[b, h])
            s_star = ex[b, h * G:(h + 1) * G, :n]
            tot = np.logaddexp.reduce(s_star, axis=1)
            chosen = sel[b, h, :cnt[b, h]]
            part = np.logaddexp.reduce(s_star[:, chosen], axis=1)
            recalls.append(float(np.mean(np.exp(part - tot))))
            # exact-LSE selection (same GSA rule on s*): best achievable recall
            z = s_star - tot[:, None]
            sig = np.logaddexp.reduce(z, axis=0)
            best = np.lexsort((np.arange(n), -sig))[:k]
            oracle_recalls.append(float(np.mean(np.exp(np.logaddexp.reduce(s_star[:, best], axis=1) - tot))))
            cs = set(chosen.tolist())
            for cpg in case.carriers[b, h]:
                if cpg >= 0:
                    total += 1
                    kept += int(cpg) in cs
    assert rt.device_error() == 0

    # The quantised, centred summary format (int4 basis, int8 coefficients and
    # centroid) on the same caches: its builder, step and scan.
    q4 = None
    if r <= 8 and not args.no_q4:
        from sparse_kv_page_rank_gb300.locks import q4_page_head_bytes
        qrts = [LocksRuntime(rt_.k_pool, rt_.v_pool, bt, sl, ns, Hq, r, budget, quantized=True) for rt_ in rts]
        torch.cuda.synchronize()
        e0.record()
        qrts[0].build_summaries(pages)
        e1.record()
        torch.cuda.synchronize()
        q4_build_ms = e0.elapsed_time(e1)
        for qrt in qrts[1:]:
            qrt.set_summaries(qrts[0].basis_t, None)
        q4_step_ms = timed(lambda i, rt_: qrts[i].decode_step(q, stream=stream), K, W)
        q4_scan_ms = timed(lambda i, rt_: qrts[i].page_scores(q, page_lse_bufs[i], stream=stream), K, W)
        qerrs = [qrt.device_error() for qrt in qrts]
        if any(qerrs):
            raise SystemExit(f"device error bits {qerrs} after the quantised-format steps: this run is invalid")
        qrts[0].decode_step(q)
        torch.cuda.synchronize()
        qsel = qrts[0].sel_pages.cpu().numpy()
        qcnt = qrts[0].sel_count.cpu().numpy()
        qrec, qkept = [], 0
        for b in range(B):
            n = int(nsum_host[b])
            for h in range(Hkv):
                s_star = ex[b, h * G:(h + 1) * G, :n]
                tot = np.logaddexp.reduce(s_star, axis=1)
                chosen = qsel[b, h, :qcnt[b, h]]
                qrec.append(float(np.mean(np.exp(np.logaddexp.reduce(s_star[:, chosen], axis=1) - tot))))
                cs = set(chosen.tolist())
                qkept += sum(int(cpg) in cs for cpg in case.carriers[b, h] if cpg >= 0)
        qb = q4_page_head_bytes(r, P)
        q_scan_alg = Hkv * int(nsum_host.sum()) * (qb + G * 4)
        q_traffic = None
        if (args.config, P) in SCAN_Q4_TRAFFIC_PER_PAGE_HEAD and SCAN_TRAFFIC_SOURCE_SHA == _scan_source_sha():
            q_traffic = SCAN_Q4_TRAFFIC_PER_PAGE_HEAD[(args.config, P)] * Hkv * int(nsum_host.sum())
        q4 = {"value": q4_step_ms * 1e3, "unit": "us", "summary_bytes_per_page_head": qb,
              "residency": qb / (2 * P * D * 2), "speedup_vs_dense": dense_ms / q4_step_ms,
              "scan_us": q4_scan_ms * 1e3, "scan_gbs": q_scan_alg / (q4_scan_ms * 1e-3) / 1e9,
              "scan_algorithmic_bytes": q_scan_alg, "scan_traffic": q_traffic,
              "mass_recall": float(np.mean(qrec)), "carrier_retention": qkept / total if total else None,
              "summary_build": {"pages_per_s": pages.numel() * Hkv / (q4_build_ms / 1e3), "ms": q4_build_ms},
              "format": "centred; int4 basis, int8 coefficients and centroid, float32 scales per vector"}
        del qrts

    n_sum_tot = int(nsum_host.sum())
    sb = dict(summaries=0, shat=0, selected_kv=0, qo=0, total=0)
    for b in range(B):
        bb = step_bytes(1, Hkv, G, int(nsum_host[b]), int(cnt[b].mean()),
                        int(case.seq_lens[b]) - int(nsum_host[b]) * P, r, P)
        for key in sb:
            sb[key] += bb[key]
    db = sum(dense_bytes(1, Hkv, G, int(case.seq_lens[b])) for b in range(B))
    scan_alg = Hkv * n_sum_tot * (summary_bytes_per_page_head(r, P) + G * 4)
    peak, peak_kind = _peaks()
    step_us = step_ms * 1e3
    eff_gbs = sb["total"] / (step_ms * 1e-3) / 1e9
    scan_gbs = scan_alg / (scan_ms * 1e-3) / 1e9
    dense_gbs = db / (dense_ms * 1e-3) / 1e9
    traffic = None
    if (args.config, P) in SCAN_TRAFFIC_PER_PAGE_HEAD and SCAN_TRAFFIC_SOURCE_SHA == _scan_source_sha():
        traffic = SCAN_TRAFFIC_PER_PAGE_HEAD[(args.config, P)] * Hkv * n_sum_tot

    # CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from synth import make_config_case as mk
        case2, cfg2 = mk(args.config, page_size=P)
        us_full, det = _oracle_sample(case2, cfg2, range(min(Hkv, 2)), args.cpu_seconds)
        cpu = {"value": us_full, "unit": "us", "cores": 1, "kind": "oracle",
               "sample": f"fp64 numpy oracle decode step (summaries precomputed) on KV heads 0-"
                         f"{min(Hkv, 2) - 1} of sequence 0, {det['problems_timed']} problems in "
                         f"~{args.cpu_seconds:.0f} s, median per problem x {B * Hkv} problems"}

    line = {
        "metric": METRIC, "value": step_us, "unit": "us", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": step_ms, "step_us_over_replays": step_pct, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": _config_dict(args.config, case, cfg, {
            "l2": f"rotating {R} independent copies of cache + summaries "
                  f"({R * per_copy / 1e9:.2f} GB > 129 MB L2)",
            "graph": "one CUDA graph of K consecutive locks_decode_step calls (rotating copies)"}),
        "effective_gbs": eff_gbs,
        "step_frac_of_hbm": eff_gbs / peak,
        "dense_us": dense_ms * 1e3, "dense_effective_gbs": dense_gbs, "speedup_vs_dense": dense_ms / step_ms,
        "step_bytes": sb, "dense_bytes": db, "kv_bytes_ratio": db / sb["total"],
        "residency": residency(r, P), "mass_recall": float(np.mean(recalls)),
        "exact_lse_selection_recall": float(np.mean(oracle_recalls)),
        "carrier_retention": kept / total if total else None,
        "summary_build": {"pages_per_s": build_pages_per_s, "ms": build_ms, "page_heads": int(pages.numel() * Hkv)},
        "roofline": {"kernel": "scan_kernel (summary scan)", "bound": "hbm", "achieved": scan_gbs,
                     "peak": peak, "unit": "GB/s", "frac": scan_gbs / peak, "traffic": traffic,
                     "peak_kind": f"{peak_kind} (hbm_gbs, burst copy)", "scan_us": scan_ms * 1e3,
                     "algorithmic_bytes": scan_alg},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_ms_dev * 1e3, "unit": "us", "h2d_bytes_per_step": int(q.numel() * 2),
                "d2h_bytes_per_step": int(B * Hq * D * 2),
                "how": "per step inside one CUDA graph: locks_decode_step reads q from and writes out to "
                       "page-locked host memory in place (the kernels move the data over the CPU-GPU link)",
                "memcpy_value": e2e_ms_copy * 1e3,
                "memcpy_how": "the same with cudaMemcpyAsync of q (pinned host -> device) before and of out "
                              "(device -> pinned host) after each step"},
        "q4": q4,
        "gpu_launches": rts[0].decode_step_launches() * K,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_growing(args):
    """The growing-cache loop of the batch-32 8K workload: each decode step
    appends one token to every sequence (lengths are advanced on the device,
    inside the graph), and whenever the sequences' last pages fill, the
    builder summarises them on a side stream while the next 64 steps run; the
    summarised-page counts advance once the build is done.  Reports the step
    time with and without the builder running beside it, and the builder's
    in-loop page-heads per second against the fill rate."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from sparse_kv_page_rank_gb300.build_lib import build
    build()
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime

    segments = max(2, args.growing_segments)
    start = 8192
    case, cfg = make_config_case("growing", context=start + P * segments)
    r, budget = cfg["rank"], cfg["budget_tokens"]
    B, Hq, Hkv = case.batch, case.num_q_heads, case.num_kv_heads

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    k, v = to_dev(case.k_pool), to_dev(case.v_pool)
    bt = torch.from_numpy(case.block_table).to(dev)
    q = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).to(dev)
    runs = {}
    for overlap in (False, True):
        sl = torch.full((B,), start, dtype=torch.int32, device=dev)
        ns = torch.full((B,), start // P, dtype=torch.int32, device=dev)
        rt = LocksRuntime(k, v, bt, sl, ns, Hq, r, budget)
        first = torch.from_numpy(np.concatenate([case.block_table[b, :start // P] for b in range(B)])).to(dev)
        rt.build_summaries(first)
        main, side = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        one = torch.ones((B,), dtype=torch.int32, device=dev)

        def segment():
            for _ in range(P):
                sl.add_(one)
                rt.decode_step(q, stream=main)

        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(main):
            segment()  # warm-up (advances the lengths; reset below)
            with torch.cuda.graph(g, stream=main):
                segment()
        torch.cuda.synchronize()
        sl.fill_(start)
        assert rt.device_error() == 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        seg_done = [torch.cuda.Event() for _ in range(segments)]
        built = [torch.cuda.Event() for _ in range(segments)]
        build_ms = []
        # the physical pages that fill at the end of each segment
        fill_ids = [bt[:, start // P + si].contiguous() for si in range(segments)]
        torch.cuda.synchronize()
        with torch.cuda.stream(main):
            e0.record(main)
            for si in range(segments):
                if overlap and si >= 2:
                    # the page filled two segments ago is summarised by now
                    main.wait_event(built[si - 2])
                    ns.add_(one)
                g.replay()
                seg_done[si].record(main)
                if overlap and si + 1 < segments:
                    # the page that just filled: build it beside the next segment
                    ids = fill_ids[si]
                    side.wait_event(seg_done[si])
                    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    b0.record(side)
                    rt.build_summaries(ids, stream=side)
                    b1.record(side)
                    built[si].record(side)
                    build_ms.append((b0, b1))
            e1.record(main)
        torch.cuda.synchronize()
        assert rt.device_error() == 0
        total_ms = e0.elapsed_time(e1)
        bms = [a.elapsed_time(b) for a, b in build_ms]
        runs[overlap] = dict(step_us=total_ms * 1e3 / (segments * P), build_ms=bms,
                             final_n_summarized=int(ns[0].item()), final_seq_len=int(sl[0].item()))
    ph_per_build = B * Hkv
    fill_rate = ph_per_build / (runs[True]["step_us"] * P * 1e-6)  # page-heads filled per second
    mean_build = float(np.mean(runs[True]["build_ms"])) if runs[True]["build_ms"] else None
    line = {
        "metric": "growing-cache decode step us with the summary builder beside it",
        "value": runs[True]["step_us"], "unit": "us", "higher_is_better": False, "n_gpus": 1,
        "config": _config_dict("growing", case, cfg, {
            "loop": f"{segments} x 64 steps from {start} tokens; lengths advanced on the device; "
                    f"one page per sequence fills every 64 steps"}),
        "step_us_without_builder": runs[False]["step_us"],
        "builder_overhead_frac": runs[True]["step_us"] / runs[False]["step_us"] - 1.0,
        "build_ms_per_fill": mean_build,
        "builder_page_heads_per_s_in_loop": ph_per_build / (mean_build * 1e-3) if mean_build else None,
        "fill_rate_page_heads_per_s": fill_rate,
        "final_n_summarized": runs[True]["final_n_summarized"], "final_seq_len": runs[True]["final_seq_len"],
    }
    print(json.dumps(line))


def run_batch_sweep(args):
    """Batched decode throughput at 256K context (32 query / 8 KV heads, r = 8,
    budget 2048): tokens per second of the sparse step against the in-library
    dense decode at several batch sizes.  The caches are drawn on the device
    (seeded normal keys and values, a random permutation as block table) and
    summarised by the builder; recall is not measured here, only time."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from sparse_kv_page_rank_gb300.build_lib import build
    build()
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime

    ctx, Hq, Hkv, r, budget = 256 * 1024, 32, 8, 8, 2048
    npg = ctx // P
    gen = torch.Generator(device=dev)
    results = []
    for B in args.batches:
        gen.manual_seed(1000 + B)
        pt = B * npg
        k = torch.empty((pt, Hkv, P, D), dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        for lo in range(0, pt, 4096):
            hi = min(pt, lo + 4096)
            k[lo:hi].normal_(generator=gen)
            v[lo:hi].normal_(generator=gen)
        bt = torch.randperm(pt, generator=gen, device=dev).to(torch.int32).view(B, npg)
        sl = torch.full((B,), ctx, dtype=torch.int32, device=dev)
        ns = torch.full((B,), npg, dtype=torch.int32, device=dev)
        q = torch.randn((B, Hq, D), generator=gen, device=dev).to(torch.bfloat16)
        rt = LocksRuntime(k, v, bt, sl, ns, Hq, r, budget)
        rt.build_summaries(bt.reshape(-1))
        torch.cuda.synchronize()
        stream = torch.cuda.Stream(device=dev)

        def per_call(fn, K):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                fn()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(K):
                        fn()
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                g.replay()  # warm-up replay
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1) / K

        step_ms = per_call(lambda: rt.decode_step(q, stream=stream), 20)
        dense_ms = per_call(lambda: rt.dense_decode(q, rt.out, rt.lse, stream=stream), 5)
        assert rt.device_error() == 0
        results.append({"batch": B, "step_us": step_ms * 1e3, "dense_us": dense_ms * 1e3,
                        "tokens_per_s": B / (step_ms * 1e-3), "dense_tokens_per_s": B / (dense_ms * 1e-3),
                        "speedup": dense_ms / step_ms})
        del rt, k, v, bt, q
        torch.cuda.empty_cache()
    print(json.dumps({"metric": "batched decode tokens/s at 256K context (one attention layer), sparse vs dense",
                      "unit": "tokens/s", "higher_is_better": True, "n_gpus": 1,
                      "config": {"workload": "256K context, 32 q heads / 8 kv heads, head_dim 128, page 64, rank 8, "
                                             "budget 2048 tokens, bf16; keys and values drawn on the device",
                                 "batches": list(args.batches)},
                      "results": results}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="llama128k", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="locks", choices=["locks", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--copies", type=int, default=0, help="independent cache copies to rotate (0 = auto)")
    ap.add_argument("--profile", action="store_true", help="only replay the step, dense and scan graphs")
    ap.add_argument("--no-q4", action="store_true", help="skip the quantised summary format's measurements")
    ap.add_argument("--page-size", type=int, default=64, choices=[64, 16],
                    help="tokens per page (16: the page size the explainer quotes its summary size at)")
    ap.add_argument("--growing-loop", action="store_true",
                    help="the batch-32 growing-cache loop with the builder on a side stream")
    ap.add_argument("--growing-segments", type=int, default=6, help="64-step segments in the growing loop")
    ap.add_argument("--batch-sweep", action="store_true", help="batched throughput at 256K context")
    ap.add_argument("--batches", type=int, nargs="+", default=[8, 32, 64])
    args = ap.parse_args()
    if args.batch_sweep:
        run_batch_sweep(args)
    elif args.growing_loop:
        run_growing(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
