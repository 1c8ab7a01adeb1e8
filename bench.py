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
    ("llama128k", 64): (50370048 + 4352) / 16384,
    ("ctx1m", 64): (100763904 + 2788608) / 32768,
}
# the same for the quantised summary format
SCAN_Q4_TRAFFIC_PER_PAGE_HEAD = {
    ("llama128k", 64): (20231936 + 0) / 16384,
    ("ctx1m", 64): (40477952 + 1024) / 32768,
}
SCAN_TRAFFIC_SOURCE_SHA = "3fab44a6cc64fe5a"


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
    """sha256 prefix of scan.cu's code: line comments and blank lines removed,
    so that editing a comment does not void the traffic figures."""
    code = []
    with open(os.path.join(ROOT, "sparse_kv_page_rank_gb300", "csrc", "scan.cu")) as f:
        for line in f:
            line = line.split("//", 1)[0].rstrip()
            if line:
                code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


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

def _oracle_inputs(case, cfg, kv_heads, max_pages: int | None = None):
    """One-sequence, one-KV-head slices of sequence 0 for the listed heads,
    optionally cut to the first ``max_pages`` pages, with the oracle's
    summaries precomputed (not timed).  Returns (problems, pages, pages_full)."""
    import oracle as O
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
    probs = []
    for h in kv_heads:
        kp = np.ascontiguousarray(case.k_pool[phys, h:h + 1])
        vp = np.ascontiguousarray(case.v_pool[phys, h:h + 1])
        basis = np.zeros((n_pages, 1, D, r))
        coeffs = np.zeros((n_pages, 1, P, r))
        for j in range(nfull):
            V, C, _, _ = O.page_summary(O.bf16_widen(kp[j, 0]), r)
            basis[j, 0], coeffs[j, 0] = V, C
        probs.append(dict(q=np.ascontiguousarray(case.q[b:b + 1, h * G:(h + 1) * G]), kp=kp, vp=vp, bt=bt,
                          seq=seq_sample, nfull=nfull, basis=basis, coeffs=coeffs,
                          budget=cfg["budget_tokens"], P=P))
    return probs, nfull, nfull_all


def _oracle_problem(prob) -> float:
    """Seconds the oracle takes for one (sequence, KV head) decode step."""
    import oracle as O
    t0 = time.perf_counter()
    O.decode_step(prob["q"], prob["kp"], prob["vp"], prob["bt"], prob["seq"], [prob["nfull"]], prob["basis"],
                  prob["coeffs"], 1, prob["budget"], page_size=prob["P"])
    return time.perf_counter() - t0


def _oracle_sample(case, cfg, kv_heads, budget_seconds: float, steps: int | None = None,
                   max_pages: int | None = None):
    """Time the oracle's decode step on one core, problem after problem
    (sequence 0, the listed KV heads, optionally its first ``max_pages``
    pages).  The time per (sequence, KV head) problem is scaled by the page
    ratio (the oracle's cost is linear in the pages it scans) and by the
    number of problems.  Returns (us per full step, detail)."""
    probs, nfull, nfull_all = _oracle_inputs(case, cfg, kv_heads, max_pages)
    times = []
    t_end = time.perf_counter() + budget_seconds
    i = 0
    while True:
        times.append(_oracle_problem(probs[i % len(probs)]))
        i += 1
        if steps is not None:
            if i >= steps:
                break
        elif time.perf_counter() > t_end and i >= len(probs):
            break
    per_problem = statistics.median(times) * (nfull_all / max(nfull, 1))
    full = per_problem * case.batch * case.num_kv_heads
    return full * 1e6, dict(problems_timed=i, per_problem_s=per_problem, times=times, pages=nfull,
                            pages_full=nfull_all)


def _oracle_pool():
    """A pool of os.cpu_count() spawned worker processes (spawned, not forked:
    safe after the CUDA context exists), warmed up so that timed work excludes
    interpreter start-up and imports."""
    import concurrent.futures as cf
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    ex = cf.ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn"))
    list(ex.map(_oracle_warm, range(cores)))
    return ex, cores


def _oracle_warm(_):
    import oracle  # noqa: F401
    return 0


def _oracle_all_cores(ex, cores, probs, nfull, nfull_all, problems_total, rounds: int = 1):
    """The oracle problems run on every host core at once (``rounds`` whole
    problems per core in the pool ``ex``): wall time scaled by pages and to
    ``problems_total`` problems.  Returns (us per full step, detail)."""
    work = [probs[i % len(probs)] for i in range(cores * rounds)]
    t0 = time.perf_counter()
    list(ex.map(_oracle_problem, work))
    wall = time.perf_counter() - t0
    per_problem_wall = wall / len(work) * (nfull_all / max(nfull, 1))
    return per_problem_wall * problems_total * 1e6, dict(problems=len(work), wall_s=wall, pages=nfull,
                                                          pages_full=nfull_all)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    case, cfg = make_config_case(args.config, page_size=args.page_size, **_rank_override(args))
    W, K = args.warmup, args.steps
    cores = os.cpu_count() or 1
    # each step: every host core runs one (sequence, KV head) problem of the
    # workload on a page window sized so that K + W steps take about two
    # minutes, scaled to a full step
    t0 = time.perf_counter()
    _, probe = _oracle_sample(case, cfg, [0], 0.0, steps=1, max_pages=256)
    per_page = probe["times"][0] / max(probe["pages"], 1)
    window = int(max(16, min(case.n_full_pages(0), 120.0 / (K + W) / max(per_page, 1e-9))))
    probs, nfull, nfull_all = _oracle_inputs(case, cfg, range(case.num_kv_heads), max_pages=window)
    ex, cores = _oracle_pool()
    total = case.batch * case.num_kv_heads
    for _ in range(W):
        _oracle_all_cores(ex, cores, probs, nfull, nfull_all, total)
    vals = [_oracle_all_cores(ex, cores, probs, nfull, nfull_all, total)[0] for _ in range(K)]
    ex.shutdown()
    us_full = statistics.median(vals)
    wall = time.perf_counter() - t0
    line = {
        "impl": "reference", "metric": METRIC, "value": us_full, "unit": "us", "n_gpus": args.gpus,
        "steps": K, "warmup": W, "ms_per_step": us_full / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config_dict(args.config, case, cfg),
        "cpu_baseline": {"value": us_full, "unit": "us", "cores": cores, "kind": "oracle",
                         "sample": f"each step = {cores} (sequence, KV head) problems of {args.config} at once, one "
                                   f"per host core, on the first {window} of {case.n_full_pages(0)} pages "
                                   f"(summaries precomputed), wall time scaled by pages and to "
                                   f"{case.batch * case.num_kv_heads} problems; median of {K} steps, {wall:.1f} s"},
        "e2e": {"value": us_full, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def _rank_override(args) -> dict:
    return {"rank": args.rank} if getattr(args, "rank", None) else {}


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

def _gpu_workload(args, name, K, W, world, dev, *, page_size=P, rank_override=None, full=True, q4=None):
    """Draw the named workload, build its summaries with the library's builder
    and time (each as one CUDA graph of K calls on R rotating cache copies):
    the decode step, the dense decode and the summary scan alone.  With
    ``full`` also the end-to-end forms; with ``q4`` (default: ``full``) the
    quantised format.  Returns a dict of measurements."""
    import torch

    from sparse_kv_page_rank_gb300.runtime import LocksRuntime

    overrides = {"rank": rank_override} if rank_override else {}
    case, cfg = make_config_case(name, page_size=page_size, **overrides)
    r, budget = cfg["rank"], cfg["budget_tokens"]
    B, Hq, Hkv, G = case.batch, case.num_q_heads, case.num_kv_heads, case.group
    Pg = case.page_size

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    k0, v0 = to_dev(case.k_pool), to_dev(case.v_pool)
    bt = torch.from_numpy(case.block_table).to(dev)
    sl = torch.from_numpy(case.seq_lens).to(dev)
    nsum_host = np.array([case.n_full_pages(b) for b in range(B)], dtype=np.int32)
    ns = torch.from_numpy(nsum_host).to(dev)
    q = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).to(dev)
    pages = torch.from_numpy(np.concatenate([case.block_table[b, :nsum_host[b]] for b in range(B)])).to(dev)
    carriers = case.carriers.copy()
    seq_lens = case.seq_lens.copy()
    config = _config_dict(name, case, cfg)
    del case

    per_copy = k0.numel() * 4 + (r * D + Pg * r) * 2 * k0.shape[0] * Hkv
    # bytes one step touches (summaries + selected pages); rotate enough copies
    # that consecutive replays of the same copy are > 4x L2 apart
    touched = Hkv * int(nsum_host.sum()) * summary_bytes_per_page_head(r, Pg) + \
        B * Hkv * min(budget // Pg, bt.shape[1]) * Pg * D * 4
    R = max(2, min(16, math.ceil(4 * 129e6 / max(touched, 1))))
    if args.copies:
        R = args.copies
    rts = []
    for i in range(R):
        kk = k0 if i == 0 else k0.clone()
        vv = v0 if i == 0 else v0.clone()
        rts.append(LocksRuntime(kk, vv, bt, sl, ns, Hq, r, budget))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    rts[0].build_summaries(pages)
    e1.record()
    torch.cuda.synchronize()
    build_ms = e0.elapsed_time(e1)
    for rt in rts[1:]:
        rt.set_summaries(rts[0].basis_t, rts[0].coeffs)
    torch.cuda.synchronize()
    assert rts[0].device_error() == 0

    stream = torch.cuda.Stream(device=dev)
    page_lse_bufs = [torch.empty((B, Hq, bt.shape[1]), dtype=torch.float32, device=dev) for _ in rts]

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
            import torch.distributed as dist
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
    res = dict(config=config, R=R, per_copy=per_copy, r=r, budget=budget, B=B, Hq=Hq, Hkv=Hkv, G=G, P=Pg,
               build_ms=build_ms, page_heads_built=int(pages.numel() * Hkv), launches=rts[0].decode_step_launches())
    if args.profile:
        # a few replays of the step, the dense decode and the scan, nothing else
        # (the command ncu captures)
        timed(step_fn, K, W)
        timed(dense_fn, K, W)
        timed(scan_fn, K, W)
        if r <= 8 and not args.no_q4:
            qrts = [LocksRuntime(rt_.k_pool, rt_.v_pool, bt, sl, ns, Hq, r, budget, quantized=True) for rt_ in rts]
            qrts[0].build_summaries(pages)
            for qrt in qrts[1:]:
                qrt.set_summaries(qrts[0].basis_t, None)
            timed(lambda i, rt_: qrts[i].decode_step(q, stream=stream), K, W)
            timed(lambda i, rt_: qrts[i].page_scores(q, page_lse_bufs[i], stream=stream), K, W)
        return res

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    step_ms = timed(step_fn, K, W, extra_replays=9)
    res["step_ms"] = step_ms
    res["step_pct"] = {f"p{p}": float(np.percentile(np.array([step_ms] + replay_ms) * 1e3, p)) for p in (10, 50, 90)}
    res["clocks"] = clocks.stop()
    res["dense_ms"] = timed(dense_fn, max(20, K // 4), W)
    res["scan_ms"] = timed(scan_fn, K, W)

    if full:
        # end to end through the public API, pinned host q in, pinned host out
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

        res["e2e_copy_ms"] = timed(e2e_fn, K, W)
        res["e2e_dev_ms"] = timed(e2e_zero_copy_fn, K, W)
        # one step as a caller sees it: replay a one-step graph, wait for the
        # stream, read the output on the host; host clock around each call.
        # Two forms: the kernels reading q from and writing out to page-locked
        # host memory, and cudaMemcpyAsync copies around the step.
        def host_clocked(fn, calls=300, skip=20):
            g1 = capture(fn, 1)
            host_us = []
            prev = torch.cuda.current_stream()
            torch.cuda.set_stream(stream)  # the graph replays on the current stream
            for _ in range(calls):
                t0 = time.perf_counter()
                g1.replay()
                stream.synchronize()
                _ = out_host[0, 0, 0].item()
                host_us.append((time.perf_counter() - t0) * 1e6)
            torch.cuda.set_stream(prev)
            del g1
            return {f"p{p}": float(np.percentile(np.array(host_us[skip:]), p)) for p in (10, 50, 90)}

        res["e2e_host_us"] = host_clocked(e2e_zero_copy_fn)
        res["e2e_host_memcpy_us"] = host_clocked(e2e_fn)
        res["io_bytes"] = (int(q.numel() * 2), int(B * Hq * D * 2))
    # every timed call must have finished without a device-side error
    # (a bounded wait that ran out, or a bad block-table entry)
    errs = [rt_.device_error() for rt_ in rts]
    if any(errs):
        raise SystemExit(f"device error bits {errs} after the timed steps of {name}: this run is invalid")

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
            for cpg in carriers[b, h]:
                if cpg >= 0:
                    total += 1
                    kept += int(cpg) in cs
    assert rt.device_error() == 0
    res.update(mass_recall=float(np.mean(recalls)), exact_lse_selection_recall=float(np.mean(oracle_recalls)),
               carrier_retention=kept / total if total else None)

    # The quantised, centred summary format (int4 basis, int8 coefficients and
    # centroid) on the same caches: its builder, step and scan.
    res["q4"] = None
    if (full if q4 is None else q4) and r <= 8 and not args.no_q4:
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
                qkept += sum(int(cpg) in cs for cpg in carriers[b, h] if cpg >= 0)
        qb = q4_page_head_bytes(r, Pg)
        q_scan_alg = Hkv * int(nsum_host.sum()) * (qb + G * 4)
        q_traffic = None
        if (name, Pg) in SCAN_Q4_TRAFFIC_PER_PAGE_HEAD and SCAN_TRAFFIC_SOURCE_SHA == _scan_source_sha():
            q_traffic = SCAN_Q4_TRAFFIC_PER_PAGE_HEAD[(name, Pg)] * Hkv * int(nsum_host.sum())
        res["q4"] = {"value": q4_step_ms * 1e3, "unit": "us", "summary_bytes_per_page_head": qb,
                     "residency": qb / (2 * Pg * D * 2), "speedup_vs_dense": res["dense_ms"] / q4_step_ms,
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
                        int(seq_lens[b]) - int(nsum_host[b]) * Pg, r, Pg)
        for key in sb:
            sb[key] += bb[key]
    res["step_bytes"] = sb
    res["dense_bytes"] = sum(dense_bytes(1, Hkv, G, int(seq_lens[b])) for b in range(B))
    res["scan_alg"] = Hkv * n_sum_tot * (summary_bytes_per_page_head(r, Pg) + G * 4)
    res["scan_traffic"] = None
    if (name, Pg) in SCAN_TRAFFIC_PER_PAGE_HEAD and SCAN_TRAFFIC_SOURCE_SHA == _scan_source_sha() and \
            r == CONFIGS[name]["rank"]:
        res["scan_traffic"] = SCAN_TRAFFIC_PER_PAGE_HEAD[(name, Pg)] * Hkv * n_sum_tot
    del rts
    torch.cuda.empty_cache()
    return res


def _roofline(res, peak, peak_kind):
    scan_gbs = res["scan_alg"] / (res["scan_ms"] * 1e-3) / 1e9
    return {"kernel": "scan_kernel (summary scan)", "bound": "hbm", "achieved": scan_gbs, "peak": peak,
            "unit": "GB/s", "frac": scan_gbs / peak, "traffic": res["scan_traffic"],
            "peak_kind": f"{peak_kind} (hbm_gbs, burst copy)", "scan_us": res["scan_ms"] * 1e3,
            "algorithmic_bytes": res["scan_alg"]}


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

    K, W = args.steps, max(3, args.warmup)
    res = _gpu_workload(args, args.config, K, W, world, dev, page_size=args.page_size, rank_override=args.rank)
    if args.profile:
        print(json.dumps({"profile": args.config, "copies": res["R"], "steps": K, "warmup": W}))
        return
    peak, peak_kind = _peaks()
    step_ms = res["step_ms"]
    sb = res["step_bytes"]
    eff_gbs = sb["total"] / (step_ms * 1e-3) / 1e9

    # the 1M-context workload beside the 128K headline (step, dense, scan)
    ctx1m = None
    if args.config == "llama128k" and args.page_size == P and not args.rank and not args.no_ctx1m:
        r1 = _gpu_workload(args, "ctx1m", K, W, world, dev, full=False, q4=True)
        e1 = r1["step_bytes"]["total"] / (r1["step_ms"] * 1e-3) / 1e9
        ctx1m = {"value": r1["step_ms"] * 1e3, "unit": "us", "config": r1["config"],
                 "step_us_over_replays": r1["step_pct"], "dense_us": r1["dense_ms"] * 1e3,
                 "speedup_vs_dense": r1["dense_ms"] / r1["step_ms"], "effective_gbs": e1,
                 "step_frac_of_hbm": e1 / peak, "step_bytes": r1["step_bytes"], "dense_bytes": r1["dense_bytes"],
                 "kv_bytes_ratio": r1["dense_bytes"] / r1["step_bytes"]["total"],
                 "mass_recall": r1["mass_recall"], "exact_lse_selection_recall": r1["exact_lse_selection_recall"],
                 "carrier_retention": r1["carrier_retention"], "roofline": _roofline(r1, peak, peak_kind),
                 "gpu_launches": r1["launches"] * K, "clocks": r1["clocks"], "q4": r1["q4"],
                 "timing": {"l2": f"rotating {r1['R']} independent copies of cache + summaries "
                                  f"({r1['R'] * r1['per_copy'] / 1e9:.2f} GB > 129 MB L2)"}}

    # the other named workloads at their stated shapes (step, dense, scan,
    # recall, clocks), and the growing-cache loop at its full 1024 steps
    workloads = None
    if args.config == "llama128k" and args.page_size == P and not args.rank and not args.no_workloads \
            and world == 1:
        workloads = {}
        for key, name, rk in (("sweep_r2", "sweep", 2), ("sweep_r4", "sweep", 4), ("sweep_r8", "sweep", 8),
                              ("tiny", "tiny", None), ("growing", "growing", None)):
            rw = _gpu_workload(args, name, K, W, world, dev, rank_override=rk, full=False, q4=False)
            ew = rw["step_bytes"]["total"] / (rw["step_ms"] * 1e-3) / 1e9
            workloads[key] = {
                "value": rw["step_ms"] * 1e3, "unit": "us", "config": rw["config"],
                "step_us_over_replays": rw["step_pct"], "dense_us": rw["dense_ms"] * 1e3,
                "speedup_vs_dense": rw["dense_ms"] / rw["step_ms"], "effective_gbs": ew, "step_frac_of_hbm": ew / peak,
                "kv_bytes_ratio": rw["dense_bytes"] / rw["step_bytes"]["total"], "residency": residency(rw["r"], rw["P"]),
                "mass_recall": rw["mass_recall"], "exact_lse_selection_recall": rw["exact_lse_selection_recall"],
                "carrier_retention": rw["carrier_retention"], "roofline": _roofline(rw, peak, peak_kind),
                "gpu_launches": rw["launches"] * K, "clocks": rw["clocks"]}
        workloads["growing_loop"] = _growing_loop(args, dev, 16)

    # batched throughput at 256K context on device-drawn page-local caches
    batched = None
    if args.config == "llama128k" and args.page_size == P and not args.rank and not args.no_batched and world == 1:
        batched = _batched_256k(args, dev, K, W, args.batches)

    # CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only), on
    # one core and on every host core
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        case2, cfg2 = make_config_case(args.config, page_size=args.page_size, **_rank_override(args))
        heads = range(min(res["Hkv"], 2))
        us_1, det = _oracle_sample(case2, cfg2, heads, args.cpu_seconds)
        probs, nfull, nfull_all = _oracle_inputs(case2, cfg2, range(res["Hkv"]), max_pages=256)
        ex, cores = _oracle_pool()
        us_all, det_all = _oracle_all_cores(ex, cores, probs, nfull, nfull_all, res["B"] * res["Hkv"], rounds=2)
        ex.shutdown()
        cpu = {"value": us_all, "unit": "us", "cores": cores, "kind": "oracle",
               "sample": f"fp64 numpy oracle decode step (summaries precomputed): {det_all['problems']} (sequence, "
                         f"KV head) problems of sequence 0, first {det_all['pages']} of {det_all['pages_full']} "
                         f"pages, on {cores} host cores at once ({det_all['wall_s']:.1f} s wall), scaled by pages "
                         f"and to {res['B'] * res['Hkv']} problems",
               "one_core": {"value": us_1, "unit": "us", "cores": 1,
                            "sample": f"KV heads 0-{min(res['Hkv'], 2) - 1} of sequence 0, {det['problems_timed']} "
                                      f"problems in ~{args.cpu_seconds:.0f} s, median per problem x "
                                      f"{res['B'] * res['Hkv']} problems"}}

    line = {
        "metric": METRIC, "value": step_ms * 1e3, "unit": "us", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": step_ms, "step_us_over_replays": res["step_pct"], "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": res["config"],
        "timing": {"l2": f"rotating {res['R']} independent copies of cache + summaries "
                         f"({res['R'] * res['per_copy'] / 1e9:.2f} GB > 129 MB L2)",
                   "graph": "one CUDA graph of K consecutive locks_decode_step calls (rotating copies)"},
        "effective_gbs": eff_gbs,
        "step_frac_of_hbm": eff_gbs / peak,
        "dense_us": res["dense_ms"] * 1e3, "dense_effective_gbs": res["dense_bytes"] / (res["dense_ms"] * 1e-3) / 1e9,
        "speedup_vs_dense": res["dense_ms"] / step_ms,
        "step_bytes": sb, "dense_bytes": res["dense_bytes"], "kv_bytes_ratio": res["dense_bytes"] / sb["total"],
        "residency": residency(res["r"], res["P"]), "mass_recall": res["mass_recall"],
        "exact_lse_selection_recall": res["exact_lse_selection_recall"],
        "carrier_retention": res["carrier_retention"],
        "summary_build": {"pages_per_s": res["page_heads_built"] / (res["build_ms"] / 1e3), "ms": res["build_ms"],
                          "page_heads": res["page_heads_built"]},
        "roofline": _roofline(res, peak, peak_kind),
        "cpu_baseline": cpu,
        "e2e": {"value": res["e2e_host_us"]["p50"], "unit": "us", "h2d_bytes_per_step": res["io_bytes"][0],
                "d2h_bytes_per_step": res["io_bytes"][1],
                "how": "one step as a caller sees it, median of 280 calls timed by the host clock: replay of a "
                       "one-step CUDA graph of locks_decode_step whose kernels read q from and write out to "
                       "page-locked host memory, stream synchronise, out read on the host",
                "host_clocked_us": res["e2e_host_us"],
                "host_clocked_memcpy_us": res["e2e_host_memcpy_us"],
                "host_clocked_memcpy_how": "the same with cudaMemcpyAsync of q (pinned host -> device) before and "
                                           "of out (device -> pinned host) after the step, inside the graph",
                "in_graph_us": res["e2e_dev_ms"] * 1e3,
                "in_graph_how": "per step inside one CUDA graph of K consecutive zero-copy steps (device clock): "
                                "the launch and host wait excluded",
                "in_graph_memcpy_us": res["e2e_copy_ms"] * 1e3},
        "q4": res["q4"],
        "ctx1m": ctx1m,
        "batched_256k": batched,
        "workloads": workloads,
        "gpu_launches": res["launches"] * K,
        "clocks": res["clocks"],
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_growing(args):
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from sparse_kv_page_rank_gb300.build_lib import build
    build()
    print(json.dumps(_growing_loop(args, dev, max(3, args.growing_segments))))


def _growing_loop(args, dev, segments) -> dict:
    """The growing-cache loop of the batch-32 8K workload (32 q / 8 KV heads,
    rank 4, budget 1024): each decode step appends one token to every
    sequence, and whenever the sequences' last pages fill, the builder
    summarises them on a side stream while the next 64 steps run
    (sparse_kv_page_rank_gb300.growing.GrowingLoop).  Reports the step time
    with the builder beside it and, over the same steps with the summaries
    already in place, without it; and the builder's in-loop page-heads per
    second against the rate at which pages fill."""
    import torch

    from sparse_kv_page_rank_gb300.growing import GrowingLoop
    from sparse_kv_page_rank_gb300.runtime import LocksRuntime

    start = 8192
    case, cfg = make_config_case("growing", context=start + P * segments)
    r, budget = cfg["rank"], cfg["budget_tokens"]
    B, Hq, Hkv = case.batch, case.num_q_heads, case.num_kv_heads

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    k, v = to_dev(case.k_pool), to_dev(case.v_pool)
    bt = torch.from_numpy(case.block_table).to(dev)
    q = to_dev(case.q)
    sl = torch.full((B,), start, dtype=torch.int32, device=dev)
    ns = torch.full((B,), start // P, dtype=torch.int32, device=dev)
    rt = LocksRuntime(k, v, bt, sl, ns, Hq, r, budget)
    rt.build_summaries(torch.from_numpy(np.concatenate([case.block_table[b, :start // P] for b in range(B)])).to(dev))
    config = _config_dict("growing", case, cfg, {
        "context": start, "context_end": start + P * segments,
        "loop": f"{segments} segments x {P} steps from {start} tokens: lengths advanced on the device inside "
                f"the segment graph; every {P} steps one page per sequence fills, is summarised on a side "
                f"stream beside the next segment, and joins the summarised pages one segment later"})
    del case
    loop = GrowingLoop(rt, q)
    loop.run(segments, build=True)  # warm-up; also leaves every filling page summarised once
    loop.reset()
    reps = 3
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    with_b, without_b = [], []
    for _ in range(reps):
        with_b.append(loop.run(segments, build=True))
        final_lens = rt.seq_lens.cpu().tolist()
        final_ns = rt.n_summarized.cpu().tolist()
        loop.reset()
        without_b.append(loop.run(segments, build=False))
        loop.reset()
    clk = clocks.stop()
    err = rt.device_error()
    if err:
        raise SystemExit(f"device error bits {err:#x} in the growing loop: this run is invalid")
    step_us = statistics.median(x["step_us"] for x in with_b)
    step_wo = statistics.median(x["step_us"] for x in without_b)
    builds = [m for x in with_b for m in x["build_ms"]]
    mean_build = float(np.mean(builds))
    ph_per_build = B * Hkv
    line = {
        "metric": "growing-cache decode step us with the summary builder beside it",
        "value": step_us, "unit": "us", "higher_is_better": False, "n_gpus": 1,
        "steps": segments * P, "warmup": segments * P, "repeats": reps, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "step_us_over_repeats": [x["step_us"] for x in with_b],
        "step_us_without_builder": step_wo,
        "builder_overhead_frac": step_us / step_wo - 1.0,
        "build_ms_per_fill": mean_build, "builds": len(builds),
        "builder_page_heads_per_s_in_loop": ph_per_build / (mean_build * 1e-3),
        "fill_rate_page_heads_per_s": ph_per_build / (step_us * P * 1e-6),
        "final_seq_len": final_lens[0], "final_n_summarized": final_ns[0],
        "gpu_launches": rt.decode_step_launches() * segments * P + (segments - 1),
        "timing": {"l2": "no flush: the loop's working set (summaries and selected pages of 32 sequences) "
                         "is what a serving loop re-reads step after step",
                   "graph": f"one CUDA graph per {P}-step segment; events on the main and side streams"},
        "clocks": clk,
    }
    del loop, rt, k, v
    torch.cuda.empty_cache()
    return line


def _batched_256k(args, dev, K, W, batches) -> dict:
    """Batched decode throughput at 256K context (32 query / 8 KV heads,
    rank 8, budget 2048 tokens): tokens per second of the sparse step against
    the in-library dense decode, per batch size.  The caches are page-local
    low-rank keys drawn on the device (synth.device_gen), summarised by the
    library's builder; recall is the selected pages' attention mass against
    the exact page LSE (locks_exact_page_lse, reading every key)."""
    import torch

    from sparse_kv_page_rank_gb300.runtime import LocksRuntime
    from synth.device_gen import make_device_cache

    ctx, Hq, Hkv, r, budget = 256 * 1024, 32, 8, 8, 2048
    G = Hq // Hkv
    peak, peak_kind = _peaks()
    stream = torch.cuda.Stream(device=dev)
    results = []
    for B in batches:
        c = make_device_cache(B, Hq, Hkv, ctx, true_rank=(8, 8), n_carriers=16, seed=1000 + B, device=dev)
        bt, q = c["block_table"], c["q"]
        rt = LocksRuntime(c["k_pool"], c["v_pool"], bt, c["seq_lens"], c["n_full"], Hq, r, budget)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        rt.build_summaries(bt.reshape(-1))
        e1.record()
        torch.cuda.synchronize()
        build_ms = e0.elapsed_time(e1)

        def per_call(fn, n, warm):
            gw, g = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                fn()
                with torch.cuda.graph(gw, stream=stream):
                    for _ in range(warm):
                        fn()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(n):
                        fn()
            torch.cuda.synchronize()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                gw.replay()
                s0.record(stream)
                g.replay()
                s1.record(stream)
            s1.synchronize()
            return s0.elapsed_time(s1) / n

        clocks = ClockSampler(dev.index if dev.index is not None else 0)
        clocks.start()
        time.sleep(0.3)
        step_ms = per_call(lambda: rt.decode_step(q, stream=stream), K, W)
        dense_ms = per_call(lambda: rt.dense_decode(q, rt.out, rt.lse, stream=stream), max(5, K // 20), 3)
        clk = clocks.stop()
        if rt.device_error():
            raise SystemExit(f"device error bits {rt.device_error():#x} at batch {B}: this run is invalid")

        # recall against the exact page LSE, and carrier retention (on the device)
        rt.decode_step(q)
        n = bt.shape[1]
        s = rt.exact_page_lse(q).double().view(B, Hkv, G, n)
        tot = torch.logsumexp(s, dim=-1)
        cnt = rt.sel_count.long()
        k = int(cnt.min())
        assert k == int(cnt.max()) == min(budget // P, n)
        sel = rt.sel_pages[..., :k].long()
        part = torch.logsumexp(s.gather(-1, sel[:, :, None, :].expand(B, Hkv, G, k)), dim=-1)
        recall = float(torch.exp(part - tot).mean())
        sig = torch.logsumexp(s - tot[..., None], dim=2)
        best = sig.topk(k, dim=-1).indices
        bpart = torch.logsumexp(s.gather(-1, best[:, :, None, :].expand(B, Hkv, G, k)), dim=-1)
        best_recall = float(torch.exp(bpart - tot).mean())
        car = c["carriers"].long()
        valid = car >= 0
        hit = (car[..., :, None] == sel[..., None, :]).any(-1) & valid
        retention = float(hit.sum()) / max(1, int(valid.sum()))
        sb = step_bytes(B, Hkv, G, n, k, 0, r)
        db = dense_bytes(B, Hkv, G, ctx)
        eff = sb["total"] / (step_ms * 1e-3) / 1e9
        results.append({
            "batch": B, "step_us": step_ms * 1e3, "dense_us": dense_ms * 1e3,
            "tokens_per_s": B / (step_ms * 1e-3), "dense_tokens_per_s": B / (dense_ms * 1e-3),
            "speedup_vs_dense": dense_ms / step_ms, "effective_gbs": eff, "step_frac_of_hbm": eff / peak,
            "step_bytes": sb["total"], "dense_bytes": db, "kv_bytes_ratio": db / sb["total"],
            "mass_recall": recall, "exact_lse_selection_recall": best_recall, "carrier_retention": retention,
            "summary_build": {"pages_per_s": B * n * Hkv / (build_ms * 1e-3), "ms": build_ms},
            "gpu_launches": rt.decode_step_launches() * K, "steps": K, "warmup": W, "clocks": clk})
        del rt, c, bt, q, s
        torch.cuda.empty_cache()
    return {"metric": "batched decode tokens/s at 256K context (one attention layer), sparse step vs dense",
            "unit": "tokens/s", "higher_is_better": True,
            "config": {"workload": "256K context, 32 q heads / 8 kv heads, head_dim 128, page 64, rank 8, "
                                   "budget 2048 tokens, bf16; page-local rank-8 keys with 16 carriers per "
                                   "(sequence, KV head), drawn on the device",
                       "batches": list(batches),
                       "l2": "no rotation: one step reads every summary (>= 805 MB at batch 8, 6x L2)"},
            "peak_kind": f"{peak_kind} (hbm_gbs)", "results": results}


def run_batch_sweep(args):
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from sparse_kv_page_rank_gb300.build_lib import build
    build()
    res = _batched_256k(args, dev, args.steps, max(3, args.warmup), args.batches)
    res["n_gpus"] = 1
    print(json.dumps(res))


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
    ap.add_argument("--growing-segments", type=int, default=16,
                    help="64-step segments in the growing loop (16: 1024 steps, 8192 -> 9216 tokens)")
    ap.add_argument("--batch-sweep", action="store_true", help="batched throughput at 256K context")
    ap.add_argument("--batches", type=int, nargs="+", default=[8, 32, 64])
    ap.add_argument("--rank", type=int, default=0, help="summary rank (0 = the workload's own)")
    ap.add_argument("--no-ctx1m", action="store_true", help="skip the 1M-context sub-measurement")
    ap.add_argument("--no-batched", action="store_true", help="skip the batched 256K sub-measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' sub-measurements (sweep, tiny, growing, growing loop)")
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
