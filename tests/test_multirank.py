"""The bench's multi-process host path on the CPU (gloo, world size 2).

The decode step of one layer is independent per (sequence, KV head), so
several GPUs run independent replicas and only the timing is combined: every
rank must end with the slowest rank's time, and the reference arm prints from
rank 0 only.  These tests run two gloo ranks as child processes; no GPU is
used.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        out[rank] = bench.max_over_ranks(values[rank], world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    values = [3.25, 7.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 7.5


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5


def test_reference_arm_prints_from_rank_zero_only(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        config, steps, warmup, gpus = "tiny", 1, 1, 2

    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
