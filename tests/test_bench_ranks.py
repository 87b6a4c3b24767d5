"""Multi-rank host logic of bench.py on CPU: two gloo ranks with different step times must
both report the slowest rank's time, and the whole-job value counts every rank's bytes."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.5, 4.0][rank]
        slowest = bench.max_over_ranks(ms)
        out.put((rank, slowest, bench.whole_job_gbs(1e9, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_gbs(2e9, 1, 2.0) == pytest.approx(1000.0)


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [4.0, 4.0]
    # 2 ranks x 1 GB per step in 4 ms -> 500 GB/s for the whole job
    assert all(r[2] == pytest.approx(500.0) for r in res)
