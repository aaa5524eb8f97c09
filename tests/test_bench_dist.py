"""The multi-rank aggregation of bench.py: independent replicas on world-size 2
(gloo on CPU), throughput = all ranks' steps / the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    def reduce_max(x):
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    elapsed = [2.0, 3.0][rank]
    value, slowest = bench.combine_over_ranks(elapsed, 60, world, reduce_max)
    q.put((rank, value, slowest))
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, slowest in out:
        assert slowest == 3.0
        assert value == pytest.approx(2 * 60 / 3.0)


def test_single_rank_identity():
    import bench
    value, slowest = bench.combine_over_ranks(1.5, 30, 1, lambda x: x)
    assert slowest == 1.5 and value == pytest.approx(20.0)


def test_bench_arguments():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.steps >= 1 and a.warmup >= 3 and a.impl == "ours"
    a = bench.parse_args(["--impl", "reference", "--steps", "5", "--warmup", "3"])
    assert a.impl == "reference" and a.steps == 5
