"""The N-GPU benchmark path as world-size-2 gloo ranks on the CPU.

bench.py runs N independent replicas (rows need no exchange, so no collective
is on the data path); what the ranks share is the timing: the job's time is
the slowest rank's and the throughput counts every rank's tokens.  Also: the
reference arm prints on rank 0 only.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [10.0, 14.5][rank]
    ms = bench.max_over_ranks(local_ms, dist, "cpu")
    tps = bench.replica_throughput(world, 8, 100, ms * 1e-3)
    out.put((rank, ms, tps))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, tps in res:
        assert ms == 14.5                      # max over ranks
        assert tps == pytest.approx(2 * 8 * 100 / 14.5e-3)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.replica_throughput(1, 8, 10, 0.5) == 160.0


def test_reference_arm_prints_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, 2
    bench.run_reference(Args(), 1, 2)  # a non-zero rank returns at once, printing nothing
    assert capsys.readouterr().out == ""
