"""The multi-GPU path of the benchmark is replicas only: every rank runs its own copy
of the workload and the ranks meet only at barriers and at the final max over their
times.  Its host logic runs here as two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, local = bench.init_replicas("gloo")
    assert (ws, r, local) == (world, rank, rank)
    dist.barrier()
    my_ms = [2.0, 5.0][rank]                     # rank 1 is the slower replica
    slowest = bench.max_over_ranks(my_ms, "cpu")
    rate = bench.whole_job_rate(1000.0, ws, slowest)
    out.put((rank, slowest, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(world))
    for rank, slowest, rate in got:
        assert slowest == 5.0                  # every rank sees the slowest replica
        assert rate == pytest.approx(2 * 1000.0 / 5e-3)   # all units over that time


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_env()[0] == 1
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(10.0, 1, 1.0) == pytest.approx(1e4)


def test_bench_reads_the_dominant_kernels_traffic_from_its_profile():
    """The bench line's roofline traffic comes from the committed ncu summary of the
    dominant kernel (DRAM bytes read + written per launch)."""
    sys.path.insert(0, ROOT)
    import bench
    t = bench.profiled_traffic()
    assert isinstance(t, int) and t > 0
