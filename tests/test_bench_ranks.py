"""The N > 1 path of the benchmark (replicas, one per GPU), on CPU: two gloo
ranks reduce their timings and bytes the way bench.py does under NCCL, and
every rank gets the whole-job throughput (all ranks' bytes over the slowest
rank's time)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [40.0, 50.0][rank]          # device time of the timed steps on this rank
        nbytes = [3.0e9, 2.0e9][rank]    # bytes this rank processed
        value, t_max = bench.job_throughput(nbytes, ms, device="cpu")
        results[rank] = (value, t_max)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_time_and_total_bytes():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    expect = (3.0e9 + 2.0e9) / 50e-3 / 1e9  # GB/s over the slower rank's 50 ms
    for r in range(world):
        assert got[r][1] == 50.0
        assert got[r][0] == pytest.approx(expect, rel=1e-12)


def test_single_process_is_its_own_job():
    import bench
    value, t = bench.job_throughput(6.0e9, 100.0)
    assert t == 100.0 and value == pytest.approx(60.0)


def test_spread_of_per_call_times():
    import bench
    ms = [0.010 * (i + 1) for i in range(11)]  # 10 .. 110 us
    st = bench.spread_us(ms)
    assert st == {"p10": 20.0, "median": 60.0, "p90": 100.0}
    assert bench.spread_us([0.025]) == {"p10": 25.0, "median": 25.0, "p90": 25.0}
    assert bench.spread_us([])["median"] is None

