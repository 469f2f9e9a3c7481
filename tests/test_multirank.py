"""The multi-rank host logic of bench.py with two gloo ranks on CPU: each rank
runs the whole workload (weak scaling), the job's time is the slowest rank's,
and the throughput counts the work of every rank.  No data-path collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.5 + rank, torch.device("cpu"))       # rank r took 1.5 + r ms
    tflops = bench.whole_job_tflops(world, 3e9, ms)
    out.put((rank, ms, tflops, bench._dist()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
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
    for rank, ms, tflops, (ws, r, _local) in res:
        assert ms == 2.5                        # max over ranks
        assert tflops == pytest.approx(2 * 3e9 / 2.5e-3 / 1e12)
        assert ws == 2 and r == rank


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(4.0, torch.device("cpu")) == 4.0
    assert bench.whole_job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
