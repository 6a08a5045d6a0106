"""The multi-rank path of the benchmark on CPU: two gloo ranks.

On N GPUs every rank runs its own replica of the pack (the layer shards by job with no collective
on the data path); the only cross-rank steps are the barrier around the timed region and the
max-over-ranks of the measured time, from which the whole-job throughput is computed."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [12.5, 20.0][rank]                    # per-rank timed-region durations
        dist.barrier()
        m = bench.max_over_ranks(ms)
        rate = bench.weak_scaling_rate(16384, world, 10, m)
        q.put((rank, m, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, rate in res:
        assert m == 20.0                            # the slowest rank's time on every rank
        assert rate == pytest.approx(16384 * 2 * 10 / 0.020)


def test_single_process_passthrough():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.weak_scaling_rate(100, 1, 4, 2.0) == pytest.approx(200000.0)
