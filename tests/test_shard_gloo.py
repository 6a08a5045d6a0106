"""The multi-rank path of the benchmark on CPU: two gloo ranks share one pack.

Under torchrun the pack's jobs are split across the ranks (whole jobs, longest first onto the
least-loaded rank, mlora_shard_jobs_multi) and each rank plans and trains only its jobs: the
layer shards by job with no collective on the data path, because a job's gradients and AdamW
step touch only its own adapters.  The only cross-rank steps are the barrier around the timed
region and the max-over-ranks of the measured time, from which the whole pack's throughput is
computed.  Here each rank builds host-only plans of its shard for all seven projections of the
Llama-3-8B layer workload and the ranks compare notes."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _tables(wl, jobs):
    """Per job of `jobs` (a host-only plan of just those jobs): its rank, padded rank-window width
    and tokens, as the planner recorded them."""
    from adapter_gemm_packed_gb300 import _mlora as M
    from adapter_gemm_packed_gb300.layer import host_plan
    ranks = [wl.ranks[j] for j in jobs]
    toks = [wl.n_tokens[j] for j in jobs]
    plan, _ = host_plan(wl.d_in, wl.d_out, ranks, toks)
    try:
        ad = M.mlora_plan_describe(plan, M.MLORA_Q_ADAPTERS)      # job, c0, r, o_lo, o_hi per entry
        co = M.mlora_plan_describe(plan, M.MLORA_Q_COLUMNS)       # c, rp per job
        summ = M.mlora_plan_describe(plan, M.MLORA_Q_SUMMARY)
    finally:
        M.mlora_plan_destroy(plan)
    return {"rank": ad[2::5], "width": co[1::2], "out": list(zip(ad[3::5], ad[4::5])), "tokens": toks,
            "N": summ[0]}


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        wl = bench.workload("layer")
        rank_of_job, load = bench.shard(wl, world)
        mine = bench.jobs_of_rank(rank_of_job, rank)
        per_part = [_tables(p, mine) for p in wl.parts]
        everyone = [None] * world
        dist.all_gather_object(everyone, mine)
        ms = [12.5, 20.0][rank]                    # per-rank timed-region durations
        dist.barrier()
        m = bench.max_over_ranks(ms)
        rate = bench.pack_rate(wl.N, 10, m)
        q.put((rank, mine, everyone, per_part, m, rate, load))
    except BaseException as e:          # report instead of leaving the parent waiting
        q.put((rank, repr(e), None, None, None, None, None))
        raise
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_the_pack_and_time_it_together():
    import bench
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=300) for _ in range(2)], key=lambda x: x[0])
    assert all(r[2] is not None for r in res), res
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    wl = bench.workload("layer")
    J = len(wl.n_tokens)
    # every job lands on exactly one rank, and both ranks agree on the split
    assert res[0][2] == res[1][2]
    jobs = sorted(j for _, mine, _, _, _, _, _ in res for j in mine)
    assert jobs == list(range(J))
    assert set(res[0][1]).isdisjoint(res[1][1]) and res[0][1] and res[1][1]
    # each rank's plans hold its jobs with the ranks, windows and tokens the whole pack's plans give them
    for rank, mine, _, per_part, m, rate, load in res:
        for p, tab in zip(wl.parts, per_part):
            whole = _tables(p, list(range(J)))
            assert tab["rank"] == [whole["rank"][j] for j in mine]
            assert tab["width"] == [whole["width"][j] for j in mine]
            assert tab["out"] == [whole["out"][j] for j in mine]
            assert tab["tokens"] == [whole["tokens"][j] for j in mine] and tab["N"] == sum(tab["tokens"])
        assert m == 20.0                            # the slowest rank's time on every rank
        assert rate == pytest.approx(wl.N * 10 / 0.020)
        # longest first: the two ranks' costs differ by at most the largest job's
        costs = [n * sum(pp.d_in * pp.d_out + 3 * r * (pp.d_in + pp.d_out) for pp in wl.parts)
                 for n, r in zip(wl.n_tokens, wl.ranks)]
        assert abs(load[0] - load[1]) <= max(costs) * (1 + 1e-9)
        assert sum(load) == pytest.approx(sum(costs))


def test_single_process_passthrough():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.pack_rate(100, 4, 2.0) == pytest.approx(200000.0)
    rank_of_job, load = bench.shard(bench.workload("qproj"), 1)
    assert rank_of_job == [0] * 8 and len(load) == 1
