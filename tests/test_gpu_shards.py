"""A pack split across ranks reproduces the whole pack: the two shards that mlora_shard_jobs gives
for two GPUs are planned and run one after the other on one GPU (each as its own pack of whole
jobs), and every output of every job is compared with the fp64 oracle of the whole pack."""
import numpy as np
import pytest
import torch

from adapter_gemm_packed_gb300 import _mlora as M
from adapter_gemm_packed_gb300 import workloads as W
import gpu_harness as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from adapter_gemm_packed_gb300 import build
    build.build()


def _want_for(want, wl, jobs):
    """The whole-pack oracle outputs restricted to `jobs` (rows and adapters), in shard order."""
    rows = np.concatenate([np.arange(wl.offsets[j], wl.offsets[j] + wl.n_tokens[j]) for j in jobs])
    out = {"Y": want["Y"][rows], "dX": want["dX"][rows]}
    for k in ("H", "dH", "dAt", "dBt", "At", "Bt", "mA", "vA", "mB", "vB"):
        out[k] = [want[k][j] for j in jobs]
    return out


@pytest.mark.parametrize("name,d_in,d_out,ranks,toks", [
    ("shards_plain", 512, 384, [4, 64, 16, 130, 8, 32], [300, 100, 150, 260, 40, 210]),
    ("shards_wide", 1024, 640, [256, 1, 8, 16, 2, 64, 32], [128, 500, 70, 130, 16, 330, 90]),
])
def test_two_shards_reproduce_the_whole_pack(name, d_in, d_out, ranks, toks):
    wl = W.custom(name, 970 + len(ranks), d_in, d_out, ranks, toks, dtype="bf16", b_std=0.05)
    T = W.materialise(wl)
    want = G.oracle_full(wl, T)
    prob = M.mlora_problem(wl.N, wl.d_in, wl.d_out, M.MLORA_BF16, M.MLORA_PLAN_HOST_ONLY)
    segs = [M.mlora_segment(o, n, r, 1.0) for o, n, r in zip(wl.offsets, wl.n_tokens, wl.ranks)]
    rank_of_job, _ = M.mlora_shard_jobs(prob, segs, 2)
    shards = [[j for j, r in enumerate(rank_of_job) if r == q] for q in range(2)]
    assert sorted(shards[0] + shards[1]) == list(range(len(ranks))) and shards[0] and shards[1]
    for jobs in shards:
        sub, S = W.materialise_jobs(wl, jobs)
        run = G.GpuRun(sub, S, flags=M.MLORA_REUSE_STAGING)
        try:
            assert run.status_after_backward == M.MLORA_OK
            G.compare(run.res, _want_for(want, wl, jobs), G.TOL["bf16"])
        finally:
            run.close()
        torch.cuda.synchronize()
