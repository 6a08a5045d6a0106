"""Full-size workloads, in the launch configuration the benchmark times, against the oracle.

Y and dX are checked on sampled token rows the oracle computes one by one (each job's first
and last row, the rows on both sides of every 128-token tile edge it crosses, and seeded
random rows); H, dH, dA, dB, and the AdamW step on A and B are checked in full."""
import numpy as np
import pytest
import torch

from adapter_gemm_packed_gb300 import _mlora as M
from adapter_gemm_packed_gb300 import workloads as W
from oracle import lora_oracle as orc
import gpu_harness as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adapter_gemm_packed_gb300 import build
    build.build()


def sample_rows(wl, max_rows=768, seed=0):
    rng = np.random.default_rng(seed)
    rows = set()
    for o, n in zip(wl.offsets, wl.n_tokens):
        rows.update({o, o + n - 1})
        for edge in range(((o // 128) + 1) * 128, o + n, 128):
            rows.update({edge - 1, edge})
    rows = sorted(rows)
    if len(rows) > max_rows:
        rows = sorted(rng.choice(rows, max_rows, replace=False).tolist())
    extra = rng.integers(0, wl.N, size=64)
    return np.unique(np.concatenate([np.array(rows, dtype=np.int64), extra]))


def check_fullsize(wl, step=True, flags=0):
    T = W.materialise(wl)
    run = G.GpuRun(wl, T, step=step, flags=flags)
    try:
        assert run.status_after_backward == M.MLORA_OK
        got = run.res
    finally:
        run.close()
    tol = G.TOL[wl.dtype]
    errs = {}
    # sampled rows of Y and dX
    rows = sample_rows(wl)
    Wm = G.base_weight_f64(wl, T)
    segs = G.oracle_segs(wl, T)
    Yo = orc.forward_rows(W.rows_as_f64(T.X[rows], wl.dtype), rows, Wm, segs)
    dXo = orc.backward_rows(W.rows_as_f64(T.dY[rows], wl.dtype), rows, Wm, segs)
    errs["Y_rows"] = G.rel_err(got["Y"][rows], Yo)
    errs["dX_rows"] = G.rel_err(got["dX"][rows], dXo)
    del Wm
    # adapter-side results in full, one job at a time
    worst = {k: 0.0 for k in ("H", "dH", "dAt", "dBt", "At", "Bt", "mA", "vA", "mB", "vB")}
    for i, sg in enumerate(segs):
        rs = slice(sg.offset, sg.offset + sg.n)
        one = [orc.Seg(0, sg.n, sg.A, sg.B, sg.alpha)]
        H, dH, dA, dB = orc.lora_grads(W.rows_as_f64(T.X[rs], wl.dtype), W.rows_as_f64(T.dY[rs], wl.dtype), one)
        cmp = {"H": (got["H"][i], H[0]), "dH": (got["dH"][i], dH[0]), "dAt": (got["dAt"][i], dA[0].T),
               "dBt": (got["dBt"][i], dB[0].T)}
        if step:
            for name, p, g, mk, vk in (("At", T.At[i], dA[0].T, "mA", "vA"), ("Bt", T.Bt[i], dB[0].T, "mB", "vB")):
                p2, m2, v2 = orc.adamw(p.astype(np.float64), g, 0.0, 0.0, wl.lr, wl.beta1, wl.beta2, wl.eps,
                                       wl.weight_decay, 1)
                cmp[name] = (got[name][i], p2)
                cmp[mk] = (got[mk][i], m2)
                cmp[vk] = (got[vk][i], v2)
        for k, (a, b) in cmp.items():
            worst[k] = max(worst[k], G.rel_err(a, b))
    errs.update(worst)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"tolerance {tol} exceeded: {bad} (all: {errs})"
    return errs


def test_qproj_llama8b_fullsize():
    check_fullsize(W.llama8b_qproj())


@pytest.mark.parametrize("fused", [False, True], ids=["expand", "fused"])
def test_qproj_llama8b_w4_base_fullsize(fused):
    check_fullsize(W.llama8b_qproj_w4(), flags=M.MLORA_W4_FUSED if fused else 0)


def test_mlp_up_lognormal_fullsize():
    check_fullsize(W.mlp_up_lognormal())


def test_many_small_jobs_llama70b_down_fullsize():
    check_fullsize(W.llama70b_down_many_small())


@pytest.mark.slow
@pytest.mark.parametrize("proj", range(7), ids=[p[0] for p in W.LLAMA8B_PROJ])
def test_llama8b_layer_projection_fullsize(proj):
    check_fullsize(W.llama8b_layer(proj))
