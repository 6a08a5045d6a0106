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


def _step1_param(got_p, want_p, g, lr):
    """A parameter after the first AdamW step, whose update is -lr g / (|g| + eps), about -lr sign(g)
    (PyTorch's AdamW at t = 1).  Where the oracle's gradient entry lies within 1e-4 of the gradient's rms
    of zero, the sign is not fixed by the arithmetic: the GPU's gradient, correct to rounding, may carry
    either sign there.  Those entries are held to the update's own bound (the two sides at most 2 lr
    apart, plus 1e-4 lr: with beta1, beta2 and the bias corrections held in fp32 the kernel's step is
    lr (1 + ~7e-6)); the others are returned for the usual comparison."""
    got_p, want_p, g = (np.asarray(x, np.float64) for x in (got_p, want_p, g))
    near = np.abs(g) <= 1e-4 * np.sqrt(np.mean(g * g))
    assert np.all(np.abs(got_p[near] - want_p[near]) <= 2 * lr * (1 + 1e-4))
    return got_p[~near], want_p[~near]


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
    # sampled rows of Y and dX (a shared-input pack: per projection's column slice, dX summed)
    rows = sample_rows(wl)
    Wm = G.base_weight_f64(wl, T)
    Xr, dYr = W.rows_as_f64(T.X[rows], wl.dtype), W.rows_as_f64(T.dY[rows], wl.dtype)
    Yo = np.zeros((len(rows), wl.d_out))
    dXo = np.zeros((len(rows), wl.d_in))
    for g, (o, w) in enumerate(zip(wl.group_offsets, wl.widths)):
        segs = G.oracle_segs(wl, T, g)
        Yo[:, o:o + w] = orc.forward_rows(Xr, rows, Wm[:, o:o + w], segs)
        dXo += orc.backward_rows(dYr[:, o:o + w], rows, Wm[:, o:o + w], segs)
    errs["Y_rows"] = G.rel_err(got["Y"][rows], Yo)
    errs["dX_rows"] = G.rel_err(got["dX"][rows], dXo)
    del Wm
    # adapter-side results in full, one adapter at a time (a job's H / dH hold its adapters'
    # blocks side by side)
    worst = {k: 0.0 for k in ("H", "dH", "dAt", "dBt", "At", "Bt", "mA", "vA", "mB", "vB")}
    Gn = wl.n_groups
    for j, (off, n) in enumerate(zip(wl.offsets, wl.n_tokens)):
        rs = slice(off, off + n)
        Xj = W.rows_as_f64(T.X[rs], wl.dtype)
        dYj = W.rows_as_f64(T.dY[rs], wl.dtype)
        t0 = 0
        for g, (o, w) in enumerate(zip(wl.group_offsets, wl.widths)):
            i = j * Gn + g
            r = wl.ranks[i]
            one = [orc.Seg(0, n, T.At[i].astype(np.float64).T, T.Bt[i].astype(np.float64).T, wl.alphas[i])]
            H, dH, dA, dB = orc.lora_grads(Xj, dYj[:, o:o + w], one)
            cmp = {"H": (got["H"][j][:, t0:t0 + r], H[0]), "dH": (got["dH"][j][:, t0:t0 + r], dH[0]),
                   "dAt": (got["dAt"][i], dA[0].T), "dBt": (got["dBt"][i], dB[0].T)}
            if step:
                for name, p, gr, mk, vk in (("At", T.At[i], dA[0].T, "mA", "vA"), ("Bt", T.Bt[i], dB[0].T, "mB", "vB")):
                    p2, m2, v2 = orc.adamw(p.astype(np.float64), gr, 0.0, 0.0, wl.lr, wl.beta1, wl.beta2, wl.eps,
                                           wl.weight_decay, 1)
                    cmp[name] = _step1_param(got[name][i], p2, gr, wl.lr)
                    cmp[mk] = (got[mk][i], m2)
                    cmp[vk] = (got[vk][i], v2)
            for k, (a, b) in cmp.items():
                worst[k] = max(worst[k], G.rel_err(a, b))
            t0 += r
    errs.update(worst)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"tolerance {tol} exceeded: {bad} (all: {errs})"
    return errs


def test_qproj_llama8b_fullsize():
    check_fullsize(W.llama8b_qproj())


def test_qproj_tiny_ranks_fullsize():
    check_fullsize(W.llama8b_qproj_tiny_ranks())


def test_qproj_f32_fullsize():
    check_fullsize(W.llama8b_qproj_f32())


@pytest.mark.parametrize("fused", [False, True], ids=["expand", "fused"])
def test_qproj_llama8b_w4_base_fullsize(fused):
    check_fullsize(W.llama8b_qproj_w4(), flags=M.MLORA_W4_FUSED if fused else 0)


def test_qkv_shared_input_llama8b_fullsize():
    check_fullsize(W.llama8b_qkv_shared())


def test_mlp_up_lognormal_fullsize():
    check_fullsize(W.mlp_up_lognormal())


def test_many_small_jobs_llama70b_down_fullsize():
    check_fullsize(W.llama70b_down_many_small())


@pytest.mark.slow
@pytest.mark.parametrize("proj", range(7), ids=[p[0] for p in W.LLAMA8B_PROJ])
def test_llama8b_layer_projection_fullsize(proj):
    check_fullsize(W.llama8b_layer(proj))
