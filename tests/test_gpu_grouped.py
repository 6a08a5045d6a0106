"""Shared-input packs: several projections stacked in W (q/k/v, gate/up), one adapter per job and
projection, one pass over X for every adapter's H.  Checked against the oracle applied to each
projection's column slice (Y side by side, dX summed, a job's H / dH its adapters' blocks side
by side), and a one-group grouped plan against the plain plan bit for bit (same tables, same
kernels)."""
import numpy as np
import pytest
import torch

from adapter_gemm_packed_gb300 import _mlora as M
from adapter_gemm_packed_gb300 import workloads as W
import gpu_harness as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adapter_gemm_packed_gb300 import build
    build.build()


CASES = {
    # ragged token tails, a 17-token job, ranks 1..128 mixed within a job
    "qkv_ragged": dict(d_in=512, widths=[256, 64, 64],
                       ranks_jg=[[8, 8, 8], [64, 16, 1], [3, 128, 32], [16, 16, 16]], n_tokens=[200, 56, 300, 17]),
    # widths that are not multiples of the 256-column tile, job windows of up to 7 chunks
    "odd_widths": dict(d_in=256, widths=[136, 48, 72],
                       ranks_jg=[[1, 2, 4], [8, 16, 32], [64, 128, 256], [5, 7, 9], [16, 16, 16]],
                       n_tokens=[16, 48, 64, 5, 130]),
    # two projections (gate / up)
    "gate_up": dict(d_in=384, widths=[640, 640], ranks_jg=[[32, 32], [128, 128], [8, 8]], n_tokens=[128, 257, 64]),
}


def _wl(name, dtype="bf16"):
    c = CASES[name]
    i = sorted(CASES).index(name)
    return W.custom_grouped(f"grouped_{name}_{dtype}", 990 + i + (10 if dtype != "bf16" else 0), c["d_in"],
                            c["widths"], c["ranks_jg"], c["n_tokens"], dtype=dtype, b_std=0.05)


@pytest.mark.parametrize("window", ["win_pairs", "win_single"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_grouped_vs_oracle(name, window):
    wl = _wl(name)
    T = W.materialise(wl)
    run = G.GpuRun(wl, T, flags=M.MLORA_WINDOW_PAIRS if window == "win_pairs" else M.MLORA_WINDOW_SINGLE)
    try:
        assert run.status_after_backward == M.MLORA_OK
        G.compare(run.res, G.oracle_full(wl, T), G.TOL["bf16"])
    finally:
        run.close()


def test_grouped_w4_base_vs_oracle():
    wl = _wl("qkv_ragged", "bf16_w4")
    T = W.materialise(wl)
    run = G.GpuRun(wl, T)
    try:
        assert run.status_after_backward == M.MLORA_OK
        G.compare(run.res, G.oracle_full(wl, T), G.TOL["bf16_w4"])
    finally:
        run.close()


def test_one_group_grouped_plan_equals_plain_plan():
    wl = W.custom("grouped_one", 997, 512, 384, [8, 64, 3, 16], [200, 56, 300, 17], b_std=0.05)
    T = W.materialise(wl)
    plain = G.GpuRun(wl, T, step=True)
    wl1 = W.custom_grouped("grouped_one_g", 997, 512, [384], [[r] for r in wl.ranks], wl.n_tokens, b_std=0.05)
    grouped = G.GpuRun(wl1, T, step=True)
    try:
        for k in ("Y", "dX"):
            assert np.array_equal(plain.res[k], grouped.res[k]), k
        for k in ("H", "dH", "dAt", "dBt", "At", "Bt", "mA", "vA", "mB", "vB"):
            assert all(np.array_equal(a, b) for a, b in zip(plain.res[k], grouped.res[k])), k
    finally:
        plain.close()
        grouped.close()


def test_grouped_rejects_fp32():
    wl = _wl("gate_up")
    with pytest.raises(M.MloraError) as e:
        G.PackedLoRA(wl.d_in, wl.d_out, wl.nest(wl.ranks), wl.n_tokens, wl.nest(G.scales_of(wl)), dtype="f32",
                     groups=wl.groups)
    assert e.value.status == M.MLORA_ERR_UNSUPPORTED
