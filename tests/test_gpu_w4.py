"""The 4-bit base (int4 codes + fp32 group scales, dequantised in shared memory by the GEMM's
converter warps) against the oracle, and against the bf16 path fed the same weight rounded to
bf16 (which must agree bit for bit: the products, their order and the rounding are the same)."""
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
    "ragged": dict(d_in=512, d_out=640, ranks=[1, 7, 64, 256], n_tokens=[200, 56, 300, 17]),
    "straddle": dict(d_in=256, d_out=384, ranks=[1, 2, 4, 8, 16, 32, 64, 128, 256, 3],
                     n_tokens=[16, 16, 32, 16, 48, 16, 16, 64, 16, 5]),
    "wide": dict(d_in=2048, d_out=1536, ranks=[16, 128, 8], n_tokens=[256, 384, 130]),
}


def _wl(name, i):
    c = CASES[name]
    return W.custom(f"w4_{name}", 970 + i, c["d_in"], c["d_out"], c["ranks"], c["n_tokens"], dtype="bf16_w4",
                    b_std=0.05)


@pytest.mark.parametrize("name", sorted(CASES))
def test_w4_base_vs_oracle(name):
    wl = _wl(name, sorted(CASES).index(name))
    T = W.materialise(wl)
    run = G.GpuRun(wl, T)
    try:
        assert run.status_after_backward == M.MLORA_OK
        G.compare(run.res, G.oracle_full(wl, T), G.TOL["bf16_w4"])
    finally:
        run.close()


@pytest.mark.parametrize("name", sorted(CASES))
def test_w4_base_matches_bf16_path_bitwise(name):
    wl = _wl(name, sorted(CASES).index(name))
    T = W.materialise(wl)
    # the bf16 weight the converter produces: fp32 product of code and scale, rounded to bf16
    q = np.empty((wl.d_out, wl.d_in), np.float32)
    q[:, 0::2] = (T.Wq & 15).astype(np.int8)
    q[:, 1::2] = (T.Wq >> 4).astype(np.int8)
    q = np.where(q >= 8, q - 16, q).astype(np.float32)
    Wt16 = W.to_bf16_bits(q * np.repeat(T.Wscale.T, 64, axis=1))
    wl16 = W.custom(wl.name + "_bf16", wl.cfg_id, wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, dtype="bf16", b_std=0.05)
    r4 = G.GpuRun(wl, T, step=False)
    r16 = G.GpuRun(wl16, T, step=False, Wt_override=Wt16)
    try:
        for k in ("Y", "dX"):
            assert np.array_equal(r4.res[k], r16.res[k]), k
        for k in ("H", "dH", "dAt", "dBt"):
            assert all(np.array_equal(a, b) for a, b in zip(r4.res[k], r16.res[k])), k
    finally:
        r4.close()
        r16.close()


def test_w4_rejects_bf16_entry_points():
    wl = _wl("ragged", 0)
    T = W.materialise(wl)
    layer = G.PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, G.scales_of(wl), dtype="bf16_w4", At=T.At, Bt=T.Bt)
    try:
        X = G.to_dev(T.X, "bf16")
        with pytest.raises(M.MloraError):
            M.mlora_forward(layer.plan, X.data_ptr(), X.data_ptr(), X.data_ptr(), layer.H.data_ptr(),
                            layer.workspace.data_ptr(), torch.cuda.current_stream().cuda_stream)
    finally:
        layer.close()
