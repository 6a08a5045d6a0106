"""The 4-bit base (int4 codes + fp32 group scales) against the oracle, and against the bf16 path
fed the same weight rounded to bf16, which must agree bit for bit (the products, their order and
the rounding are the same).  Both ways of expanding the codes are covered: once per call into the
workspace (the default, also on single-CTA tiles) and inside the CTA-pair GEMMs by converter
warps (MLORA_W4_FUSED); so is the backward's reuse of the forward's expansion."""
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


MODES = {"expand": 0, "fused": M.MLORA_W4_FUSED, "expand_1cta": M.MLORA_GEMM_SINGLE_CTA}


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("name", sorted(CASES))
def test_w4_base_vs_oracle(name, mode):
    wl = _wl(name, sorted(CASES).index(name))
    T = W.materialise(wl)
    run = G.GpuRun(wl, T, flags=MODES[mode])
    try:
        assert run.status_after_backward == M.MLORA_OK
        G.compare(run.res, G.oracle_full(wl, T), G.TOL["bf16_w4"])
    finally:
        run.close()


def _bf16_weight(wl, T):
    """The bf16 weight the expansion produces: fp32 product of code and scale, rounded to bf16."""
    q = np.empty((wl.d_out, wl.d_in), np.float32)
    q[:, 0::2] = (T.Wq & 15).astype(np.int8)
    q[:, 1::2] = (T.Wq >> 4).astype(np.int8)
    q = np.where(q >= 8, q - 16, q).astype(np.float32)
    return W.to_bf16_bits(q * np.repeat(T.Wscale.T, 64, axis=1))


@pytest.mark.parametrize("mode", ["expand", "fused"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_w4_base_matches_bf16_path_bitwise(name, mode):
    wl = _wl(name, sorted(CASES).index(name))
    T = W.materialise(wl)
    Wt16 = _bf16_weight(wl, T)
    wl16 = W.custom(wl.name + "_bf16", wl.cfg_id, wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, dtype="bf16", b_std=0.05)
    r4 = G.GpuRun(wl, T, step=False, flags=MODES[mode])
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


def _dev_w4(Wq, Ws):
    return torch.from_numpy(np.ascontiguousarray(Wq)).cuda(), torch.from_numpy(np.ascontiguousarray(Ws)).cuda()


def test_w4_backward_reuses_or_reexpands():
    """With MLORA_REUSE_STAGING the backward skips the expansion only when the forward expanded
    the same Wq / Wscale buffers: given other buffers (here holding other codes) it expands
    those, and dX matches a plan without reuse that saw only the other weight."""
    wl = _wl("wide", 2)
    T = W.materialise(wl)
    rng = np.random.default_rng(5)
    Wq2 = rng.integers(0, 256, size=T.Wq.shape, dtype=np.uint8)
    sc = G.scales_of(wl)
    X, dY = G.to_dev(T.X, "bf16"), G.to_dev(T.dY, "bf16")
    outs = {}
    for name, flags, fwd_w, bwd_w in (("reuse_same", M.MLORA_REUSE_STAGING, T.Wq, T.Wq),
                                      ("plain_same", 0, T.Wq, T.Wq),
                                      ("reuse_other", M.MLORA_REUSE_STAGING, T.Wq, Wq2),
                                      ("plain_other", 0, Wq2, Wq2)):
        layer = G.PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, sc, dtype="bf16_w4", At=T.At, Bt=T.Bt,
                             flags=flags)
        try:
            wf = _dev_w4(fwd_w, T.Wscale)
            wb = wf if bwd_w is fwd_w else _dev_w4(bwd_w, T.Wscale)
            layer.forward(X, wf)
            dX = layer.backward(X, wb, dY)
            torch.cuda.synchronize()
            assert layer.sync_status() == M.MLORA_OK
            outs[name] = G.from_dev(dX, "bf16")
        finally:
            layer.close()
    assert np.array_equal(outs["reuse_same"], outs["plain_same"])
    assert np.array_equal(outs["reuse_other"], outs["plain_other"])
    assert not np.array_equal(outs["reuse_other"], outs["reuse_same"])


def test_w4_fused_rejects_single_cta():
    wl = _wl("ragged", 0)
    with pytest.raises(M.MloraError):
        G.PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, G.scales_of(wl), dtype="bf16_w4",
                     flags=M.MLORA_W4_FUSED | M.MLORA_GEMM_SINGLE_CTA)
