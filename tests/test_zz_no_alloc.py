"""mlora_forward_static_ws: the forward pass for callers that cannot allocate device memory.

Such callers (a runtime that forbids cudaMalloc after start-up, a framework that only hands
out memory from its own pools) cannot provide the workspace mlora_forward takes, so the
library offers a variant whose scratch is a static device array of its own, shared by every
plan on the device.  These checks call it through the C ABI.  The GPU check interleaves two
plans of different shapes and ranks on that one array (A, B, A, B), both built with
MLORA_REUSE_STAGING, so a plan that trusted what it had left in the array would read the
other plan's adapters.  Every call must equal mlora_forward on the plan's own workspace bit
for bit (the kernels are the same) and the fp64 oracle within the bf16 tolerance.  This file
is collected last on purpose."""
import numpy as np
import pytest
import torch

from adapter_gemm_packed_gb300 import _mlora as M
from adapter_gemm_packed_gb300 import workloads as W
from adapter_gemm_packed_gb300.layer import PackedLoRA, host_plan
from oracle import lora_oracle as orc
import gpu_harness as G


@pytest.fixture(scope="module", autouse=True)
def built():
    from adapter_gemm_packed_gb300 import build
    build.build()


def test_static_ws_rejects_plans_beyond_its_capacity():
    # 32 jobs of rank 256 on 8192 x 8192: the forward's bf16 shadows alone are 256 MiB
    plan, _ = host_plan(8192, 8192, [256] * 32, [128] * 32)
    try:
        st = M.lib().mlora_forward_static_ws(plan, 0x1000, 0x1000, 0x1000, 0x1000, None)
        assert st == M.MLORA_ERR_UNSUPPORTED
        assert "static" in M.lib().mlora_last_error().decode()
    finally:
        M.mlora_plan_destroy(plan)


def test_static_ws_rejects_4bit_base_plans():
    plan, _ = host_plan(256, 256, [8, 16], [64, 64], dtype="bf16_w4")
    try:
        st = M.lib().mlora_forward_static_ws(plan, 0x1000, 0x1000, 0x1000, 0x1000, None)
        assert st == M.MLORA_ERR_UNSUPPORTED
        assert "4-bit" in M.lib().mlora_last_error().decode()
    finally:
        M.mlora_plan_destroy(plan)


def _bits(t):
    return t.view(torch.int16).cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy().view(np.int32)


@pytest.mark.gpu
def test_static_ws_two_plans_interleaved_match_workspace_forward_and_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wls = [W.custom("static_ws_a", 960, 512, 384, [4, 64, 130], [300, 100, 150], dtype="bf16", b_std=0.05),
           W.custom("static_ws_b", 961, 384, 640, [32, 8, 16, 256], [90, 200, 40, 170], dtype="bf16", b_std=0.05)]
    Ts = [W.materialise(wl) for wl in wls]
    layers = [PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, G.scales_of(wl), dtype="bf16", At=T.At,
                         Bt=T.Bt, flags=M.MLORA_REUSE_STAGING) for wl, T in zip(wls, Ts)]
    try:
        Wts = [G.to_dev(T.Wt, "bf16") for T in Ts]
        stream = torch.cuda.current_stream().cuda_stream
        order = [0, 1, 0, 1]
        # a different activation each call, so a stale result would show
        Xs = [W.to_bf16_bits(W.normal_f32(wls[k].cfg_id, 500 + call, wls[k].N * wls[k].d_in, 1.0))
              .reshape(wls[k].N, wls[k].d_in) for call, k in enumerate(order)]
        # first the static-scratch calls back to back, so that each plan's second call follows the
        # other plan's call on the shared array with nothing in between
        got = []
        for call, k in enumerate(order):
            layer = layers[k]
            X = G.to_dev(Xs[call], "bf16")
            Y = torch.full((wls[k].N, wls[k].d_out), float("nan"), dtype=torch.bfloat16, device="cuda")
            H = torch.full_like(layer.H, float("nan"))
            M.mlora_forward_static_ws(layer.plan, X.data_ptr(), Wts[k].data_ptr(), Y.data_ptr(), H.data_ptr(), stream)
            torch.cuda.synchronize()
            assert layer.sync_status() == M.MLORA_OK
            got.append((Y, H))
        for call, k in enumerate(order):
            wl, T, layer = wls[k], Ts[k], layers[k]
            Y, H = got[call]
            X = G.to_dev(Xs[call], "bf16")
            Y_ref = layer.forward(X, Wts[k])
            torch.cuda.synchronize()
            # the same kernels on the same inputs: identical bits
            assert np.array_equal(_bits(Y), _bits(Y_ref)), f"call {call}: Y differs from mlora_forward"
            assert np.array_equal(_bits(H), _bits(layer.H)), f"call {call}: H differs from mlora_forward"
            # and the oracle on this call's inputs
            segs = [orc.Seg(o, n, T.At[i].astype(np.float64).T, T.Bt[i].astype(np.float64).T, wl.alphas[i])
                    for i, (o, n) in enumerate(zip(wl.offsets, wl.n_tokens))]
            Yo, Ho = orc.forward(W.rows_as_f64(Xs[call], "bf16"), W.rows_as_f64(T.Wt, "bf16").T, segs)
            tol = G.TOL["bf16"]
            assert G.rel_err(G.from_dev(Y, "bf16"), Yo) <= tol
            Hb = [h.cpu().numpy().astype(np.float64) for h in layer.h_blocks(H)]
            assert max(G.rel_err(a, b) for a, b in zip(Hb, Ho)) <= tol
    finally:
        for layer in layers:
            layer.close()
