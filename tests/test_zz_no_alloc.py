"""mlora_forward_static_ws: the forward pass for callers that cannot allocate device memory.

Such callers (a runtime that forbids cudaMalloc after start-up, a framework that only hands
out memory from its own pools) cannot provide the workspace mlora_forward takes, so the
library offers a variant whose scratch is a static device array of its own.  These checks
call it through the C ABI and compare it with mlora_forward on a caller workspace, on two
calls in a row with different inputs (the shared array keeps the previous call's contents,
which must not leak into the next result).  This file is collected last on purpose."""
import ctypes as C

import numpy as np
import pytest
import torch

from adapter_gemm_packed_gb300 import _mlora as M
from adapter_gemm_packed_gb300 import workloads as W
from adapter_gemm_packed_gb300.layer import PackedLoRA, host_plan
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


@pytest.mark.gpu
def test_static_ws_forward_matches_workspace_forward_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = W.custom("static_ws", 960, 512, 384, [4, 64, 130], [300, 100, 150], dtype="bf16", b_std=0.05)
    T = W.materialise(wl)
    layer = PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, G.scales_of(wl), dtype="bf16", At=T.At, Bt=T.Bt)
    try:
        Wt = G.to_dev(T.Wt, "bf16")
        stream = torch.cuda.current_stream().cuda_stream
        for call in range(2):
            # a different activation each call, so stale scratch from the first call would show
            X_np = W.to_bf16_bits(W.normal_f32(wl.cfg_id, 500 + call, wl.N * wl.d_in, 1.0)).reshape(wl.N, wl.d_in)
            X = G.to_dev(X_np, "bf16")
            Y_ref = layer.forward(X, Wt)
            H_ref = layer.H.clone()
            Y = torch.empty_like(Y_ref)
            H = torch.zeros_like(layer.H)
            M.mlora_forward_static_ws(layer.plan, X.data_ptr(), Wt.data_ptr(), Y.data_ptr(), H.data_ptr(), stream)
            torch.cuda.synchronize()
            assert layer.sync_status() == M.MLORA_OK
            tol = G.TOL["bf16"]
            assert G.rel_err(G.from_dev(Y, "bf16"), G.from_dev(Y_ref, "bf16")) <= tol
            assert G.rel_err(H.cpu().numpy(), H_ref.cpu().numpy()) <= tol
    finally:
        layer.close()
