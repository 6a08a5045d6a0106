"""A pack of LoRA jobs on one GPU: device buffers (allocated through PyTorch) plus one plan.

:class:`PackedLoRA` owns the per-job fp32 masters A_i^T / B_i^T, their gradients and AdamW
moments, the saved activations H / dH and the workspace, and calls the C ABI
(``mlora_forward`` / ``mlora_backward`` / ``mlora_adamw``) on the current PyTorch stream.
It performs no arithmetic of its own.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _mlora as M

_DT = {"bf16": (M.MLORA_BF16, torch.bfloat16), "f32": (M.MLORA_F32, torch.float32),
       "bf16_w4": (M.MLORA_BF16_W4, torch.bfloat16)}


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class PackedLoRA:
    def __init__(self, d_in: int, d_out: int, ranks, n_tokens, scales, dtype: str = "bf16",
                 device: str | torch.device = "cuda", flags: int = 0, At=None, Bt=None,
                 with_grads: bool = True, with_moments: bool = True):
        self.d_in, self.d_out = int(d_in), int(d_out)
        self.ranks = [int(r) for r in ranks]
        self.n_tokens = [int(n) for n in n_tokens]
        self.scales = [float(s) for s in scales]
        self.dtype = dtype
        self.code, self.tdtype = _DT[dtype]
        self.device = torch.device(device)
        self.N = sum(self.n_tokens)
        f32 = dict(dtype=torch.float32, device=self.device)
        self.At = [torch.as_tensor(a).to(**f32).contiguous() if At is not None else torch.zeros((r, self.d_in), **f32)
                   for r, a in zip(self.ranks, At if At is not None else self.ranks)]
        self.Bt = [torch.as_tensor(b).to(**f32).contiguous() if Bt is not None else torch.zeros((self.d_out, r), **f32)
                   for r, b in zip(self.ranks, Bt if Bt is not None else self.ranks)]
        z = lambda t: torch.zeros_like(t)
        self.dAt = [z(a) for a in self.At] if with_grads else [None] * len(self.ranks)
        self.dBt = [z(b) for b in self.Bt] if with_grads else [None] * len(self.ranks)
        self.mA = [z(a) for a in self.At] if with_moments else [None] * len(self.ranks)
        self.vA = [z(a) for a in self.At] if with_moments else [None] * len(self.ranks)
        self.mB = [z(b) for b in self.Bt] if with_moments else [None] * len(self.ranks)
        self.vB = [z(b) for b in self.Bt] if with_moments else [None] * len(self.ranks)
        segs, off = [], 0
        for i, (r, n, s) in enumerate(zip(self.ranks, self.n_tokens, self.scales)):
            segs.append(M.mlora_segment(off, n, r, s, _ptr(self.At[i]), _ptr(self.Bt[i]), _ptr(self.dAt[i]),
                                        _ptr(self.dBt[i]), _ptr(self.mA[i]), _ptr(self.vA[i]), _ptr(self.mB[i]),
                                        _ptr(self.vB[i])))
            off += n
        self.problem = M.mlora_problem(self.N, self.d_in, self.d_out, self.code, flags)
        self.plan, self.ws_bytes = M.mlora_plan(self.problem, segs)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=self.device)
        h = M.mlora_h_elems(self.plan)
        self.H = torch.zeros(max(h, 1), **f32)
        self.dH = torch.zeros(max(h, 1), **f32)

    # ---------------------------------------------------------------- calls
    def forward(self, X, Wt, Y=None, stream=None):
        """Wt: the bf16/fp32 weight, or a (codes, scales) pair for a 4-bit-base plan."""
        if Y is None:
            Y = torch.empty((self.N, self.d_out), dtype=self.tdtype, device=self.device)
        if self.dtype == "bf16_w4":
            Wq, Ws = Wt
            M.mlora_forward_w4(self.plan, X.data_ptr(), Wq.data_ptr(), Ws.data_ptr(), Y.data_ptr(), self.H.data_ptr(),
                               self.workspace.data_ptr(), _stream(stream))
        else:
            M.mlora_forward(self.plan, X.data_ptr(), Wt.data_ptr(), Y.data_ptr(), self.H.data_ptr(),
                            self.workspace.data_ptr(), _stream(stream))
        return Y

    def backward(self, X, Wt, dY, dX=None, stream=None):
        if dX is None:
            dX = torch.empty((self.N, self.d_in), dtype=self.tdtype, device=self.device)
        if self.dtype == "bf16_w4":
            Wq, Ws = Wt
            M.mlora_backward_w4(self.plan, X.data_ptr(), Wq.data_ptr(), Ws.data_ptr(), dY.data_ptr(),
                                self.H.data_ptr(), dX.data_ptr(), self.dH.data_ptr(), self.workspace.data_ptr(),
                                _stream(stream))
        else:
            M.mlora_backward(self.plan, X.data_ptr(), Wt.data_ptr(), dY.data_ptr(), self.H.data_ptr(), dX.data_ptr(),
                             self.dH.data_ptr(), self.workspace.data_ptr(), _stream(stream))
        return dX

    def adamw(self, lr, beta1, beta2, eps, weight_decay, step, stream=None):
        M.mlora_adamw(self.plan, lr, beta1, beta2, eps, weight_decay, step, _stream(stream))

    def sync_status(self, stream=None) -> int:
        return M.mlora_sync_status(self.plan, _stream(stream))

    def describe(self, what: int):
        return M.mlora_plan_describe(self.plan, what)

    def h_blocks(self, H=None):
        """Split the packed H (or dH) into per-job [n_i, r_i] views."""
        H = self.H if H is None else H
        out, o = [], 0
        for n, r in zip(self.n_tokens, self.ranks):
            out.append(H[o:o + n * r].view(n, r))
            o += n * r
        return out

    def close(self):
        if getattr(self, "plan", None):
            M.mlora_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def host_plan(d_in, d_out, ranks, n_tokens, dtype="bf16", scales=None, offsets=None, n_total=None,
              with_moments=True, flags=0):
    """Build a host-only plan (no CUDA call) over placeholder pointers, for inspecting the
    planner's tables.  Returns (handle, workspace_bytes); destroy with mlora_plan_destroy."""
    code = _DT[dtype][0]
    segs, off = [], 0
    fake = lambda i, k: 0x100000 * (1 + 16 * i + k)
    for i, (r, n) in enumerate(zip(ranks, n_tokens)):
        o = off if offsets is None else offsets[i]
        s = 1.0 if scales is None else scales[i]
        ptrs = [fake(i, k) for k in range(8)]
        if not with_moments:
            ptrs[4:] = [None] * 4
        segs.append(M.mlora_segment(o, n, r, s, *ptrs))
        off += n
    prob = M.mlora_problem(sum(n_tokens) if n_total is None else n_total, d_in, d_out, code,
                           M.MLORA_PLAN_HOST_ONLY | flags)
    return M.mlora_plan(prob, segs)
