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
    """One plan and its buffers.

    ``groups`` (optional, a list of output widths summing to d_out) makes a shared-input pack:
    then ``ranks[j]``, ``scales[j]`` (and ``At[j]``, ``Bt[j]`` if given) are lists with one entry
    per group, job j's adapter on that group, whose Bt is [width_g, r].  The flat lists
    ``self.At``, ``self.Bt``, ``self.dAt``, ... follow the segment table's job-major order."""

    def __init__(self, d_in: int, d_out: int, ranks, n_tokens, scales, dtype: str = "bf16",
                 device: str | torch.device = "cuda", flags: int = 0, At=None, Bt=None,
                 with_grads: bool = True, with_moments: bool = True, groups=None):
        self.d_in, self.d_out = int(d_in), int(d_out)
        self.n_tokens = [int(n) for n in n_tokens]
        self.groups = None if groups is None else [int(w) for w in groups]
        G = 1 if groups is None else len(self.groups)
        widths = [self.d_out] if groups is None else self.groups
        nest = (lambda x: [[v] for v in x]) if groups is None else (lambda x: [list(v) for v in x])
        ranks_jg = nest(ranks)
        scales_jg = nest(scales)
        At_jg = None if At is None else nest(At)
        Bt_jg = None if Bt is None else nest(Bt)
        self.ranks = [int(r) for rj in ranks_jg for r in rj]              # per entry, job-major
        self.scales = [float(x) for sj in scales_jg for x in sj]
        self.job_rank = [sum(int(r) for r in rj) for rj in ranks_jg]       # R_j: width of job j's H block
        self.dtype = dtype
        self.code, self.tdtype = _DT[dtype]
        self.device = torch.device(device)
        self.N = sum(self.n_tokens)
        f32 = dict(dtype=torch.float32, device=self.device)
        self.At, self.Bt = [], []
        for j, rj in enumerate(ranks_jg):
            for g, r in enumerate(rj):
                self.At.append(torch.as_tensor(At_jg[j][g]).to(**f32).contiguous() if At is not None
                               else torch.zeros((r, self.d_in), **f32))
                self.Bt.append(torch.as_tensor(Bt_jg[j][g]).to(**f32).contiguous() if Bt is not None
                               else torch.zeros((widths[g], r), **f32))
        z = lambda t: torch.zeros_like(t)
        n_e = len(self.ranks)
        self.dAt = [z(a) for a in self.At] if with_grads else [None] * n_e
        self.dBt = [z(b) for b in self.Bt] if with_grads else [None] * n_e
        self.mA = [z(a) for a in self.At] if with_moments else [None] * n_e
        self.vA = [z(a) for a in self.At] if with_moments else [None] * n_e
        self.mB = [z(b) for b in self.Bt] if with_moments else [None] * n_e
        self.vB = [z(b) for b in self.Bt] if with_moments else [None] * n_e
        segs, off = [], 0
        for j, n in enumerate(self.n_tokens):
            for g in range(G):
                i = j * G + g
                segs.append(M.mlora_segment(off, n, self.ranks[i], self.scales[i], _ptr(self.At[i]), _ptr(self.Bt[i]),
                                            _ptr(self.dAt[i]), _ptr(self.dBt[i]), _ptr(self.mA[i]), _ptr(self.vA[i]),
                                            _ptr(self.mB[i]), _ptr(self.vB[i])))
            off += n
        self.problem = M.mlora_problem(self.N, self.d_in, self.d_out, self.code, flags)
        if groups is None:
            self.plan, self.ws_bytes = M.mlora_plan(self.problem, segs)
        else:
            offs = [sum(widths[:g]) for g in range(G)]
            self.plan, self.ws_bytes = M.mlora_plan_grouped(self.problem, list(zip(offs, widths)), segs)
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

    def adamw(self, lr, beta1, beta2, eps, weight_decay, step, stream=None, refresh_shadows=True):
        """One AdamW step on every adapter; by default it also refreshes the bf16 shadows in this
        layer's workspace (mlora_adamw_ws), which the next forward reuses under MLORA_REUSE_STAGING."""
        if refresh_shadows:
            M.mlora_adamw_ws(self.plan, lr, beta1, beta2, eps, weight_decay, step, self.workspace.data_ptr(),
                             _stream(stream))
        else:
            M.mlora_adamw(self.plan, lr, beta1, beta2, eps, weight_decay, step, _stream(stream))

    def sync_status(self, stream=None) -> int:
        return M.mlora_sync_status(self.plan, _stream(stream))

    def describe(self, what: int):
        return M.mlora_plan_describe(self.plan, what)

    def h_blocks(self, H=None):
        """Split the packed H (or dH) into per-job [n_j, R_j] views (R_j = r_j, or the sum of the
        job's ranks over the groups of a shared-input pack)."""
        H = self.H if H is None else H
        out, o = [], 0
        for n, r in zip(self.n_tokens, self.job_rank):
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
              with_moments=True, flags=0, mem_budget=0):
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
                           M.MLORA_PLAN_HOST_ONLY | flags, mem_budget)
    return M.mlora_plan(prob, segs)


def host_plan_grouped(d_in, widths, ranks_jg, n_tokens, dtype="bf16", flags=0):
    """Host-only shared-input plan over placeholder pointers (see host_plan); ranks_jg[j][g] is
    job j's rank on group g.  Returns (handle, workspace_bytes)."""
    code = _DT[dtype][0]
    segs, off, k = [], 0, 0
    for rj, n in zip(ranks_jg, n_tokens):
        for r in rj:
            segs.append(M.mlora_segment(off, n, r, 1.0, *[0x100000 * (1 + 16 * k + u) for u in range(8)]))
            k += 1
        off += n
    offs = [sum(widths[:g]) for g in range(len(widths))]
    prob = M.mlora_problem(sum(n_tokens), d_in, sum(widths), code, M.MLORA_PLAN_HOST_ONLY | flags)
    return M.mlora_plan_grouped(prob, list(zip(offs, widths)), segs)


class _PackedLoRAFn(torch.autograd.Function):
    """Autograd bridge: forward -> mlora_forward, backward -> mlora_backward (dX to the caller,
    the adapters' gradients into the layer's dAt / dBt buffers)."""

    @staticmethod
    def forward(ctx, X, layer, Wt):
        ctx.layer = layer
        ctx.Wt = Wt
        ctx.save_for_backward(X)
        return layer.forward(X, Wt)

    @staticmethod
    def backward(ctx, dY):
        (X,) = ctx.saved_tensors
        dX = ctx.layer.backward(X, ctx.Wt, dY.contiguous())
        return dX, None, None


class PackedLoRALinear(torch.nn.Module):
    """A packed LoRA layer as a module: ``y = mod(x)`` runs the fused forward, ``backward`` of the
    graph runs the fused backward (the gradient of x flows on; the adapters' gradients stay in
    ``mod.layer.dAt`` / ``dBt``), and ``mod.step(...)`` applies the library's AdamW to every adapter.

    The frozen weight ``Wt`` (bf16 / fp32 tensor, or a (codes, scales) pair for a 4-bit base) is
    held as given; each forward must be followed by its backward before the next forward (the
    layer keeps one H)."""

    def __init__(self, layer: PackedLoRA, Wt):
        super().__init__()
        self.layer = layer
        self.Wt = Wt
        self._t = 0

    def forward(self, X):
        return _PackedLoRAFn.apply(X, self.layer, self.Wt)

    def step(self, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01):
        self._t += 1
        self.layer.adamw(lr, betas[0], betas[1], eps, weight_decay, self._t)
