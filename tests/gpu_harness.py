"""Runs one workload through the CUDA path (C ABI) and through the fp64 oracle on the same
seeded inputs, and compares them tensor by tensor.

Tolerances (relative Frobenius error per output tensor): 1e-4 for fp32 workloads, 2e-2 for
bf16 workloads (bf16 inputs, fp32 accumulation, bf16 Y/dX).  An all-zero reference tensor
uses an absolute bound instead (1e-6 times the largest input magnitude, see ``rel_err``).
"""
from __future__ import annotations

import numpy as np
import torch

from adapter_gemm_packed_gb300 import workloads as W
from adapter_gemm_packed_gb300.layer import PackedLoRA
from oracle import lora_oracle as orc

TOL = {"f32": 1e-4, "bf16": 2e-2, "bf16_w4": 2e-2}


def rel_err(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    nw = np.linalg.norm(want)
    d = np.linalg.norm(got - want)
    if nw == 0:
        return d / 1e-6
    return d / nw


def to_dev(a: np.ndarray, dtype: str):
    if dtype in ("bf16", "bf16_w4"):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def from_dev(t, dtype: str) -> np.ndarray:
    if dtype in ("bf16", "bf16_w4"):
        return W.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return t.float().cpu().numpy().astype(np.float64)


def scales_of(wl):
    # the segment table's scale s_i = alpha_i / r_i (exact in fp32 for every workload here)
    return [np.float32(a) / np.float32(r) for a, r in zip(wl.alphas, wl.ranks)]


def make_layer(wl, T, flags=0):
    """The PackedLoRA of a workload (a shared-input pack when the workload has groups)."""
    if wl.groups is None:
        return PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, scales_of(wl), dtype=wl.dtype,
                          At=T.At, Bt=T.Bt, flags=flags)
    return PackedLoRA(wl.d_in, wl.d_out, wl.nest(wl.ranks), wl.n_tokens, wl.nest(scales_of(wl)), dtype=wl.dtype,
                      At=wl.nest(T.At), Bt=wl.nest(T.Bt), flags=flags, groups=wl.groups)


def oracle_segs(wl, T, g=0):
    """The oracle's job list for projection g (the only one unless the workload has groups)."""
    G = wl.n_groups
    return [orc.Seg(o, n, T.At[j * G + g].astype(np.float64).T, T.Bt[j * G + g].astype(np.float64).T,
                    wl.alphas[j * G + g])
            for j, (o, n) in enumerate(zip(wl.offsets, wl.n_tokens))]


class GpuRun:
    """Forward, backward and one AdamW step of a workload on the GPU; results as float64 numpy."""

    def __init__(self, wl, T, step=True, flags=0, Wt_override=None):
        self.wl = wl
        torch.cuda.synchronize()
        self.layer = make_layer(wl, T, flags)
        self.X = to_dev(T.X, wl.dtype)
        if wl.dtype == "bf16_w4":
            self.Wt = (torch.from_numpy(T.Wq).cuda(), torch.from_numpy(T.Wscale).cuda())
        else:
            self.Wt = to_dev(T.Wt if Wt_override is None else Wt_override, wl.dtype)
        self.dY = to_dev(T.dY, wl.dtype)
        self.Y = self.layer.forward(self.X, self.Wt)
        self.dX = self.layer.backward(self.X, self.Wt, self.dY)
        torch.cuda.synchronize()
        self.status_after_backward = self.layer.sync_status()
        self.res = dict(
            Y=from_dev(self.Y, wl.dtype), dX=from_dev(self.dX, wl.dtype),
            H=[h.cpu().numpy().astype(np.float64) for h in self.layer.h_blocks()],
            dH=[h.cpu().numpy().astype(np.float64) for h in self.layer.h_blocks(self.layer.dH)],
            dAt=[a.cpu().numpy().astype(np.float64) for a in self.layer.dAt],
            dBt=[b.cpu().numpy().astype(np.float64) for b in self.layer.dBt])
        if step:
            self.layer.adamw(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, 1)
            torch.cuda.synchronize()
            self.res.update(
                At=[a.cpu().numpy().astype(np.float64) for a in self.layer.At],
                Bt=[b.cpu().numpy().astype(np.float64) for b in self.layer.Bt],
                mA=[a.cpu().numpy().astype(np.float64) for a in self.layer.mA],
                vA=[a.cpu().numpy().astype(np.float64) for a in self.layer.vA],
                mB=[b.cpu().numpy().astype(np.float64) for b in self.layer.mB],
                vB=[b.cpu().numpy().astype(np.float64) for b in self.layer.vB])

    def close(self):
        self.layer.close()


def base_weight_f64(wl, T, Wt_override=None):
    """W (d_in x d_out) in fp64: the stored bf16/fp32 values, or the dequantised 4-bit base."""
    if wl.dtype == "bf16_w4":
        return orc.dequantize_w4(T.Wq, T.Wscale)
    return W.rows_as_f64(T.Wt if Wt_override is None else Wt_override, wl.dtype).T


def oracle_full(wl, T, Wt_override=None):
    """Every output of the layer (and the AdamW step at t=1 from zero moments), fp64.

    A shared-input pack is the oracle applied to each projection's column slice of W and dY
    with that projection's adapters: Y is the slices side by side, dX their sum, a job's H and
    dH its adapters' blocks side by side."""
    X = W.rows_as_f64(T.X, wl.dtype)
    Wm = base_weight_f64(wl, T, Wt_override)
    dY = W.rows_as_f64(T.dY, wl.dtype)
    G, J = wl.n_groups, len(wl.n_tokens)
    Y = np.zeros((wl.N, wl.d_out))
    dX = np.zeros((wl.N, wl.d_in))
    Hj, dHj = [[] for _ in range(J)], [[] for _ in range(J)]
    dAt, dBt = [None] * wl.n_adapters, [None] * wl.n_adapters
    for g, (o, w) in enumerate(zip(wl.group_offsets, wl.widths)):
        segs = oracle_segs(wl, T, g)
        Yg, Hg = orc.forward(X, Wm[:, o:o + w], segs)
        dXg, dAg, dBg, dHg = orc.backward(X, Wm[:, o:o + w], dY[:, o:o + w], segs)
        Y[:, o:o + w] = Yg
        dX += dXg
        for j in range(J):
            Hj[j].append(Hg[j])
            dHj[j].append(dHg[j])
            dAt[j * G + g] = dAg[j].T
            dBt[j * G + g] = dBg[j].T
    out = dict(Y=Y, dX=dX, H=[np.hstack(h) for h in Hj], dH=[np.hstack(h) for h in dHj], dAt=dAt, dBt=dBt)
    out.update(adamw_expect(wl, T, out["dAt"], out["dBt"]))
    return out


def adamw_expect(wl, T, dAt, dBt):
    At, Bt, mA, vA, mB, vB = [], [], [], [], [], []
    for i in range(wl.n_adapters):
        for p, g, P, Mm, V in ((T.At[i], dAt[i], At, mA, vA), (T.Bt[i], dBt[i], Bt, mB, vB)):
            p2, m2, v2 = orc.adamw(p.astype(np.float64), g, np.zeros_like(g), np.zeros_like(g), wl.lr, wl.beta1,
                                   wl.beta2, wl.eps, wl.weight_decay, 1)
            P.append(p2)
            Mm.append(m2)
            V.append(v2)
    return dict(At=At, Bt=Bt, mA=mA, vA=vA, mB=mB, vB=vB)


def compare(got: dict, want: dict, tol: float, keys=None) -> dict:
    """Max relative Frobenius error per key (lists: per job, reporting the worst)."""
    errs = {}
    for k in (keys or want.keys()):
        if k not in got or k not in want:
            continue
        g, w = got[k], want[k]
        if isinstance(w, list):
            errs[k] = max(rel_err(a, b) for a, b in zip(g, w))
        else:
            errs[k] = rel_err(g, w)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"tolerance {tol} exceeded: {bad} (all: {errs})"
    return errs
