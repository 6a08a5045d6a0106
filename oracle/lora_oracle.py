"""fp64 CPU oracle for the packed multi-adapter LoRA layer (forward, backward, AdamW).

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the packed LoRA layer computes.  It exists so the CUDA path
can be checked against it; only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import it.  It shares no code with the CUDA
library and imports nothing from the product package.

Sources (page title, section):
  * PLoRA: Efficient Concurrent LoRA Training for Large Language Models
    (full text), §2.1 "Low-Rank Adaptation": W in R^{d x k} frozen, trainable
    A in R^{d x r} and B in R^{r x k}; the adapted layer adds a scaled A.B
    to W.  The page prints the product as "B x A", which does not type-check
    with the stated shapes; the only product of these shapes is A.B (d x k).
  * same page, §2.4 "Packed LoRA fine-tuning": every job keeps its own
    adapter, data and loss; the per-job computation is the single-adapter one.
  * same page, §9.2 "Packed LoRA Kernels", Cases 1-4: the four backward
    products (grad of B's weight, grad of B's input, grad of A's weight, grad
    of A's input).  The case wording for 2 and 3 names the wrong reduction
    axis; the math below follows the chain rule instead.
  * same page, §8 "LoRA Memory Constraints": AdamW keeps a first moment
    ("momentum"), a second moment ("velocity") and the gradient per parameter.
    The step itself is not printed; it is read as decoupled-weight-decay AdamW
    in the order PyTorch applies it (decay, moments, bias correction, update).
  * Scale: s_i = alpha_i / r_i (the benchmark spec; the page writes alpha).

Notation: X_i (n_i x d_in) is job i's token rows, Y_i = X_i W + s_i (X_i A_i) B_i.
With H_i = X_i A_i and dH_i = s_i dY_i B_i^T:
    dB_i = s_i H_i^T dY_i            (Case 1)
    dH_i = s_i dY_i B_i^T            (Case 2, reduction over d_out)
    dA_i = X_i^T dH_i                (Case 3, reduction over tokens)
    dX_i = dY_i W^T + dH_i A_i^T     (Case 4 plus the frozen base term)
Everything is float64; stored bf16/fp32 inputs are widened exactly by the caller.

Parity pins (tests/test_oracle.py): hand-worked example, pure-Python brute
force on tiny inputs, explicit-product identity X(W + sAB), B=0 / A=0 / W=0
special cases, packed == separate, central finite differences of <Y, dY>,
torch.autograd (fp64) gradients, linearity, and torch.optim.AdamW (fp64).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Seg:
    """One job of the pack: rows [offset, offset+n) of X/dY, A (d_in x r), B (r x d_out), alpha."""
    offset: int
    n: int
    A: np.ndarray
    B: np.ndarray
    alpha: float

    @property
    def r(self) -> int:
        return self.A.shape[1]

    @property
    def s(self) -> float:
        # s_i = alpha_i / r_i
        return float(self.alpha) / float(self.r)


def forward(X: np.ndarray, W: np.ndarray, segs: list[Seg]):
    """Y = X W + s_i (X_i A_i) B_i on every job's rows (PLoRA §2.1, §2.4).

    Returns (Y, H) with H[i] = X_i A_i (the saved low-rank activation)."""
    X = np.asarray(X, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    Y = np.zeros((X.shape[0], W.shape[1]), dtype=np.float64)
    H = []
    for sg in segs:
        Xi = X[sg.offset:sg.offset + sg.n]
        Hi = Xi @ sg.A
        Y[sg.offset:sg.offset + sg.n] = Xi @ W + sg.s * (Hi @ sg.B)
        H.append(Hi)
    return Y, H


def backward(X: np.ndarray, W: np.ndarray, dY: np.ndarray, segs: list[Seg]):
    """Gradients of <Y, dY> for every job (PLoRA §9.2 Cases 1-4, by the chain rule).

    Returns (dX, dA, dB, dH): dX packed like X, lists per job otherwise."""
    X = np.asarray(X, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    dX = np.zeros_like(X)
    dA, dB, dH = [], [], []
    for sg in segs:
        rows = slice(sg.offset, sg.offset + sg.n)
        Xi, dYi = X[rows], dY[rows]
        Hi = Xi @ sg.A
        dBi = sg.s * (Hi.T @ dYi)                 # Case 1
        dHi = sg.s * (dYi @ sg.B.T)               # Case 2
        dAi = Xi.T @ dHi                          # Case 3
        dX[rows] = dYi @ W.T + dHi @ sg.A.T       # Case 4 + base
        dA.append(dAi)
        dB.append(dBi)
        dH.append(dHi)
    return dX, dA, dB, dH


def _seg_of_rows(rows: np.ndarray, segs: list[Seg]) -> np.ndarray:
    starts = np.array([sg.offset for sg in segs])
    ends = starts + np.array([sg.n for sg in segs])
    j = np.searchsorted(starts, rows, side="right") - 1
    if np.any(j < 0) or np.any(rows >= ends[j]):
        raise ValueError("row outside every job's segment")
    return j


def forward_rows(X_rows: np.ndarray, rows: np.ndarray, W: np.ndarray, segs: list[Seg]) -> np.ndarray:
    """The rows ``rows`` of Y (same definition as :func:`forward`), for sampled checks at full size."""
    X_rows = np.asarray(X_rows, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    j = _seg_of_rows(np.asarray(rows), segs)
    Y = X_rows @ W
    for k, sg in enumerate(segs):
        sel = np.nonzero(j == k)[0]
        if sel.size:
            Y[sel] += sg.s * ((X_rows[sel] @ sg.A) @ sg.B)
    return Y


def backward_rows(dY_rows: np.ndarray, rows: np.ndarray, W: np.ndarray, segs: list[Seg]) -> np.ndarray:
    """The rows ``rows`` of dX (same definition as :func:`backward`)."""
    dY_rows = np.asarray(dY_rows, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    j = _seg_of_rows(np.asarray(rows), segs)
    dX = dY_rows @ W.T
    for k, sg in enumerate(segs):
        sel = np.nonzero(j == k)[0]
        if sel.size:
            dX[sel] += (sg.s * (dY_rows[sel] @ sg.B.T)) @ sg.A.T
    return dX


def lora_grads(X: np.ndarray, dY: np.ndarray, segs: list[Seg]):
    """Only the adapter-side results (H, dH, dA, dB): what :func:`backward` gives minus the
    frozen-base term, which is the expensive part at full size."""
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    H, dH, dA, dB = [], [], [], []
    for sg in segs:
        rows = slice(sg.offset, sg.offset + sg.n)
        Xi, dYi = X[rows], dY[rows]
        Hi = Xi @ sg.A
        dHi = sg.s * (dYi @ sg.B.T)
        H.append(Hi)
        dH.append(dHi)
        dB.append(sg.s * (Hi.T @ dYi))
        dA.append(Xi.T @ dHi)
    return H, dH, dA, dB


def dequantize_w4(Wq: np.ndarray, Wscale: np.ndarray) -> np.ndarray:
    """The frozen base weight of a 4-bit-base layer, W (d_in x d_out), in float64.

    "PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §5 / §11.3 name a
    4-bit (QLoRA) base without fixing its format; the reading used here: Wq [d_out, d_in/2]
    bytes hold signed 4-bit codes q[o][k] in [-8, 7] (even k in the low nibble, two's
    complement) and Wscale [d_in/64, d_out] one scale per 64 consecutive k of each column:
    W[k][o] = q[o][k] * Wscale[k // 64][o]."""
    Wq = np.asarray(Wq, dtype=np.uint8)
    d_out, half = Wq.shape
    d_in = 2 * half
    lo = (Wq & 0x0F).astype(np.int64)
    hi = (Wq >> 4).astype(np.int64)
    nib = np.empty((d_out, d_in), dtype=np.int64)
    nib[:, 0::2] = lo
    nib[:, 1::2] = hi
    q = np.where(nib >= 8, nib - 16, nib).astype(np.float64)          # two's complement nibble
    scale = np.repeat(np.asarray(Wscale, dtype=np.float64), 64, axis=0)  # [d_in, d_out]
    return q.T * scale


def adamw(p, g, m, v, lr, beta1, beta2, eps, weight_decay, t):
    """One decoupled-weight-decay AdamW step at step count t >= 1 (PLoRA §8 names the state;
    the order is PyTorch's AdamW): returns new (p, m, v)."""
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    p = p * (1.0 - lr * weight_decay)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p = p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v
