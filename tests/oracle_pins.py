"""Independent checks ("pins") of the fp64 oracle.

Every pin takes an oracle-like object ``orc`` exposing ``Seg``, ``forward``,
``backward``, ``forward_rows``, ``backward_rows``, ``lora_grads`` and
``adamw`` and returns ``None`` when the oracle passes, or a string saying what
failed.  The oracle test asserts that every pin passes; the mutation test
plants mistakes into copies of the oracle and asserts that some pin catches
each one.  No pin re-types the oracle's formula: each compares it with
something fixed independently (hand-worked values, brute-force loops, a
different association of the same product, special cases that reduce to a
plain matmul, finite differences, torch autograd or torch.optim.AdamW).
"""
from __future__ import annotations

import os
import re

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            rows = [r.split() for r in v.split(";")]
            if len(rows) == 1 and len(rows[0]) == 1:
                vals[k] = rows[0][0]
            else:
                vals[k] = np.array([[float(x) for x in r] for r in rows], dtype=np.float64)
    return vals


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def _rand_segs(orc, rng, d_in, d_out, ranks, ns, alphas=None):
    segs, off = [], 0
    for i, (r, n) in enumerate(zip(ranks, ns)):
        A = rng.standard_normal((d_in, r))
        B = rng.standard_normal((r, d_out))
        a = float(alphas[i]) if alphas is not None else 2.0 * r + 1.0
        segs.append(orc.Seg(off, n, A, B, a))
        off += n
    return segs, off


# ---------------------------------------------------------------- forward/backward

def pin_hand_worked(orc):
    g = _parse_golden("hand_worked_packed_lora.txt")
    X, W, dY = g["X"], g["W"], g["dY"]
    col = lambda m: m.reshape(-1, 1) if m.ndim == 1 else m
    segs = [orc.Seg(0, 2, g["A0"], g["B0"], 4.0),
            orc.Seg(2, 1, col(g["A1"]).reshape(2, 1), g["B1"].reshape(1, 3), 3.0)]
    Y, H = orc.forward(X, W, segs)
    dX, dA, dB, dH = orc.backward(X, W, dY, segs)
    checks = [("Y", Y, g["Y"]), ("H0", H[0], g["H0"]), ("H1", H[1], np.array([[1.0]])),
              ("dX", dX, g["dX"]), ("dA0", dA[0], g["dA0"]), ("dA1", dA[1], g["dA1"].reshape(2, 1)),
              ("dB0", dB[0], g["dB0"]), ("dB1", dB[1], g["dB1"].reshape(1, 3)),
              ("dH0", dH[0], g["dH0"]), ("dH1", dH[1], np.array([[6.0]]))]
    for name, got, want in checks:
        if got.shape != want.shape or not np.array_equal(got, want):
            return f"hand-worked {name}: got {got.tolist()} want {want.tolist()}"
    return None


def pin_brute_force(orc, seed=11):
    """Scalar loops over the index definitions on a tiny pack (3 jobs, ranks 1..3)."""
    rng = np.random.default_rng(seed)
    d_in, d_out = 4, 3
    segs, N = _rand_segs(orc, rng, d_in, d_out, [1, 3, 2], [2, 1, 3])
    X = rng.standard_normal((N, d_in))
    W = rng.standard_normal((d_in, d_out))
    dY = rng.standard_normal((N, d_out))
    Y, _ = orc.forward(X, W, segs)
    dX, dA, dB, _ = orc.backward(X, W, dY, segs)
    for sg_i, sg in enumerate(segs):
        s = sg.alpha / sg.r
        for n in range(sg.offset, sg.offset + sg.n):
            for k in range(d_out):
                acc = 0.0
                for d in range(d_in):
                    acc += X[n, d] * W[d, k]
                for t in range(sg.r):
                    h = 0.0
                    for d in range(d_in):
                        h += X[n, d] * sg.A[d, t]
                    acc += s * h * sg.B[t, k]
                if abs(acc - Y[n, k]) > 1e-12 * (1 + abs(acc)):
                    return f"brute force Y[{n},{k}]"
        # gradients of L = sum_{n,k} Y[n,k] dY[n,k], by index
        for d in range(d_in):
            for t in range(sg.r):
                acc = 0.0
                for n in range(sg.offset, sg.offset + sg.n):
                    for k in range(d_out):
                        acc += dY[n, k] * s * X[n, d] * sg.B[t, k]
                if abs(acc - dA[sg_i][d, t]) > 1e-12 * (1 + abs(acc)):
                    return f"brute force dA{sg_i}[{d},{t}]"
        for t in range(sg.r):
            for k in range(d_out):
                acc = 0.0
                for n in range(sg.offset, sg.offset + sg.n):
                    h = sum(X[n, d] * sg.A[d, t] for d in range(d_in))
                    acc += dY[n, k] * s * h
                if abs(acc - dB[sg_i][t, k]) > 1e-12 * (1 + abs(acc)):
                    return f"brute force dB{sg_i}[{t},{k}]"
        for n in range(sg.offset, sg.offset + sg.n):
            for d in range(d_in):
                acc = 0.0
                for k in range(d_out):
                    acc += dY[n, k] * W[d, k]
                    for t in range(sg.r):
                        acc += dY[n, k] * s * sg.A[d, t] * sg.B[t, k]
                if abs(acc - dX[n, d]) > 1e-12 * (1 + abs(acc)):
                    return f"brute force dX[{n},{d}]"
    return None


def pin_explicit_product(orc, seed=12):
    """Y_i = X_i (W + s_i A_i B_i) with the d_in x d_out update formed explicitly."""
    rng = np.random.default_rng(seed)
    d_in, d_out = 24, 16
    segs, N = _rand_segs(orc, rng, d_in, d_out, [3, 1, 7, 4], [5, 9, 2, 6])
    X = rng.standard_normal((N, d_in))
    W = rng.standard_normal((d_in, d_out))
    Y, _ = orc.forward(X, W, segs)
    for sg in segs:
        dW = (sg.alpha / sg.r) * (sg.A @ sg.B)
        want = X[sg.offset:sg.offset + sg.n] @ (W + dW)
        if _rel(Y[sg.offset:sg.offset + sg.n], want) > 1e-13:
            return "explicit-product identity"
    # and the rows API agrees with the packed one
    rows = np.array([0, 4, 5, 13, 15, 21])
    if _rel(orc.forward_rows(X[rows], rows, W, segs), Y[rows]) > 1e-13:
        return "forward_rows disagrees with forward"
    dY = rng.standard_normal((N, d_out))
    dX, _, _, _ = orc.backward(X, W, dY, segs)
    if _rel(orc.backward_rows(dY[rows], rows, W, segs), dX[rows]) > 1e-13:
        return "backward_rows disagrees with backward"
    for sg in segs:
        dWt = (sg.alpha / sg.r) * (sg.A @ sg.B)
        want = dY[sg.offset:sg.offset + sg.n] @ (W + dWt).T
        if _rel(dX[sg.offset:sg.offset + sg.n], want) > 1e-13:
            return "explicit-product identity (dX)"
    return None


def pin_special_cases(orc, seed=13):
    """B=0 -> Y = XW and dA = 0; A=0 -> dB = 0 and dX = dY W^T; W=0 isolates the LoRA term."""
    rng = np.random.default_rng(seed)
    d_in, d_out = 20, 12
    segs, N = _rand_segs(orc, rng, d_in, d_out, [2, 5], [7, 4])
    X = rng.standard_normal((N, d_in))
    W = rng.standard_normal((d_in, d_out))
    dY = rng.standard_normal((N, d_out))
    base = X @ W
    zB = [orc.Seg(s.offset, s.n, s.A, np.zeros_like(s.B), s.alpha) for s in segs]
    Y, _ = orc.forward(X, W, zB)
    if _rel(Y, base) > 1e-14:
        return "B=0 forward is not XW"
    _, dA, _, _ = orc.backward(X, W, dY, zB)
    if any(np.any(a != 0) for a in dA):
        return "B=0 gives nonzero dA"
    zA = [orc.Seg(s.offset, s.n, np.zeros_like(s.A), s.B, s.alpha) for s in segs]
    dX, _, dB, _ = orc.backward(X, W, dY, zA)
    if any(np.any(b != 0) for b in dB):
        return "A=0 gives nonzero dB"
    if _rel(dX, dY @ W.T) > 1e-14:
        return "A=0 dX is not dY W^T"
    Y0, _ = orc.forward(X, np.zeros_like(W), segs)
    for sg in segs:
        want = (sg.alpha / sg.r) * (X[sg.offset:sg.offset + sg.n] @ sg.A) @ sg.B
        if _rel(Y0[sg.offset:sg.offset + sg.n], want) > 1e-13:
            return "W=0 forward is not the rank-r term"
    return None


def pin_packed_equals_separate(orc, seed=14):
    rng = np.random.default_rng(seed)
    d_in, d_out = 16, 10
    segs, N = _rand_segs(orc, rng, d_in, d_out, [4, 1, 6], [3, 8, 5])
    X = rng.standard_normal((N, d_in))
    W = rng.standard_normal((d_in, d_out))
    dY = rng.standard_normal((N, d_out))
    Y, _ = orc.forward(X, W, segs)
    dX, dA, dB, _ = orc.backward(X, W, dY, segs)
    for i, sg in enumerate(segs):
        rows = slice(sg.offset, sg.offset + sg.n)
        alone = [orc.Seg(0, sg.n, sg.A, sg.B, sg.alpha)]
        Yi, _ = orc.forward(X[rows], W, alone)
        dXi, dAi, dBi, _ = orc.backward(X[rows], W, dY[rows], alone)
        if _rel(Yi, Y[rows]) > 1e-14 or _rel(dXi, dX[rows]) > 1e-14:
            return f"job {i}: packed != separate (Y/dX)"
        if _rel(dAi[0], dA[i]) > 1e-14 or _rel(dBi[0], dB[i]) > 1e-14:
            return f"job {i}: packed != separate (dA/dB)"
    return None


def pin_finite_differences(orc, seed=15):
    """Central differences of L = <Y, dY> (d=8, ranks 1..3, 5 tokens per job, h=1e-6)."""
    rng = np.random.default_rng(seed)
    d_in = d_out = 8
    segs, N = _rand_segs(orc, rng, d_in, d_out, [1, 2, 3], [5, 5, 5])
    X = rng.standard_normal((N, d_in))
    W = rng.standard_normal((d_in, d_out))
    dY = rng.standard_normal((N, d_out))
    h = 1e-6

    def loss(X_, segs_):
        Y, _ = orc.forward(X_, W, segs_)
        return float(np.sum(Y * dY))

    dX, dA, dB, _ = orc.backward(X, W, dY, segs)
    fd = np.zeros_like(X)
    for idx in np.ndindex(*X.shape):
        Xp = X.copy(); Xp[idx] += h
        Xm = X.copy(); Xm[idx] -= h
        fd[idx] = (loss(Xp, segs) - loss(Xm, segs)) / (2 * h)
    if _rel(dX, fd) > 1e-7:
        return f"finite differences dX rel {_rel(dX, fd):.2e}"
    for i, sg in enumerate(segs):
        for name, mat, grad in (("A", sg.A, dA[i]), ("B", sg.B, dB[i])):
            fdm = np.zeros_like(mat)
            for idx in np.ndindex(*mat.shape):
                def with_delta(delta):
                    m2 = mat.copy(); m2[idx] += delta
                    s2 = list(segs)
                    s2[i] = orc.Seg(sg.offset, sg.n, m2 if name == "A" else sg.A, m2 if name == "B" else sg.B, sg.alpha)
                    return loss(X, s2)
                fdm[idx] = (with_delta(h) - with_delta(-h)) / (2 * h)
            if _rel(grad, fdm) > 1e-7:
                return f"finite differences d{name}{i} rel {_rel(grad, fdm):.2e}"
    return None


def pin_autograd(orc, seed=16):
    """torch.autograd (fp64) differentiates the layer built from torch ops."""
    import torch
    rng = np.random.default_rng(seed)
    d_in, d_out = 12, 9
    segs, N = _rand_segs(orc, rng, d_in, d_out, [2, 4, 1], [6, 3, 7])
    X = rng.standard_normal((N, d_in))
    W = rng.standard_normal((d_in, d_out))
    dY = rng.standard_normal((N, d_out))
    tX = torch.tensor(X, requires_grad=True)
    tW = torch.tensor(W)
    tA = [torch.tensor(s.A, requires_grad=True) for s in segs]
    tB = [torch.tensor(s.B, requires_grad=True) for s in segs]
    lin = torch.nn.functional.linear
    outs = []
    for s, a, b in zip(segs, tA, tB):
        xi = tX[s.offset:s.offset + s.n]
        outs.append(lin(xi, tW.T) + (s.alpha / s.r) * lin(lin(xi, a.T), b.T))
    torch.cat(outs).backward(torch.tensor(dY))
    dX, dA, dB, _ = orc.backward(X, W, dY, segs)
    if _rel(dX, tX.grad.numpy()) > 1e-13:
        return "autograd dX"
    for i in range(len(segs)):
        if _rel(dA[i], tA[i].grad.numpy()) > 1e-13 or _rel(dB[i], tB[i].grad.numpy()) > 1e-13:
            return f"autograd dA/dB job {i}"
    H, dH, dA2, dB2 = orc.lora_grads(X, dY, segs)
    for i in range(len(segs)):
        if _rel(dA2[i], dA[i]) > 1e-14 or _rel(dB2[i], dB[i]) > 1e-14:
            return f"lora_grads disagrees with backward, job {i}"
    return None


def pin_linearity(orc, seed=17):
    rng = np.random.default_rng(seed)
    d_in, d_out = 10, 6
    segs, N = _rand_segs(orc, rng, d_in, d_out, [3, 2], [4, 5])
    X = rng.standard_normal((N, d_in))
    W = rng.standard_normal((d_in, d_out))
    dY = rng.standard_normal((N, d_out))
    c = -2.5
    g1 = orc.backward(X, W, dY, segs)
    g2 = orc.backward(X, W, c * dY, segs)
    if _rel(g2[0], c * g1[0]) > 1e-14:
        return "dX not linear in dY"
    for a1, a2 in zip(g1[1] + g1[2], g2[1] + g2[2]):
        if _rel(a2, c * a1) > 1e-14:
            return "dA/dB not linear in dY"
    return None


# ---------------------------------------------------------------- AdamW

def pin_adamw_hand_worked(orc):
    g = _parse_golden("hand_worked_adamw.txt")
    f = {k: float(v) for k, v in g.items()}
    hp = (f["lr"], f["beta1"], f["beta2"], f["eps"], f["weight_decay"])
    p, m, v = orc.adamw(np.array([f["p0"]]), np.array([f["g1"]]), np.zeros(1), np.zeros(1), *hp, 1)
    close = lambda a, b: abs(a - b) <= 1e-14 * abs(b)
    if not (close(p[0], f["p1"]) and close(m[0], f["m1"]) and close(v[0], f["v1"])):
        return f"AdamW t=1: {p[0]!r} {m[0]!r} {v[0]!r}"
    p, m, v = orc.adamw(p, np.array([f["g2"]]), m, v, *hp, 2)
    if not (close(p[0], f["p2"]) and close(m[0], f["m2"]) and close(v[0], f["v2"])):
        return f"AdamW t=2: {p[0]!r} {m[0]!r} {v[0]!r}"
    return None


def pin_adamw_closed_form(orc, seed=18):
    """t = 1 from zero moments: p' = p (1 - lr wd) - lr g / (|g| + eps)."""
    rng = np.random.default_rng(seed)
    p = rng.standard_normal(1000)
    g = rng.standard_normal(1000) * 1e-3
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.01
    p2, m2, v2 = orc.adamw(p, g, np.zeros_like(p), np.zeros_like(p), lr, b1, b2, eps, wd, 1)
    want = p * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    if np.max(np.abs(p2 - want)) > 1e-15:
        return "AdamW t=1 closed form"
    return None


def pin_adamw_torch(orc, seed=19):
    """torch.optim.AdamW in fp64 over three steps with fresh gradients."""
    import torch
    rng = np.random.default_rng(seed)
    p0 = rng.standard_normal(257)
    lr, b1, b2, eps, wd = 3e-3, 0.8, 0.95, 1e-6, 0.1
    tp = torch.nn.Parameter(torch.tensor(p0))
    opt = torch.optim.AdamW([tp], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    for t in (1, 2, 3):
        g = rng.standard_normal(257) * 10.0 ** (-t)
        tp.grad = torch.tensor(g)
        opt.step()
        p, m, v = orc.adamw(p, g, m, v, lr, b1, b2, eps, wd, t)
        st = opt.state[tp]
        if (_rel(p, tp.detach().numpy()) > 1e-13 or _rel(m, st["exp_avg"].numpy()) > 1e-13
                or _rel(v, st["exp_avg_sq"].numpy()) > 1e-13):
            return f"AdamW vs torch at t={t}"
    return None


def pin_dequantize_w4(orc):
    """Hand-worked codes: byte 0x7F holds code -1 (low nibble, even k) and code 7 (high nibble);
    0x80 holds 0 and -8; 0x08 holds -8 and 0.  Columns k < 64 use scale row 0, k >= 64 row 1."""
    d_out, d_in = 2, 128
    Wq = np.zeros((d_out, d_in // 2), dtype=np.uint8)
    Wq[0, 0] = 0x7F          # k=0: -1, k=1: 7
    Wq[0, 40] = 0x80         # k=80 (byte 40, low): 0, k=81: -8
    Wq[1, 10] = 0x08         # k=20: -8, k=21: 0
    Wq[1, 63] = 0x5A         # k=126: 0xA -> -6, k=127: 5
    Ws = np.array([[0.5, 2.0], [0.25, 4.0]])
    W = orc.dequantize_w4(Wq, Ws)
    want = {(0, 0): -0.5, (1, 0): 3.5, (80, 0): 0.0, (81, 0): -2.0, (20, 1): -16.0, (21, 1): 0.0,
            (126, 1): -24.0, (127, 1): 20.0, (2, 0): 0.0, (64, 1): 0.0}
    if W.shape != (d_in, d_out):
        return f"dequantize_w4 shape {W.shape}"
    for (k, o), v in want.items():
        if W[k, o] != v:
            return f"dequantize_w4 W[{k},{o}] = {W[k, o]}, want {v}"
    full = orc.dequantize_w4(np.full((3, 64), 0x88, dtype=np.uint8), np.full((2, 3), 0.125))
    if not np.all(full == -1.0):
        return "dequantize_w4: all codes -8 at scale 1/8 must give -1"
    return None


ALL_PINS = [pin_hand_worked, pin_brute_force, pin_explicit_product, pin_special_cases,
            pin_packed_equals_separate, pin_finite_differences, pin_autograd, pin_linearity,
            pin_adamw_hand_worked, pin_adamw_closed_form, pin_adamw_torch, pin_dequantize_w4]
