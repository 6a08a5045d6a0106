"""The fp64 oracle against its pins (no GPU)."""
import types

import numpy as np
import pytest

from oracle import lora_oracle as orc
import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    assert pin(orc) is None


# ---------------------------------------------------------------- planted mistakes
# Each mutant is the oracle with one plausible mistake; some pin must catch it.

def _mutant(**over):
    ns = types.SimpleNamespace(Seg=orc.Seg, forward=orc.forward, backward=orc.backward,
                               forward_rows=orc.forward_rows, backward_rows=orc.backward_rows,
                               lora_grads=orc.lora_grads, adamw=orc.adamw, dequantize_w4=orc.dequantize_w4)
    for k, v in over.items():
        setattr(ns, k, v)
    return ns


class SegAlphaScale(orc.Seg):
    @property
    def s(self):                      # mistake: scale alpha instead of alpha / r
        return float(self.alpha)


def _fwd_no_lora(X, W, segs):
    Y, H = orc.forward(X, W, [orc.Seg(s.offset, s.n, s.A, np.zeros_like(s.B), s.alpha) for s in segs])
    return Y, [np.asarray(X, float)[s.offset:s.offset + s.n] @ s.A for s in segs]


def _bwd_dB_unscaled(X, W, dY, segs):
    dX, dA, dB, dH = orc.backward(X, W, dY, segs)
    return dX, dA, [b / s.s for b, s in zip(dB, segs)], dH


def _bwd_dX_base_only(X, W, dY, segs):
    dX, dA, dB, dH = orc.backward(X, W, dY, segs)
    return np.asarray(dY, float) @ np.asarray(W, float).T, dA, dB, dH


def _bwd_dA_unscaled(X, W, dY, segs):
    dX, dA, dB, dH = orc.backward(X, W, dY, segs)
    return dX, [a / s.s for a, s in zip(dA, segs)], dB, dH


def _fwd_row_shift(X, W, segs):
    # mistake: each job reads the rows one below its segment (wraps at the end)
    X = np.roll(np.asarray(X, float), -1, axis=0)
    return orc.forward(X, W, segs)


def _bwd_wrong_adapter(X, W, dY, segs):
    # mistake: job i's dH uses job (i+1)'s B when shapes allow, else its own
    out = orc.backward(X, W, dY, segs)
    swapped = []
    for i, s in enumerate(segs):
        j = (i + 1) % len(segs)
        B = segs[j].B if segs[j].B.shape == s.B.shape and j != i else -s.B
        swapped.append(orc.Seg(s.offset, s.n, s.A, B, s.alpha))
    dX, dA, _, dH = orc.backward(X, W, dY, swapped)
    return dX, dA, out[2], dH


def _adamw_no_bias_correction(p, g, m, v, lr, b1, b2, eps, wd, t):
    p = np.asarray(p, float) * (1 - lr * wd)
    m = b1 * np.asarray(m, float) + (1 - b1) * np.asarray(g, float)
    v = b2 * np.asarray(v, float) + (1 - b2) * np.asarray(g, float) ** 2
    return p - lr * m / (np.sqrt(v) + eps), m, v


def _adamw_decay_after(p, g, m, v, lr, b1, b2, eps, wd, t):
    p2, m2, v2 = orc.adamw(p, g, m, v, lr, b1, b2, eps, 0.0, t)
    return p2 * (1 - lr * wd), m2, v2


def _adamw_eps_in_sqrt(p, g, m, v, lr, b1, b2, eps, wd, t):
    p = np.asarray(p, float) * (1 - lr * wd)
    m = b1 * np.asarray(m, float) + (1 - b1) * np.asarray(g, float)
    v = b2 * np.asarray(v, float) + (1 - b2) * np.asarray(g, float) ** 2
    return p - lr * (m / (1 - b1 ** t)) / np.sqrt(v / (1 - b2 ** t) + eps), m, v


def _dq_unsigned(Wq, Ws):
    # mistake: codes read as unsigned 0..15
    Wq = np.asarray(Wq, dtype=np.uint8)
    nib = np.empty((Wq.shape[0], 2 * Wq.shape[1]))
    nib[:, 0::2] = Wq & 15
    nib[:, 1::2] = Wq >> 4
    return nib.T * np.repeat(np.asarray(Ws, float), 64, axis=0)


def _dq_swapped_nibbles(Wq, Ws):
    return orc.dequantize_w4(((np.asarray(Wq, dtype=np.uint8) >> 4) | (np.asarray(Wq, dtype=np.uint8) << 4)).astype(np.uint8), Ws)


MUTANTS = {
    "w4_codes_unsigned": _mutant(dequantize_w4=_dq_unsigned),
    "w4_nibbles_swapped": _mutant(dequantize_w4=_dq_swapped_nibbles),
    "scale_alpha_not_alpha_over_r": _mutant(Seg=SegAlphaScale),
    "forward_drops_lora_term": _mutant(forward=_fwd_no_lora),
    "dB_missing_scale": _mutant(backward=_bwd_dB_unscaled),
    "dA_missing_scale": _mutant(backward=_bwd_dA_unscaled),
    "dX_missing_lora_term": _mutant(backward=_bwd_dX_base_only),
    "forward_rows_off_by_one": _mutant(forward=_fwd_row_shift),
    "dH_uses_wrong_adapter": _mutant(backward=_bwd_wrong_adapter),
    "adamw_no_bias_correction": _mutant(adamw=_adamw_no_bias_correction),
    "adamw_decay_after_update": _mutant(adamw=_adamw_decay_after),
    "adamw_eps_inside_sqrt": _mutant(adamw=_adamw_eps_in_sqrt),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = MUTANTS[name]
    failures = []
    for pin in pins.ALL_PINS:
        try:
            r = pin(m)
        except Exception as e:          # a crash also counts as caught
            r = f"raised {type(e).__name__}"
        if r is not None:
            failures.append((pin.__name__, r))
    assert failures, f"no pin caught mutant {name}"
