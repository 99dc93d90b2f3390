"""An independent float64 restatement of the AttnRes mixture, for pinning the
oracle at tiny hidden sizes.

It is written differently from the oracle on purpose: whole-array numpy, rows
normalised first and dotted second, the softmax taken from scipy, the bf16
rounding of the current-layer row done through a float32 add and the usual
bit trick.  Definition followed: the implementation walkthrough of the
vllm-ascend Kimi K3 attention-residual fusion PR (#14840) -- candidates are the
valid bank rows then the current-layer row; RMS-normalise each, score against
norm.weight * proj.weight, softmax, weighted sum of the raw rows -- and the
output RMSNorm of the vllm #54261 kernel excerpt.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
from scipy.special import softmax


def widen(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_round_via_f32(x32: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
            >> np.uint32(16)).astype(np.uint16)


def restate(prefix, delta, blocks, S, res_w, rms_w, out_norm_w, eps, out_eps):
    """Returns (c_bits [T,H], weights [T,N], logits [T,N], y [T,H] float64
    before the final bf16 rounding)."""
    eps = float(np.float32(eps))
    out_eps = float(np.float32(out_eps))
    H = res_w.shape[0]
    P32 = widen(prefix[:, :H]).astype(np.float32)
    if delta is not None:
        c_bits = bf16_round_via_f32(P32 + widen(delta[:, :H]).astype(np.float32))
    else:
        c_bits = np.ascontiguousarray(prefix[:, :H])
    rows = [widen(blocks[:, i, :H]) for i in range(S)] + [widen(c_bits)]
    X = np.stack(rows, axis=1)                      # [T, N, H]
    q = widen(rms_w) * widen(res_w)                 # [H]
    rms = np.sqrt(np.mean(X * X, axis=2) + eps)     # [T, N]
    Xhat = X / rms[:, :, None]
    L = Xhat @ q                                    # [T, N]
    W = softmax(L, axis=1)
    acc = np.einsum("tn,tnh->th", W, X)
    if out_norm_w is not None:
        r = np.sqrt(np.mean(acc * acc, axis=1) + out_eps)
        y = acc / r[:, None] * widen(out_norm_w)[None, :]
    else:
        y = acc
    return c_bits, W, L, y


# ---- correct rounding checks, exact rational arithmetic ------------------

def _all_finite_bf16():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)     # +0 .. largest finite
    vals = [Fraction(float(v)) for v in (bits << 16).view(np.float32)]
    return bits.astype(np.uint16), vals


_POS = None


def bf16_rne_exact(x: float) -> int:
    """Round a double to bf16 by exhaustive search over the positive finite
    bf16 values, ties to even, IEEE overflow rule.  Slow; for pins only."""
    global _POS
    if _POS is None:
        _POS = _all_finite_bf16()
    bits, vals = _POS
    if np.isnan(x):
        return None
    sign = 0x8000 if np.signbit(x) else 0
    if np.isinf(x):
        return sign | 0x7F80
    a = Fraction(abs(float(x)))
    maxv = vals[-1]
    # midpoint between the largest finite value and 2^128
    over = maxv + (Fraction(2) ** 128 - maxv) / 2
    if a >= over:
        return sign | 0x7F80
    # binary search for the largest value <= a
    lo, hi = 0, len(vals) - 1
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if vals[mid] <= a:
            lo = mid
        else:
            hi = mid - 1
    below = lo
    if vals[below] == a or below == len(vals) - 1:
        return sign | int(bits[below])
    above = below + 1
    db = a - vals[below]
    da = vals[above] - a
    if db < da:
        pick = below
    elif da < db:
        pick = above
    else:
        pick = below if (int(bits[below]) & 1) == 0 else above
    return sign | int(bits[pick])


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (the gap above |v|'s binade floor)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def is_nearest_bf16(out_bits: np.ndarray, y: np.ndarray, rel_slack: float = 1e-12) -> np.ndarray:
    """True where out_bits is a nearest bf16 value to y (up to a tiny slack
    for y's own double rounding)."""
    o = widen(out_bits)
    b = np.asarray(out_bits, dtype=np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    sign = b & 0x8000
    up = sign | np.minimum(mag + 1, 0x7F7F)
    # one step toward (and, from zero, across) zero
    dn = np.where(mag == 0, (sign ^ 0x8000) | 1, sign | np.maximum(mag - 1, 0))
    ou = widen(up.astype(np.uint16))
    od = widen(dn.astype(np.uint16))
    err = np.abs(o - y)
    slack = rel_slack * np.abs(y) + 1e-300
    return (err <= np.abs(ou - y) + slack) & (err <= np.abs(od - y) + slack)
