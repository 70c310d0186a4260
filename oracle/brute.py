"""Dense, padded NumPy float64 formulation of GDPA (TEST INFRASTRUCTURE ONLY).

Every sample is padded to [Lq_max, Lkv_max] and an explicit boolean mask
selects the valid (query, key) pairs, so the jagged bookkeeping of the C
loops is checked against whole-matrix algebra on small inputs:

    X  = alpha * Q K^T            (per sample, per head)
    P  = act(X) * M               (M: valid pairs)
    O  = P V
    G  = (dO V^T) * act'(X) * M
    dV = P^T dO,  dQ = alpha G K,  dK = alpha G^T Q

The activations are evaluated through SciPy's special functions (normal CDF,
logistic, softmax for the softmax variant) rather than the formulas used by
the C loops.
"""

from __future__ import annotations

import math

import numpy as np
from scipy import special


def act(kind: str, x: np.ndarray) -> np.ndarray:
    if kind == "gelu_erf":
        return x * special.ndtr(x)
    if kind == "gelu_tanh":
        u = math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)
        return 0.5 * x * (1.0 + np.tanh(u))
    if kind == "silu":
        return x * special.expit(x)
    if kind == "gelu_taylor6":
        c = 1.0 / math.sqrt(2.0 * math.pi)
        # coefficients of x^0 .. x^6
        return np.polynomial.polynomial.polyval(x, [0.0, 0.5, c, 0.0, -c / 6.0, 0.0, c / 40.0])
    if kind == "identity":
        return x.copy()
    raise ValueError(kind)


def dact(kind: str, x: np.ndarray) -> np.ndarray:
    if kind == "gelu_erf":
        return special.ndtr(x) + x * np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)
    if kind == "gelu_tanh":
        k = math.sqrt(2.0 / math.pi)
        t = np.tanh(k * (x + 0.044715 * x ** 3))
        return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * k * (1.0 + 3 * 0.044715 * x * x)
    if kind == "silu":
        s = special.expit(x)
        return s + x * s * (1.0 - s)
    if kind == "gelu_taylor6":
        c = 1.0 / math.sqrt(2.0 * math.pi)
        return np.polynomial.polynomial.polyval(x, [0.5, 2 * c, 0.0, -4 * c / 6.0, 0.0, 6 * c / 40.0])
    if kind == "identity":
        return np.ones_like(x)
    raise ValueError(kind)


def _pad(x, off, L):
    B = len(off) - 1
    out = np.zeros((B, L) + x.shape[1:], dtype=np.float64)
    for b in range(B):
        n = off[b + 1] - off[b]
        out[b, :n] = x[off[b]:off[b + 1]]
    return out


def _mask(q_off, kv_off, Lq, Lkv, mask, window):
    B = len(q_off) - 1
    i = np.arange(Lq)[:, None]
    j = np.arange(Lkv)[None, :]
    M = np.zeros((B, Lq, Lkv), dtype=bool)
    for b in range(B):
        lq = q_off[b + 1] - q_off[b]
        lkv = kv_off[b + 1] - kv_off[b]
        m = (i < lq) & (j < lkv)
        if mask == "causal_window":
            m &= (j <= i) & (j > i - window)
        M[b] = m
    return M


def _unpad(xp, off, T):
    out = np.zeros((T,) + xp.shape[2:], dtype=np.float64)
    for b in range(len(off) - 1):
        n = off[b + 1] - off[b]
        out[off[b]:off[b + 1]] = xp[b, :n]
    return out


def _setup(q_off, kv_off, q, k, v, mask, window):
    q_off = np.asarray(q_off, dtype=np.int64)
    kv_off = np.asarray(kv_off, dtype=np.int64)
    Lq = int(max(1, np.max(np.diff(q_off), initial=0)))
    Lkv = int(max(1, np.max(np.diff(kv_off), initial=0)))
    Qp = _pad(np.asarray(q, np.float64), q_off, Lq)     # [B, Lq, H, d]
    Kp = _pad(np.asarray(k, np.float64), kv_off, Lkv)
    Vp = _pad(np.asarray(v, np.float64), kv_off, Lkv)
    M = _mask(q_off, kv_off, Lq, Lkv, mask, window)[:, None]  # [B, 1, Lq, Lkv]
    return q_off, kv_off, Lq, Lkv, Qp, Kp, Vp, M


def fwd(q_off, kv_off, q, k, v, alpha, kind, mask="none", window=0):
    q_off, kv_off, Lq, Lkv, Qp, Kp, Vp, M = _setup(q_off, kv_off, q, k, v, mask, window)
    X = alpha * np.einsum("bihc,bjhc->bhij", Qp, Kp)
    if kind == "softmax":
        # SciPy's softmax over the key axis with masked scores at -inf; rows
        # with no valid key are all -inf (NaN from SciPy) and are set to 0
        Xm = np.where(M, X, -np.inf)
        with np.errstate(invalid="ignore"):
            P = special.softmax(Xm, axis=-1)
        P = np.where(M, P, 0.0)
    else:
        P = np.where(M, act(kind, X), 0.0)
    Op = np.einsum("bhij,bjhc->bihc", P, Vp)
    return _unpad(Op, q_off, int(q_off[-1]))


def bwd(q_off, kv_off, q, k, v, do, alpha, kind, mask="none", window=0):
    if kind == "softmax":
        raise ValueError("the dense form has no softmax backward (finite differences pin it)")
    q_off, kv_off, Lq, Lkv, Qp, Kp, Vp, M = _setup(q_off, kv_off, q, k, v, mask, window)
    dOp = _pad(np.asarray(do, np.float64), q_off, Lq)
    X = alpha * np.einsum("bihc,bjhc->bhij", Qp, Kp)
    P = np.where(M, act(kind, X), 0.0)
    G = np.where(M, np.einsum("bihc,bjhc->bhij", dOp, Vp) * dact(kind, X), 0.0)
    dVp = np.einsum("bhij,bihc->bjhc", P, dOp)
    dQp = alpha * np.einsum("bhij,bjhc->bihc", G, Kp)
    dKp = alpha * np.einsum("bhij,bihc->bjhc", G, Qp)
    return (_unpad(dQp, q_off, int(q_off[-1])), _unpad(dKp, kv_off, int(kv_off[-1])),
            _unpad(dVp, kv_off, int(kv_off[-1])))
