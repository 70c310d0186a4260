"""RMSNorm prologue of GDPA, restated in float64.  TEST INFRASTRUCTURE ONLY
(see the package docstring).

The GEM page ("GEM 트레이닝: Meta가 LLM 규모의 광고 파운데이션 모델 효율성을
두 배로 높인 방법", techlist.io, section on why high GPU utilisation is hard
for recommendation models) counts the normalisation layers among the
memory-bound operations; the GDPA page (the caption of its chart comparing
tanh GELU with the 6th-order Taylor form) has RMSNorm keep the activation's
inputs in the polynomial's accurate range.  A fused prologue applies the
norm to Q and K inside the attention instead of in a separate pass.  Per
(token, head) row of d values, with a scalar gain g and eps:

    r = sqrt(mean(x^2) + eps),   y = g x / r,

and, given dL/dy, the row's gradient

    dL/dx = (g / r) (dy - x (x . dy) / (d r^2)).

The fused variant's oracle is GDPA on the normalised Q and K (V as given),
its gradients the GDPA gradients of the normalised inputs pulled back
through the norm.
"""

from __future__ import annotations

import numpy as np

from . import ref


def rmsnorm(x, gain: float = 1.0, eps: float = 1e-6) -> np.ndarray:
    """y = gain * x / sqrt(mean(x^2) + eps) over the last axis."""
    x = ref.to_f64(x)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return gain * x / r


def rmsnorm_bwd(x, dy, gain: float = 1.0, eps: float = 1e-6) -> np.ndarray:
    """dL/dx of y = rmsnorm(x) given dL/dy (the formula in the docstring)."""
    x = ref.to_f64(x)
    dy = ref.to_f64(dy)
    d = x.shape[-1]
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    xdy = np.sum(x * dy, axis=-1, keepdims=True)
    return (gain / r) * (dy - x * xdy / (d * r * r))


def fwd(q_off, kv_off, q_raw, k_raw, v, alpha: float, act: str, gain: float = 1.0,
        eps: float = 1e-6, mask: str = "none", window: int = 0) -> np.ndarray:
    """O of GDPA with the RMSNorm prologue on Q and K."""
    return ref.fwd(q_off, kv_off, rmsnorm(q_raw, gain, eps), rmsnorm(k_raw, gain, eps), v,
                   alpha, act, mask, window)


def bwd(q_off, kv_off, q_raw, k_raw, v, do, alpha: float, act: str, gain: float = 1.0,
        eps: float = 1e-6, mask: str = "none", window: int = 0):
    """(dQ_raw, dK_raw, dV) of the same."""
    qn, kn = rmsnorm(q_raw, gain, eps), rmsnorm(k_raw, gain, eps)
    dq, dk, dv = ref.bwd(q_off, kv_off, qn, kn, v, do, alpha, act, mask, window)
    return rmsnorm_bwd(q_raw, dq, gain, eps), rmsnorm_bwd(k_raw, dk, gain, eps), dv
