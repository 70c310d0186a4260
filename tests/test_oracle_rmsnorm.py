"""Pins of the oracle's RMSNorm prologue (``oracle/rmsnorm.py``), CPU only:

* every normalised row has root mean square gain * rms / sqrt(rms^2 + eps)
  (exactly gain when eps = 0), and the norm ignores a positive rescaling of
  its row when eps = 0;
* with eps = 0 the row gradient is orthogonal to the row (the output does
  not change along x), a closed-form consequence the formula must meet;
* the row gradient against central differences of sum(y * dy);
* the fused GDPA gradients with respect to the raw Q and K against central
  differences of sum(O * dO), for two activations and the causal window.
"""

import numpy as np
import pytest

from oracle import rmsnorm as rn
from workloads import offsets_from_lengths


def test_rms_of_output_and_scale_invariance():
    g = np.random.default_rng(0)
    x = g.standard_normal((5, 3, 16)) * 3.0
    y = rn.rmsnorm(x, gain=1.7, eps=0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.7, rtol=1e-13)
    assert np.allclose(rn.rmsnorm(4.5 * x, 1.7, 0.0), y, rtol=1e-13)
    eps = 0.3
    y2 = rn.rmsnorm(x, 1.0, eps)
    ms = np.mean(x * x, axis=-1)
    assert np.allclose(np.sqrt(np.mean(y2 * y2, axis=-1)), np.sqrt(ms / (ms + eps)), rtol=1e-13)


def test_gradient_orthogonal_to_row_without_eps():
    g = np.random.default_rng(1)
    x = g.standard_normal((7, 2, 8))
    dy = g.standard_normal((7, 2, 8))
    dx = rn.rmsnorm_bwd(x, dy, gain=0.8, eps=0.0)
    assert np.allclose(np.sum(dx * x, axis=-1), 0.0, atol=1e-12)


def test_row_gradient_matches_central_differences():
    g = np.random.default_rng(2)
    x = g.standard_normal((3, 2, 6))
    dy = g.standard_normal((3, 2, 6))
    dx = rn.rmsnorm_bwd(x, dy, gain=1.3, eps=1e-2)
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (np.sum(rn.rmsnorm(xp, 1.3, 1e-2) * dy) -
                   np.sum(rn.rmsnorm(xm, 1.3, 1e-2) * dy)) / (2 * h)
    assert np.allclose(dx, fd, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("act,mask,window", [("gelu_erf", "none", 0), ("silu", "causal_window", 3),
                                             ("softmax", "none", 0)])
def test_fused_gradients_match_central_differences(act, mask, window):
    g = np.random.default_rng(3)
    lq, lkv = [3, 2], ([4, 5] if mask == "none" else [3, 2])
    qo, ko = offsets_from_lengths(np.array(lq)), offsets_from_lengths(np.array(lkv))
    q = g.standard_normal((qo[-1], 1, 4))
    k = g.standard_normal((ko[-1], 1, 4))
    v = g.standard_normal((ko[-1], 1, 4))
    do = g.standard_normal((qo[-1], 1, 4))
    kw = dict(gain=0.9, eps=1e-3, mask=mask, window=window)
    dq, dk, _ = rn.bwd(qo, ko, q, k, v, do, 0.7, act, **kw)

    def loss(qq, kk):
        return float(np.sum(rn.fwd(qo, ko, qq, kk, v, 0.7, act, **kw) * do))

    h = 1e-6
    for which, x, got in (("q", q, dq), ("k", k, dk)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            if which == "q":
                fd[idx] = (loss(xp, k) - loss(xm, k)) / (2 * h)
            else:
                fd[idx] = (loss(q, xp) - loss(q, xm)) / (2 * h)
        assert np.allclose(got, fd, rtol=1e-5, atol=1e-7), which
