"""The kernels' activation device functions against the float64 oracle's
definitions (through the library's activation test hook).

Precise flavour (float32 CUDA-core path): CUDA's erff / tanhf / expf, within
float32 rounding.  Fast flavour (bf16 tensor-core path): one tanh.approx.f32
per element, whose relative error is about 2^-11 (taken here as 2^-10.9); for
GELU-erf also the fitted tanh form of the Gaussian CDF (max error 3.4e-4 for
the value, 6.7e-4 for the derivative, in exact arithmetic).  With t = tanh(u)
in error by e|t|, e = 2^-10.9, the value x/2 (1 + t) is off by at most
|x|/2 e and the derivative (1 + t)/2 + x/2 (1 - t^2) u' by at most
e/2 + |x| e |u'|; the bounds below are those plus the fit error.
"""

import numpy as np
import pytest

from oracle import ref

pytestmark = pytest.mark.gpu

E = 2.0 ** -10.9


@pytest.fixture(scope="module")
def gd():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import recommender_model_attention_gb300 as g
    g.build()
    return g


def _grid():
    x = np.concatenate([np.linspace(-8.0, 8.0, 16001), [-30.0, -15.0, -9.5, 9.5, 15.0, 30.0, 0.0]])
    return x.astype(np.float32)


def _run(gd, act, fast):
    import torch
    x = _grid()
    y, dy = gd.act_eval(torch.from_numpy(x).cuda(), act, fast)
    torch.cuda.synchronize()
    xr = x.astype(np.float64)
    want = np.array([ref.act(act, v) for v in xr])
    dwant = np.array([ref.dact(act, v) for v in xr])
    return xr, y.cpu().double().numpy(), dy.cpu().double().numpy(), want, dwant


@pytest.mark.parametrize("act", ["gelu_erf", "gelu_tanh", "silu", "gelu_taylor6", "identity"])
def test_precise_flavour(gd, act):
    x, y, dy, want, dwant = _run(gd, act, False)
    scale = np.maximum(1.0, np.abs(want))
    assert np.max(np.abs(y - want) / scale) <= 2e-6
    dscale = np.maximum(1.0, np.abs(dwant))
    assert np.max(np.abs(dy - dwant) / dscale) <= 2e-6


def _u_prime(act, x):
    if act == "gelu_erf":
        return 0.7999136459 + 3 * 0.0349731511 * x * x
    if act == "gelu_tanh":
        return np.sqrt(2 / np.pi) * (1 + 3 * 0.044715 * x * x)
    return np.full_like(x, 0.5)   # silu: u = x / 2


@pytest.mark.parametrize("act,fit,dfit", [("gelu_erf", 3.4e-4, 6.7e-4), ("gelu_tanh", 0.0, 0.0),
                                          ("silu", 0.0, 0.0)])
def test_fast_flavour_tanh_forms(gd, act, fit, dfit):
    x, y, dy, want, dwant = _run(gd, act, True)
    bound = fit + 0.5 * np.abs(x) * E + 1e-6 * np.maximum(1, np.abs(want))
    assert np.all(np.abs(y - want) <= bound), float(np.max(np.abs(y - want) - bound))
    dbound = dfit + 0.5 * E + np.abs(x) * E * _u_prime(act, x) + 1e-6
    assert np.all(np.abs(dy - dwant) <= dbound), float(np.max(np.abs(dy - dwant) - dbound))
    # saturation: far tails are exact limits (0 and x for the value, 0 and 1
    # for the derivative) within float32 rounding
    far = np.abs(x) >= 9.5
    assert np.all(np.abs(y[far] - want[far]) <= 1e-6 * np.abs(want[far]) + 1e-6)
    assert np.all(np.abs(dy[far] - dwant[far]) <= 1e-5)


@pytest.mark.parametrize("act", ["gelu_taylor6", "identity"])
def test_fast_flavour_polynomials(gd, act):
    x, y, dy, want, dwant = _run(gd, act, True)
    assert np.max(np.abs(y - want) / np.maximum(1.0, np.abs(want))) <= 2e-6
    assert np.max(np.abs(dy - dwant) / np.maximum(1.0, np.abs(dwant))) <= 2e-6


@pytest.mark.parametrize("act", ["gelu_erf", "gelu_tanh", "silu", "gelu_taylor6", "identity"])
@pytest.mark.parametrize("odd", [False, True])
def test_pair_form_is_the_scalar_form_bit_for_bit(gd, act, odd):
    """The tensor-core kernels evaluate the activation two scores at a time
    in f32x2 arithmetic: lane by lane the same operations as the scalar form
    (the derivative's 1 - t^2 formed as t^2 - 1 with the sign carried by -u',
    both exact negations), so every value and derivative must match the
    scalar form's bits, including the tails, signed zeros and an odd last
    element paired with itself.  The hook also checks in the kernel that the
    value of the value-and-derivative pair form (the backward's P) has the
    bits of the value-only pair form (the forward's), writing NaN where not."""
    import torch
    x = _grid()
    rng = np.random.default_rng(7)
    x = np.concatenate([x, rng.standard_normal(4001).astype(np.float32) * 3,
                        np.float32([-0.0, 1e-30, -1e-30, 3e38, -3e38])])
    if (x.size % 2 == 1) != odd:
        x = x[:-1]
    xt = torch.from_numpy(x).cuda()
    y1, d1 = gd.act_eval(xt, act, True)
    y2, d2 = gd.act_eval(xt, act, 2)
    torch.cuda.synchronize()
    b = lambda t: t.cpu().numpy().view(np.uint32)
    assert np.array_equal(b(y1), b(y2)), act
    assert np.array_equal(b(d1), b(d2)), act
