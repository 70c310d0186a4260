"""Pins of the float64 oracle to facts outside itself (CPU only).

* the Taylor GELU against the constants printed on the GDPA page, against the
  Maclaurin series of x*Phi(x) derived symbolically, and within the
  alternating-series error bound of that series on |x| <= 2;
* each activation against a library routine or an identity it must satisfy,
  and each derivative against central differences;
* the C loops against a dense padded NumPy formulation (brute force), the
  associativity identity (identity activation), finite-difference gradients
  and closed-form special cases.
"""

import math
import os

import numpy as np
import pytest
from scipy import integrate, special

from oracle import brute, ref
from workloads import offsets_from_lengths, small_case

ACTS = ["gelu_erf", "gelu_tanh", "silu", "gelu_taylor6", "identity"]
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _vec(kind, xs, f=ref.act):
    return np.array([f(kind, float(x)) for x in xs])


# ---------------------------------------------------------------- activations

def test_taylor6_matches_page_constants():
    g = _golden("taylor6_page_constants.txt")
    c1, c2, c4, c6 = g["c1"][0], g["c2"][0], g["c4"][0], g["c6"][0]
    xs = np.linspace(-3, 3, 601)
    printed = c1 * xs + c2 * xs ** 2 + c4 * xs ** 4 + c6 * xs ** 6
    got = _vec("gelu_taylor6", xs)
    # the printed constants carry 10 decimals
    assert np.max(np.abs(got - printed) / (1 + xs ** 6)) < 2e-10


def test_taylor6_is_truncated_maclaurin_series_of_erf_gelu():
    sympy = pytest.importorskip("sympy")
    x = sympy.symbols("x")
    gelu = x * (1 + sympy.erf(x / sympy.sqrt(2))) / 2
    series = sympy.series(gelu, x, 0, 7).removeO()
    poly = sympy.lambdify(x, series, "math")
    for xv in np.linspace(-2.5, 2.5, 51):
        assert abs(ref.act("gelu_taylor6", xv) - poly(float(xv))) < 1e-12 * (1 + xv ** 6)


def test_taylor6_error_bound_against_erf_gelu():
    # x*Phi(x) = x/2 + (x^2 - x^4/6 + x^6/40 - x^8/336 + ...)/sqrt(2 pi); for
    # |x| <= 2 the terms alternate and shrink, so the error of the cut after
    # x^6 is at most the first omitted term.
    xs = np.linspace(-2, 2, 4001)
    exact = xs * special.ndtr(xs)
    err = np.abs(_vec("gelu_taylor6", xs) - exact)
    bound = xs ** 8 / (336 * math.sqrt(2 * math.pi))
    assert np.all(err <= bound + 1e-15)
    for xv, expect in ((0.5, 4.53e-6), (1.0, 1.081e-3), (2.0, 0.2157)):
        e = abs(ref.act("gelu_taylor6", xv) - xv * special.ndtr(xv))
        assert abs(e - expect) < 0.01 * expect
    assert ref.act("gelu_taylor6", 0.0) == 0.0
    assert abs(ref.dact("gelu_taylor6", 0.0) - 0.5) < 1e-15


def test_gelu_erf_against_normal_cdf():
    xs = np.linspace(-8, 8, 321)
    assert np.max(np.abs(_vec("gelu_erf", xs) - xs * special.ndtr(xs))) < 1e-14
    # Phi by quadrature of the normal density, independent of erf
    for xv in (-2.5, -0.3, 0.0, 0.7, 3.1):
        phi_int, _ = integrate.quad(lambda t: math.exp(-t * t / 2) / math.sqrt(2 * math.pi),
                                    -math.inf, xv)
        assert abs(ref.act("gelu_erf", xv) - xv * phi_int) < 1e-10


def test_gelu_tanh_properties():
    xs = np.linspace(-8, 8, 1601)
    t = _vec("gelu_tanh", xs)
    # the tanh fit stays within 1e-3 of x*Phi(x) everywhere; dropping the cubic
    # term or flipping its sign breaks this by more than 1e-2
    assert np.max(np.abs(t - xs * special.ndtr(xs))) < 1e-3
    # tanh is odd, so gelu(x) - gelu(-x) = x
    assert np.max(np.abs(t - t[::-1] - xs)) < 1e-13
    assert abs(ref.act("gelu_tanh", 30.0) - 30.0) < 1e-12
    assert abs(ref.act("gelu_tanh", -30.0)) < 1e-12


def test_silu_against_logistic():
    xs = np.linspace(-30, 30, 601)
    s = _vec("silu", xs)
    assert np.max(np.abs(s - xs * special.expit(xs)) / (1 + np.abs(xs))) < 1e-15
    assert np.max(np.abs(s - 0.5 * xs * (1 + np.tanh(xs / 2))) / (1 + np.abs(xs))) < 1e-14


@pytest.mark.parametrize("kind", ACTS)
def test_activation_derivative_by_central_differences(kind):
    h = 1e-5
    for xv in np.linspace(-3, 3, 61):
        fd = (ref.act(kind, xv + h) - ref.act(kind, xv - h)) / (2 * h)
        assert abs(ref.dact(kind, xv) - fd) < 1e-8 * (1 + abs(fd))


def test_identity():
    for xv in (-3.5, 0.0, 2.25):
        assert ref.act("identity", xv) == xv
        assert ref.dact("identity", xv) == 1.0


# ---------------------------------------------------------------- loops vs brute force

def _rel(a, b):
    scale = max(np.max(np.abs(b)) if b.size else 0.0, 1e-300)
    return np.max(np.abs(a - b)) / scale if a.size else 0.0


@pytest.mark.parametrize("kind", ACTS)
@pytest.mark.parametrize("mask,window", [("none", 0), ("causal_window", 5), ("causal_window", 1)])
def test_loops_match_dense_brute_force(kind, mask, window):
    for seed in range(3):
        kv_range = None if mask == "causal_window" else (1, 16)
        c = small_case(seed, B=4, H=2, d=8, q_range=(1, 16), kv_range=kv_range,
                       zero_lengths=(seed == 2))
        args = (c["q_off"], c["kv_off"], c["q"].numpy(), c["k"].numpy(), c["v"].numpy())
        o = ref.fwd(*args, 0.7, kind, mask, window)
        ob = brute.fwd(*args, 0.7, kind, mask, window)
        assert _rel(o, ob) < 1e-12
        g = ref.bwd(*args, c["do"].numpy(), 0.7, kind, mask, window)
        gb = brute.bwd(*args, c["do"].numpy(), 0.7, kind, mask, window)
        for a, b in zip(g, gb):
            assert _rel(a, b) < 1e-12


def test_tiny_workload_matches_brute_force():
    from workloads import get_config, make_inputs
    w = get_config(0)
    x = make_inputs(w)
    args = (x["q_off"], x["kv_off"], x["q"].numpy(), x["k"].numpy(), x["v"].numpy())
    assert _rel(ref.fwd(*args, w.alpha, w.act), brute.fwd(*args, w.alpha, w.act)) < 1e-12
    g = ref.bwd(*args, x["do"].numpy(), w.alpha, w.act)
    gb = brute.bwd(*args, x["do"].numpy(), w.alpha, w.act)
    for a, b in zip(g, gb):
        assert _rel(a, b) < 1e-12


def test_associativity_identity_activation():
    # (alpha Q K^T) V = alpha Q (K^T V) per sample and head, with no mask
    c = small_case(11, B=5, H=3, d=16, q_range=(1, 40), kv_range=(1, 40))
    q, k, v = (c[n].numpy().astype(np.float64) for n in ("q", "k", "v"))
    o = ref.fwd(c["q_off"], c["kv_off"], q, k, v, 0.3, "identity")
    qo, ko = c["q_off"], c["kv_off"]
    for b in range(len(qo) - 1):
        for h in range(q.shape[1]):
            kv = k[ko[b]:ko[b + 1], h].T @ v[ko[b]:ko[b + 1], h]     # [d, d]
            expect = 0.3 * q[qo[b]:qo[b + 1], h] @ kv
            got = o[qo[b]:qo[b + 1], h]
            assert np.max(np.abs(got - expect)) <= 1e-12 * max(1.0, np.max(np.abs(expect)))


@pytest.mark.parametrize("kind", ACTS)
@pytest.mark.parametrize("mask,window", [("none", 0), ("causal_window", 2)])
def test_gradients_by_finite_differences(kind, mask, window):
    rng = np.random.Generator(np.random.PCG64(5))
    lq = np.array([3, 5]) if mask == "causal_window" else np.array([3, 4])
    lkv = lq.copy() if mask == "causal_window" else np.array([5, 2])
    qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
    H, d, alpha = 1, 4, 0.8
    q = rng.standard_normal((qo[-1], H, d))
    k = rng.standard_normal((ko[-1], H, d))
    v = rng.standard_normal((ko[-1], H, d))
    do = rng.standard_normal((qo[-1], H, d))
    dq, dk, dv = ref.bwd(qo, ko, q, k, v, do, alpha, kind, mask, window)

    def loss(qq, kk, vv):
        return float(np.sum(ref.fwd(qo, ko, qq, kk, vv, alpha, kind, mask, window) * do))

    h = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        base = [q, k, v]
        fd = np.zeros_like(base[which])
        for idx in np.ndindex(*fd.shape):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        assert np.max(np.abs(grad - fd)) <= 1e-6 * max(1.0, np.max(np.abs(fd)))


# ---------------------------------------------------------------- special cases

def test_single_key_sample():
    c = small_case(3, B=3, H=2, d=8, q_range=(2, 9), kv_range=(1, 1))
    q, k, v = (c[n].numpy().astype(np.float64) for n in ("q", "k", "v"))
    o = ref.fwd(c["q_off"], c["kv_off"], q, k, v, 0.5, "silu")
    for b in range(3):
        for h in range(2):
            k0, v0 = k[c["kv_off"][b], h], v[c["kv_off"][b], h]
            for t in range(c["q_off"][b], c["q_off"][b + 1]):
                x = 0.5 * float(q[t, h] @ k0)
                expect = x * special.expit(x) * v0
                assert np.max(np.abs(o[t, h] - expect)) < 1e-14


def test_one_hot_values_pick_activation_column():
    # V = one-hot(key index) makes O the matrix of activations itself
    lq = np.array([4, 6])
    lkv = np.array([3, 5])
    qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
    rng = np.random.Generator(np.random.PCG64(9))
    d = 8
    q = rng.standard_normal((qo[-1], 1, d))
    k = rng.standard_normal((ko[-1], 1, d))
    v = np.zeros((ko[-1], 1, d))
    for b in range(2):
        for j in range(lkv[b]):
            v[ko[b] + j, 0, j] = 1.0
    o = ref.fwd(qo, ko, q, k, v, 0.9, "gelu_erf")
    for b in range(2):
        for i in range(lq[b]):
            for j in range(d):
                if j < lkv[b]:
                    x = 0.9 * float(q[qo[b] + i, 0] @ k[ko[b] + j, 0])
                    assert abs(o[qo[b] + i, 0, j] - x * special.ndtr(x)) < 1e-14
                else:
                    assert o[qo[b] + i, 0, j] == 0.0


@pytest.mark.parametrize("L,W", [(1, 4), (3, 4), (4, 4), (10, 4), (700, 256), (2048, 256), (255, 256)])
def test_causal_window_pair_count_closed_form(L, W):
    expect = W * (W + 1) // 2 + (L - W) * W if L >= W else L * (L + 1) // 2
    off = np.array([0, L], dtype=np.int32)
    assert ref.pairs(off, off, "causal_window", W) == expect
    assert ref.pairs(off, off, "none", 0) == L * L


def test_empty_rows_are_zero():
    # Lkv = 0 sample and rows outside the window give exactly zero
    qo = np.array([0, 3, 5], dtype=np.int32)
    ko = np.array([0, 0, 4], dtype=np.int32)
    rng = np.random.Generator(np.random.PCG64(1))
    q = rng.standard_normal((5, 1, 4))
    k = rng.standard_normal((4, 1, 4))
    v = rng.standard_normal((4, 1, 4))
    o = ref.fwd(qo, ko, q, k, v, 1.0, "gelu_erf")
    assert np.all(o[0:3] == 0.0)
    assert np.any(o[3:5] != 0.0)
    dq, dk, dv = ref.bwd(qo, ko, q, k, v, np.ones_like(q), 1.0, "gelu_erf")
    assert np.all(dq[0:3] == 0.0)
