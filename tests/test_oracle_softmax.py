"""Pins of the oracle's softmax variant (Jagged Flash Attention) to facts
outside its loops (CPU only):

* the dense padded formulation through SciPy's softmax (brute force);
* partition of unity: with V = 1 every row with a valid key gives exactly 1;
* equal scores (Q = 0) average the valid V rows;
* a row-wise constant added to every score of a row (an extra feature
  dimension) changes nothing (shift invariance);
* a single valid key returns its V row; a huge scale selects the argmax key;
* rows without a valid key are zero;
* the gradients against central differences of the forward, the row
  log-sum-exp against SciPy's logsumexp, and dV's column sums (each query
  row's weights sum to one).
"""

import numpy as np
import pytest

from oracle import brute, ref
from workloads import offsets_from_lengths, small_case


def _case(seed, lq, lkv, H=2, d=8):
    g = np.random.default_rng(seed)
    qo, ko = offsets_from_lengths(np.asarray(lq)), offsets_from_lengths(np.asarray(lkv))
    q = g.standard_normal((qo[-1], H, d))
    k = g.standard_normal((ko[-1], H, d))
    v = g.standard_normal((ko[-1], H, d))
    return qo, ko, q, k, v


@pytest.mark.parametrize("mask,window", [("none", 0), ("causal_window", 3), ("causal_window", 1)])
def test_softmax_loops_match_dense_brute_force(mask, window):
    lq = [5, 1, 9, 0, 7]
    lkv = lq if mask != "none" else [3, 6, 1, 4, 0]
    qo, ko, q, k, v = _case(1, lq, lkv)
    got = ref.fwd(qo, ko, q, k, v, 0.7, "softmax", mask, window)
    want = brute.fwd(qo, ko, q, k, v, 0.7, "softmax", mask, window)
    assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))


def test_softmax_partition_of_unity():
    qo, ko, q, k, v = _case(2, [4, 6, 3], [5, 2, 0])
    o = ref.fwd(qo, ko, q, k, np.ones_like(v), 1.3, "softmax")
    lkv = np.diff(ko)
    for b in range(3):
        rows = o[qo[b]:qo[b + 1]]
        assert np.allclose(rows, 1.0 if lkv[b] > 0 else 0.0, atol=1e-14, rtol=0)


def test_softmax_equal_scores_average_values():
    qo, ko, q, k, v = _case(3, [6, 4], [6, 4])
    o = ref.fwd(qo, ko, np.zeros_like(q), k, v, 1.0, "softmax", "causal_window", 3)
    for b in range(2):
        for i in range(qo[b + 1] - qo[b]):
            js = [j for j in range(ko[b + 1] - ko[b]) if i - 3 < j <= i]
            want = v[ko[b] + np.array(js)].mean(axis=0)
            assert np.allclose(o[qo[b] + i], want, atol=1e-14, rtol=0)


def test_softmax_row_shift_invariance():
    qo, ko, q, k, v = _case(4, [5, 8], [7, 3], H=1, d=6)
    shift = np.random.default_rng(5).standard_normal(q.shape[0]) * 20.0
    q2 = np.concatenate([q, shift[:, None, None]], axis=2)
    k2 = np.concatenate([k, np.ones(k.shape[:2] + (1,))], axis=2)
    v2 = np.concatenate([v, np.zeros(v.shape[:2] + (1,))], axis=2)
    a = ref.fwd(qo, ko, q, k, v, 0.9, "softmax")
    b = ref.fwd(qo, ko, q2, k2, v2, 0.9, "softmax")[..., :6]
    assert np.max(np.abs(a - b)) <= 1e-12


def test_softmax_single_key_and_argmax_limit():
    qo, ko, q, k, v = _case(6, [3, 4], [1, 5])
    o = ref.fwd(qo, ko, q, k, v, 1.0, "softmax")
    assert np.allclose(o[0:3], v[0], atol=1e-14, rtol=0)
    big = ref.fwd(qo, ko, q, k, v, 1e5, "softmax")
    for i in range(4):
        for h in range(q.shape[1]):
            s = k[1:6, h] @ q[3 + i, h]
            assert np.allclose(big[3 + i, h], v[1 + int(np.argmax(s)), h], atol=1e-12, rtol=0)


def test_softmax_empty_rows_are_zero():
    qo, ko, q, k, v = _case(7, [4, 3], [0, 2])
    o = ref.fwd(qo, ko, q, k, v, 1.0, "softmax", "causal_window", 1)
    assert np.all(o[0:4] == 0.0)
    # window 1 on sample 1: row i sees key i only (rows 0, 1), row 2 none
    assert np.allclose(o[4], v[0], atol=1e-14) and np.allclose(o[5], v[1], atol=1e-14)
    assert np.all(o[6] == 0.0)


def test_softmax_bf16_like_case_against_brute():
    c = small_case(8, B=4, H=2, d=16, q_range=(1, 40), kv_range=(1, 30), dtype="bf16")
    got = ref.fwd(c["q_off"], c["kv_off"], c["q"], c["k"], c["v"], 0.25, "softmax")
    want = brute.fwd(c["q_off"], c["kv_off"], ref.to_f64(c["q"]), ref.to_f64(c["k"]),
                     ref.to_f64(c["v"]), 0.25, "softmax")
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))


@pytest.mark.parametrize("mask,window", [("none", 0), ("causal_window", 2)])
def test_softmax_gradients_by_finite_differences(mask, window):
    rng = np.random.Generator(np.random.PCG64(9))
    lq = np.array([3, 5]) if mask == "causal_window" else np.array([3, 4])
    lkv = lq.copy() if mask == "causal_window" else np.array([5, 2])
    qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
    H, d, alpha = 1, 4, 0.8
    q = rng.standard_normal((qo[-1], H, d))
    k = rng.standard_normal((ko[-1], H, d))
    v = rng.standard_normal((ko[-1], H, d))
    do = rng.standard_normal((qo[-1], H, d))
    dq, dk, dv = ref.bwd(qo, ko, q, k, v, do, alpha, "softmax", mask, window)

    def loss(qq, kk, vv):
        return float(np.sum(ref.fwd(qo, ko, qq, kk, vv, alpha, "softmax", mask, window) * do))

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


def test_softmax_lse_against_scipy_logsumexp():
    from scipy import special
    qo, ko, q, k, v = _case(10, [6, 3, 0, 5], [4, 0, 3, 5])
    got = ref.lse(qo, ko, q, k, 0.6, "causal_window", 3)
    for b in range(4):
        for i in range(qo[b + 1] - qo[b]):
            js = [j for j in range(ko[b + 1] - ko[b]) if i - 3 < j <= i]
            for h in range(q.shape[1]):
                if not js:
                    assert got[qo[b] + i, h] == -np.inf
                    continue
                s = 0.6 * (k[ko[b] + np.array(js), h] @ q[qo[b] + i, h])
                assert abs(got[qo[b] + i, h] - special.logsumexp(s)) <= 1e-12


def test_softmax_gradient_of_values_is_weighted_do():
    # dV_j = sum_i P_ij dO_i: with dO = 1 per row, each column of dV is the
    # total softmax weight key j receives
    qo, ko, q, k, v = _case(11, [4, 2], [3, 3])
    do = np.ones_like(q)
    _, _, dv = ref.bwd(qo, ko, q, k, v, do, 1.0, "softmax")
    # every query row's weights sum to 1, so a sample's dV rows sum to its Lq
    for b in range(2):
        tot = dv[ko[b]:ko[b + 1]].sum(axis=0)
        assert np.allclose(tot, qo[b + 1] - qo[b], atol=1e-12)
