"""Pins of the oracle's shared-query mode (pooling attention with seed
queries shared by every sample), CPU only:

* the per-token Q it builds against an explicit per-sample loop over the
  seeds, and the forward on it against the dense padded brute force with
  each sample given the seeds as its own queries;
* the seeds' gradient against central differences of the scalar loss
  sum(O * dO) with respect to each seed entry (a shared parameter's
  gradient is the sum over its uses; the differences know nothing of that);
* samples shorter than the seed set use a prefix of it, an empty sample
  contributes nothing.
"""

import numpy as np
import pytest

from oracle import brute, ref
from workloads import offsets_from_lengths


def _case(seed, lq, lkv, n_seeds, H=2, d=8):
    g = np.random.default_rng(seed)
    qo, ko = offsets_from_lengths(np.asarray(lq)), offsets_from_lengths(np.asarray(lkv))
    seeds = g.standard_normal((n_seeds, H, d))
    k = g.standard_normal((ko[-1], H, d))
    v = g.standard_normal((ko[-1], H, d))
    return qo, ko, seeds, k, v


def test_tokens_are_the_seeds_per_sample():
    qo, ko, seeds, k, v = _case(0, [4, 2, 0, 4], [3, 5, 1, 2], 4)
    q = ref.shared_q_tokens(seeds, qo)
    assert q.shape == (10, 2, 8)
    for b, n in enumerate([4, 2, 0, 4]):
        for i in range(n):
            assert np.array_equal(q[qo[b] + i], seeds[i])


@pytest.mark.parametrize("act", ["gelu_erf", "silu", "softmax"])
def test_forward_matches_brute_force_per_sample(act):
    qo, ko, seeds, k, v = _case(1, [3, 3, 1], [5, 2, 7], 3)
    o = ref.fwd(qo, ko, ref.shared_q_tokens(seeds, qo), k, v, 0.4, act)
    for b, n in enumerate([3, 3, 1]):
        kb = k[ko[b]:ko[b + 1]]
        vb = v[ko[b]:ko[b + 1]]
        want = brute.fwd(np.array([0, n]), np.array([0, len(kb)]), seeds[:n], kb, vb, 0.4, act)
        assert np.allclose(o[qo[b]:qo[b + 1]], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["gelu_erf", "gelu_taylor6", "softmax"])
def test_seed_gradient_matches_central_differences(act):
    lq, lkv, n = [3, 2, 3, 0], [4, 6, 2, 3], 3
    qo, ko, seeds, k, v = _case(2, lq, lkv, n, H=1, d=4)
    g = np.random.default_rng(7)
    do = g.standard_normal((qo[-1], 1, 4))
    dq, _, _ = ref.bwd(qo, ko, ref.shared_q_tokens(seeds, qo), k, v, do, 0.6, act)
    got = ref.shared_q_grad(dq, qo, n)

    def loss(s):
        return float(np.sum(ref.fwd(qo, ko, ref.shared_q_tokens(s, qo), k, v, 0.6, act) * do))

    h = 1e-6
    fd = np.zeros_like(seeds)
    for idx in np.ndindex(*seeds.shape):
        sp, sm = seeds.copy(), seeds.copy()
        sp[idx] += h
        sm[idx] -= h
        fd[idx] = (loss(sp) - loss(sm)) / (2 * h)
    assert np.allclose(got, fd, rtol=1e-6, atol=1e-7)


def test_short_and_empty_samples_use_a_prefix():
    qo, ko, seeds, k, v = _case(3, [1, 0, 2], [2, 2, 2], 4)
    dq_tok = np.arange(qo[-1] * 2 * 8, dtype=np.float64).reshape(qo[-1], 2, 8)
    got = ref.shared_q_grad(dq_tok, qo, 4)
    assert np.array_equal(got[0], dq_tok[0] + dq_tok[1])
    assert np.array_equal(got[1], dq_tok[2])
    assert not got[2:].any()
