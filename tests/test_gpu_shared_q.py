"""GPU parity of shared-query mode (pooling attention: seed queries shared
by every sample, so Q is [n_seeds, H, d] and the backward's dQ is each
seed's gradient summed over the samples).

The oracle runs the ordinary float64 loops on the per-token Q the seeds
stand for (``ref.shared_q_tokens``) and sums the per-token dQ back onto the
seeds (``ref.shared_q_grad``, pinned by central differences on the CPU).
bf16 tolerance as everywhere: 1e-2 of max|ref| per output.
"""

import numpy as np
import pytest

from gpu_util import TOL, check, max_rel, to_dev
from oracle import ref
from workloads import offsets_from_lengths

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gd():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import recommender_model_attention_gb300 as g
    g.build()
    return g


def _case(lq, lkv, n_seeds, H, d, seed, dtype="bf16"):
    import torch
    qo, ko = offsets_from_lengths(np.asarray(lq)), offsets_from_lengths(np.asarray(lkv))
    g = torch.Generator().manual_seed(seed)
    x = {"q_off": qo, "kv_off": ko}
    for n, rows in (("q", n_seeds), ("k", ko[-1]), ("v", ko[-1]), ("do", qo[-1])):
        t = torch.randn((int(rows), H, d), generator=g) / 3
        x[n] = t.to(torch.bfloat16) if dtype == "bf16" else t
    return to_dev(x)


def _oracle(x, n_seeds, alpha, act):
    qt = ref.shared_q_tokens(ref.to_f64(x["q"]), x["q_off"])
    o = ref.fwd(x["q_off"], x["kv_off"], qt, x["k"], x["v"], alpha, act)
    dq, dk, dv = ref.bwd(x["q_off"], x["kv_off"], qt, x["k"], x["v"], x["do"], alpha, act)
    return o, ref.shared_q_grad(dq, x["q_off"], n_seeds), dk, dv


def _assert(errs, tol=TOL["bf16"]):
    check(errs, tol)


# 32 seeds; samples of 32 queries (the pooling shape), shorter ones, an
# empty one, one key-less one, keys over several blocks with ragged tails
LQ = [32, 32, 7, 0, 32, 20, 32]
LKV = [700, 129, 300, 40, 0, 1, 1000]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("act", ["gelu_erf", "gelu_taylor6", "silu"])
def test_shared_q_forward_backward(gd, d, act):
    import torch
    x = _case(LQ, LKV, 32, 2, d, 5 + d)
    alpha = d ** -0.5
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, d)
    plan.set_shared_q(32)
    o = gd.gdpa_fwd(plan, x["q"], x["k"], x["v"], alpha=alpha, act=act)
    dq, dk, dv = gd.gdpa_bwd(plan, x["q"], x["k"], x["v"], x["do"], alpha=alpha, act=act)
    plan.check()
    torch.cuda.synchronize()
    assert o.shape == (sum(LQ), 2, d) and dq.shape == (32, 2, d)
    ro, rdq, rdk, rdv = _oracle(x, 32, alpha, act)
    _assert({"o": max_rel(ref.to_f64(o), ro), "dq": max_rel(ref.to_f64(dq), rdq),
             "dk": max_rel(ref.to_f64(dk), rdk), "dv": max_rel(ref.to_f64(dv), rdv)})
    plan.destroy()


def test_shared_q_softmax_variant(gd):
    import torch
    x = _case(LQ, LKV, 48, 2, 128, 9)
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, 128)
    plan.set_shared_q(48)   # more seeds than any sample uses
    o, lse = gd.gdpa_softmax_fwd(plan, x["q"], x["k"], x["v"])
    dq, dk, dv = gd.gdpa_softmax_bwd(plan, x["q"], x["k"], x["v"], o, x["do"], lse)
    plan.check()
    torch.cuda.synchronize()
    ro, rdq, rdk, rdv = _oracle(x, 48, 128 ** -0.5, "softmax")
    _assert({"o": max_rel(ref.to_f64(o), ro), "dq": max_rel(ref.to_f64(dq), rdq),
             "dk": max_rel(ref.to_f64(dk), rdk), "dv": max_rel(ref.to_f64(dv), rdv)})
    assert not dq[32:].any()   # seeds 32..47 are used by no sample
    plan.destroy()


def test_shared_q_with_key_split_and_repeat(gd):
    # key-split forward and a second backward (dQ cleared, not added to)
    import torch
    x = _case([32] * 6, [1500, 64, 900, 2000, 128, 300], 32, 1, 128, 13)
    plan = gd.Plan(x["q_off"], x["kv_off"], 1, 128, max_kv_blocks="auto")
    plan.set_shared_q(32)
    o = gd.gdpa_fwd(plan, x["q"], x["k"], x["v"])
    dq1 = gd.gdpa_bwd(plan, x["q"], x["k"], x["v"], x["do"])[0].clone()
    dq2 = gd.gdpa_bwd(plan, x["q"], x["k"], x["v"], x["do"])[0]
    plan.check()
    torch.cuda.synchronize()
    ro, rdq, _, _ = _oracle(x, 32, 128 ** -0.5, "gelu_erf")
    _assert({"o": max_rel(ref.to_f64(o), ro), "dq": max_rel(ref.to_f64(dq1), rdq)})
    assert max_rel(ref.to_f64(dq2), ref.to_f64(dq1)) <= 1e-5
    plan.destroy()


@pytest.mark.parametrize("dtype,d", [("f32", 128), ("f32", 40), ("bf16", 32)])
@pytest.mark.parametrize("act", ["gelu_tanh", "softmax"])
def test_shared_q_on_cuda_cores(gd, dtype, d, act):
    import torch
    x = _case([4, 4, 0, 2], [30, 10, 5, 200], 6, 2, d, 3 + d, dtype=dtype)
    alpha = d ** -0.5
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, d)
    plan.set_shared_q(6)
    if act == "softmax":
        o, lse = gd.gdpa_softmax_fwd(plan, x["q"], x["k"], x["v"], alpha=alpha)
        dq, dk, dv = gd.gdpa_softmax_bwd(plan, x["q"], x["k"], x["v"], o, x["do"], lse, alpha=alpha)
    else:
        o = gd.gdpa_fwd(plan, x["q"], x["k"], x["v"], alpha=alpha, act=act)
        dq, dk, dv = gd.gdpa_bwd(plan, x["q"], x["k"], x["v"], x["do"], alpha=alpha, act=act)
    plan.check()
    torch.cuda.synchronize()
    ro, rdq, rdk, rdv = _oracle(x, 6, alpha, act)
    _assert({"o": max_rel(ref.to_f64(o), ro), "dq": max_rel(ref.to_f64(dq), rdq),
             "dk": max_rel(ref.to_f64(dk), rdk), "dv": max_rel(ref.to_f64(dv), rdv)}, TOL[dtype])
    plan.destroy()
