"""The fused RMSNorm prologue on the tensor-core kernels against the oracle's
RMSNorm composed with GDPA (``oracle/rmsnorm.py``), through the C ABI.

The kernels take the raw Q and K rows, normalise every (token, head) row of
both (the keys in a pass of their own, rounded to bf16; each query row's
scale folded into alpha), and return the gradients with respect to the raw
rows.  Raw rows here carry random per-row scales so that the norm matters.
The bf16 rounding of the normalised keys is the largest error term beside
P's: with the Taylor GELU at |x| up to 3.2 (first case) it alone moves O by
about 5e-3 of max|O| (float64 emulation), within the bf16 tolerance.
"""

import numpy as np
import pytest
import torch

from gpu_util import TOL, check, max_rel, to_dev
from oracle import ref
from oracle import rmsnorm as rn
from workloads import get_config, make_inputs, offsets_from_lengths

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import recommender_model_attention_gb300 as g
    g.build()
    return g


def _raw_case(seed, lq, lkv, H, d):
    """bf16 raw rows N(0, 1) times a per-row scale in [0.2, 5]."""
    g = np.random.default_rng(seed)
    qo, ko = offsets_from_lengths(np.asarray(lq)), offsets_from_lengths(np.asarray(lkv))

    def rows(n, scaled):
        x = g.standard_normal((int(n), H, d)).astype(np.float32)
        if scaled:
            x *= np.exp(g.uniform(np.log(0.2), np.log(5.0), size=(int(n), H, 1))).astype(np.float32)
        return torch.from_numpy(x).to(torch.bfloat16)

    x = {"q_off": qo, "kv_off": ko, "q": rows(qo[-1], True), "k": rows(ko[-1], True),
         "v": rows(ko[-1], False), "do": rows(qo[-1], False)}
    return to_dev(x)


def _run(gd, x, H, d, act, gain, eps, mask="none", window=0, alpha=None, backward=True,
         max_kv_blocks=0):
    alpha = d ** -0.5 if alpha is None else alpha
    plan = gd.Plan(x["q_off"], x["kv_off"], H, d, mask=mask, window=window,
                   max_kv_blocks=max_kv_blocks)
    plan.set_kernel("tcgen05")
    plan.set_qk_norm(gain, eps)
    args = (x["q_off"], x["kv_off"], x["q"], x["k"], x["v"])
    errs = {}
    if act == "softmax":
        o, lse = gd.gdpa_softmax_fwd(plan, x["q"], x["k"], x["v"], alpha=alpha)
    else:
        o = gd.gdpa_fwd(plan, x["q"], x["k"], x["v"], alpha=alpha, act=act)
    plan.check()
    errs["o"] = max_rel(ref.to_f64(o), rn.fwd(*args, alpha, act, gain, eps, mask, window))
    if backward:
        if act == "softmax":
            grads = gd.gdpa_softmax_bwd(plan, x["q"], x["k"], x["v"], o, x["do"], lse, alpha=alpha)
        else:
            grads = gd.gdpa_bwd(plan, x["q"], x["k"], x["v"], x["do"], alpha=alpha, act=act)
        plan.check()
        want = rn.bwd(*args, x["do"], alpha, act, gain, eps, mask, window)
        for name, g, w in zip(("dq", "dk", "dv"), grads, want):
            errs[name] = max_rel(ref.to_f64(g), w)
    plan.destroy()
    return errs


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("act", ["gelu_erf", "silu", "gelu_taylor6", "softmax"])
def test_fused_rmsnorm_fwd_bwd(gd, d, act):
    # one and several key blocks, a sample shorter than a tile, ragged tails
    x = _raw_case(11, [300, 5, 129, 64, 1], [70, 300, 1, 257, 40], 2, d)
    check(_run(gd, x, 2, d, act, gain=0.9, eps=1e-6), TOL["bf16"])


@pytest.mark.parametrize("window", [1, 77])
def test_fused_rmsnorm_causal_window(gd, window):
    lens = [300, 129, 7]
    x = _raw_case(12, lens, lens, 2, 128)
    check(_run(gd, x, 2, 128, "silu", gain=1.0, eps=1e-6, mask="causal_window", window=window),
          TOL["bf16"])


def test_fused_rmsnorm_gain_and_eps(gd):
    # the Taylor GELU with the PMA workload's gain (|alpha q.k| <= 2) and a
    # large eps, which changes every row's scale
    x = _raw_case(13, [32, 32, 32], [500, 9, 130], 4, 128)
    g = float(np.sqrt(2.0) * 128 ** -0.25)
    check(_run(gd, x, 4, 128, "gelu_taylor6", gain=g, eps=0.05), TOL["bf16"])


def test_fused_rmsnorm_key_split(gd):
    x = _raw_case(14, [32, 40], [1100, 300], 2, 128)
    check(_run(gd, x, 2, 128, "gelu_tanh", gain=1.0, eps=1e-6, backward=True, max_kv_blocks=2),
          TOL["bf16"])


def test_fused_rmsnorm_shared_seeds(gd):
    # pooling attention: the seeds are the raw Q rows, normalised like tokens
    g = np.random.default_rng(15)
    H, d, n = 2, 128, 32
    lkv = [300, 17, 140]
    qo, ko = offsets_from_lengths(np.full(3, n)), offsets_from_lengths(np.asarray(lkv))
    seeds = torch.from_numpy((g.standard_normal((n, H, d)) * 3).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy((g.standard_normal((ko[-1], H, d)) * 0.5).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(g.standard_normal((ko[-1], H, d)).astype(np.float32)).to(torch.bfloat16)
    do = torch.from_numpy(g.standard_normal((qo[-1], H, d)).astype(np.float32)).to(torch.bfloat16)
    plan = gd.Plan(qo, ko, H, d)
    plan.set_shared_q(n)
    plan.set_qk_norm(1.0, 1e-6)
    dev = [t.cuda() for t in (seeds, k, v, do)]
    o = gd.gdpa_fwd(plan, dev[0], dev[1], dev[2], act="gelu_erf")
    dq, dk, dv = gd.gdpa_bwd(plan, dev[0], dev[1], dev[2], dev[3], act="gelu_erf")
    plan.check()
    qt = ref.shared_q_tokens(ref.to_f64(seeds), qo)
    a = d ** -0.5
    want_o = rn.fwd(qo, ko, qt, k, v, a, "gelu_erf")
    wdq, wdk, wdv = rn.bwd(qo, ko, qt, k, v, do, a, "gelu_erf")
    check({"o": max_rel(ref.to_f64(o), want_o),
           "dq": max_rel(ref.to_f64(dq), ref.shared_q_grad(wdq, qo, n)),
           "dk": max_rel(ref.to_f64(dk), wdk), "dv": max_rel(ref.to_f64(dv), wdv)}, TOL["bf16"])
    plan.destroy()


def test_fused_rmsnorm_training_workload_sampled(gd):
    # a prefix of the training workload with raw (unnormalised) Q and K
    w = get_config("training_cross_fwd_bwd")
    from workloads import draw_lengths
    lq, lkv = draw_lengths(w)
    x = make_inputs(w, device="cpu", seed=21, lengths=(lq[:24], lkv[:24]))
    g = np.random.default_rng(16)
    for n in ("q", "k"):
        s = np.exp(g.uniform(-1.5, 1.5, size=(x[n].shape[0], w.H, 1))).astype(np.float32)
        x[n] = (x[n].float() * torch.from_numpy(s)).to(torch.bfloat16)
    x = to_dev(x)
    check(_run(gd, x, w.H, w.d, w.act, gain=1.0, eps=1e-6), TOL["bf16"])


def test_fused_rmsnorm_refused_on_cuda_cores(gd):
    x = _raw_case(17, [10], [10], 1, 64)
    plan = gd.Plan(x["q_off"], x["kv_off"], 1, 64)
    plan.set_kernel("simt")
    plan.set_qk_norm(1.0, 1e-6)
    with pytest.raises(gd.GdpaError) as e:
        gd.gdpa_fwd(plan, x["q"], x["k"], x["v"], act="silu")
    assert e.value.status == 2   # GDPA_ERR_UNSUPPORTED
    plan.set_qk_norm(0.0, 0.0)   # off again: the CUDA-core kernels run
    gd.gdpa_fwd(plan, x["q"], x["k"], x["v"], act="silu")
    plan.check()
    plan.destroy()
