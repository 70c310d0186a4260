"""GPU parity of key-split forward plans (max_kv_blocks > 0).

A key-split plan cuts a query tile's key range into chunks of at most
`max_kv_blocks` 128-row key blocks, each its own forward tile, so that a
sample with a long key sequence and few query rows (the pooling-attention
shape) spreads over many SMs.  Each chunk adds its float32 partial sum of O
into a zeroed workspace and a second kernel rounds it to bf16.  Since
O = act(alpha Q K^T) V is a plain sum over keys for GDPA, the result must
match the oracle to the same bf16 tolerance as an unsplit plan; the backward
pass must be unaffected (the tensor-core backward has its own per-key-block
units; the CUDA-core dQ kernel adds each chunk's share atomically).  The
tensor-core forward splits d = 128; float32 inputs and other head dims
(bf16 d = 64 included, under the automatic kernel choice) split on the
CUDA-core kernels, checked to 1e-5 for float32; the softmax variant's
forward, whose normalisation couples the chunks, refuses split plans.
"""

import numpy as np
import pytest

from gpu_util import TOL, check, compare_full, max_rel, to_dev
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


def _case(lq, lkv, H, d, seed, dtype="bf16"):
    import torch
    qo, ko = offsets_from_lengths(np.asarray(lq)), offsets_from_lengths(np.asarray(lkv))
    g = torch.Generator().manual_seed(seed)
    x = {"q_off": qo, "kv_off": ko}
    for n, rows in (("q", qo[-1]), ("k", ko[-1]), ("v", ko[-1]), ("do", qo[-1])):
        t = torch.randn((int(rows), H, d), generator=g) / 4
        x[n] = t.to(torch.bfloat16) if dtype == "bf16" else t
    return to_dev(x)


def _assert(errs, tol=TOL["bf16"]):
    check(errs, tol)


# few query rows against long key sequences (the pooling-attention shape),
# a sample with several query tiles, ragged key tails, an empty sample
LQ = [32, 1, 300, 0, 129, 64]
LKV = [1000, 700, 900, 50, 0, 1]


@pytest.mark.parametrize("max_kvb", [1, 2, 3])
@pytest.mark.parametrize("act", ["gelu_erf", "gelu_tanh", "silu", "gelu_taylor6", "identity"])
def test_split_matches_oracle(gd, max_kvb, act):
    x = _case(LQ, LKV, 2, 128, 11 + max_kvb)
    errs = compare_full(gd, x, 2, 128, 128 ** -0.5, act, "bf16", max_kv_blocks=max_kvb)
    _assert(errs)


@pytest.mark.parametrize("window", [1, 100, 300])
def test_split_causal_window(gd, window):
    lq = [700, 260, 5]
    x = _case(lq, lq, 2, 128, 40 + window)
    errs = compare_full(gd, x, 2, 128, 128 ** -0.5, "gelu_erf", "bf16",
                        mask="causal_window", window=window, max_kv_blocks=1)
    _assert(errs)


def test_split_plan_is_split_and_counts_two_launches(gd):
    import torch
    x = _case(LQ, LKV, 2, 128, 5)
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, 128, max_kv_blocks=2)
    whole = gd.Plan(x["q_off"], x["kv_off"], 2, 128)
    assert plan.sizes()[0] > whole.sizes()[0]
    n0 = plan.launches
    gd.gdpa_fwd(plan, x["q"], x["k"], x["v"])
    plan.check()
    assert plan.launches == n0 + 2   # the tile kernel and the bf16 rounding kernel
    plan.destroy()
    whole.destroy()
    torch.cuda.synchronize()


def test_split_repeat_is_stable_and_close_to_whole(gd):
    # the workspace is cleared on every call: a second forward gives the same
    # O up to summation order, and so does the unsplit plan
    import torch
    x = _case([16, 16], [1024, 640], 1, 128, 9)
    split = gd.Plan(x["q_off"], x["kv_off"], 1, 128, max_kv_blocks=1)
    whole = gd.Plan(x["q_off"], x["kv_off"], 1, 128)
    o1 = gd.gdpa_fwd(split, x["q"], x["k"], x["v"]).clone()
    o2 = gd.gdpa_fwd(split, x["q"], x["k"], x["v"])
    ow = gd.gdpa_fwd(whole, x["q"], x["k"], x["v"])
    split.check()
    whole.check()
    torch.cuda.synchronize()
    # (the chunks' float32 adds may land in a different order on each call,
    # so the bound is one bf16 rounding step, not bit equality)
    assert max_rel(ref.to_f64(o1), ref.to_f64(o2)) <= 2 ** -8
    assert max_rel(ref.to_f64(o1), ref.to_f64(ow)) <= 2 ** -7
    split.destroy()
    whole.destroy()


@pytest.mark.parametrize("what", ["bf16_d64", "f32_d128", "f32_d40"])
@pytest.mark.parametrize("act", ["gelu_erf", "silu"])
def test_split_on_cuda_cores(gd, what, act):
    dtype, d = what.split("_d")[0], int(what.split("_d")[1])
    x = _case([8, 130, 1], [600, 300, 0], 2, d, 3 + d, dtype=dtype)
    errs = compare_full(gd, x, 2, d, d ** -0.5, act, dtype, max_kv_blocks=1)
    _assert(errs, TOL[dtype])


def test_split_softmax_forward_refused_backward_runs(gd):
    import torch
    x = _case([8, 40], [600, 300], 1, 128, 3)
    split = gd.Plan(x["q_off"], x["kv_off"], 1, 128, max_kv_blocks=1)
    whole = gd.Plan(x["q_off"], x["kv_off"], 1, 128)
    with pytest.raises(gd.GdpaError):
        gd.gdpa_softmax_fwd(split, x["q"], x["k"], x["v"])
    # the statistics of an unsplit forward feed the split plan's backward
    o, lse = gd.gdpa_softmax_fwd(whole, x["q"], x["k"], x["v"])
    got = gd.gdpa_softmax_bwd(split, x["q"], x["k"], x["v"], o, x["do"], lse)
    want = gd.gdpa_softmax_bwd(whole, x["q"], x["k"], x["v"], o, x["do"], lse)
    split.check()
    whole.check()
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        assert max_rel(ref.to_f64(g), ref.to_f64(w)) <= 1e-5
    split.destroy()
    whole.destroy()


def test_automatic_split_matches_oracle(gd):
    # keys up to 1500 rows (12 blocks): the planner picks 2-block chunks
    x = _case([32, 32, 5, 200], [1500, 900, 1200, 30], 2, 128, 21)
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, 128, max_kv_blocks="auto")
    whole = gd.Plan(x["q_off"], x["kv_off"], 2, 128)
    assert plan.sizes()[0] > whole.sizes()[0]
    plan.destroy()
    whole.destroy()
    errs = compare_full(gd, x, 2, 128, 128 ** -0.5, "gelu_erf", "bf16", max_kv_blocks="auto")
    _assert(errs)
