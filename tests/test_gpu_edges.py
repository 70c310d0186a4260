"""GPU parity on edge cases of the jagged layout and of the launch.

Same tolerances as the main parity file (bf16 inputs: 1e-2 of max|ref| for
O, dQ, dK, dV separately).  Cases: a batch of zero samples, a batch whose
lengths are all zero, lengths on and next to the 128-row tile boundaries,
many heads, d = 64 with the causal window in the backward pass, key blocks
on and next to 64 keys (the forward's score product and P V run in halves
of 64 keys, the second skipped for a block of at most 64), the round-robin
dealing policy, fewer persistent CTAs than SMs, and a launch on a side
stream.
"""

import numpy as np
import pytest

from gpu_util import TOL, check, compare_full, to_dev
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


def _case(lq, lkv, H, d, seed):
    import torch
    qo, ko = offsets_from_lengths(np.asarray(lq)), offsets_from_lengths(np.asarray(lkv))
    g = torch.Generator().manual_seed(seed)
    x = {"q_off": qo, "kv_off": ko}
    for n, rows in (("q", qo[-1]), ("k", ko[-1]), ("v", ko[-1]), ("do", qo[-1])):
        x[n] = (torch.randn((int(rows), H, d), generator=g) / 4).to(torch.bfloat16)
    return to_dev(x)


def _assert(errs, tol=TOL["bf16"]):
    check(errs, tol)


def test_zero_samples(gd):
    import torch
    x = _case([], [], 2, 128, 0)
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, 128)
    assert plan.sizes()[:2] == (0, 0)
    o = gd.gdpa_fwd(plan, x["q"], x["k"], x["v"])
    dq, dk, dv = gd.gdpa_bwd(plan, x["q"], x["k"], x["v"], x["do"])
    plan.check()
    assert o.shape == (0, 2, 128) and dq.numel() == dk.numel() == dv.numel() == 0
    assert plan.launches == 0
    plan.destroy()
    torch.cuda.synchronize()


def test_all_lengths_zero_keys(gd):
    # queries but no keys anywhere: O = 0 and dQ = 0 (zero tiles, cleared dQ)
    import torch
    x = _case([5, 130, 0, 256], [0, 0, 0, 0], 2, 128, 1)
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, 128)
    o = torch.full_like(x["q"], 3.0)
    gd.gdpa_fwd(plan, x["q"], x["k"], x["v"], o=o)
    dq = torch.full(x["q"].shape, 3.0, device="cuda")
    dk = torch.empty((0, 2, 128), device="cuda")
    gd.gdpa_bwd(plan, x["q"], x["k"], x["v"], x["do"], dq, dk, dk.clone())
    plan.check()
    assert torch.all(o == 0) and torch.all(dq == 0)
    plan.destroy()


@pytest.mark.parametrize("act", ["gelu_erf", "silu"])
def test_tile_boundary_lengths(gd, act):
    lens = [127, 128, 129, 255, 256, 257, 383, 384, 385, 1]
    x = _case(lens, lens[::-1], 2, 128, 2)
    _assert(compare_full(gd, x, 2, 128, 128 ** -0.5, act, "bf16"))


def test_tile_boundary_lengths_window(gd):
    lens = [127, 128, 129, 255, 256, 257, 511, 512, 513]
    x = _case(lens, lens, 2, 128, 3)
    _assert(compare_full(gd, x, 2, 128, 128 ** -0.5, "gelu_tanh", "bf16", "causal_window", 128))


@pytest.mark.parametrize("act,mask,window", [("gelu_erf", "none", 0), ("silu", "causal_window", 100)])
def test_key_half_boundary_lengths(gd, act, mask, window):
    lkv = [63, 64, 65, 66, 79, 80, 191, 192, 193, 200]
    lq = lkv if mask == "causal_window" else [70, 130, 64, 65, 200, 1, 129, 300, 64, 190]
    x = _case(lq, lkv, 2, 128, 11)
    _assert(compare_full(gd, x, 2, 128, 128 ** -0.5, act, "bf16", mask, window))


def test_many_heads(gd):
    x = _case([200, 37, 300], [150, 260, 9], 16, 64, 4)
    _assert(compare_full(gd, x, 16, 64, 0.125, "gelu_erf", "bf16"))


@pytest.mark.parametrize("window", [1, 64, 129])
def test_d64_window_backward(gd, window):
    lens = [300, 129, 64, 500]
    x = _case(lens, lens, 2, 64, 5 + window)
    _assert(compare_full(gd, x, 2, 64, 0.125, "gelu_taylor6", "bf16", "causal_window", window))


@pytest.mark.parametrize("sched", ["round_robin", "zigzag"])
@pytest.mark.parametrize("num_sms", [1, 7])
def test_dealing_and_cta_count(gd, sched, num_sms):
    x = _case([400, 3, 129, 0, 260, 77], [90, 300, 128, 5, 0, 200], 2, 128, 6)
    _assert(compare_full(gd, x, 2, 128, 128 ** -0.5, "gelu_erf", "bf16", sched=sched,
                         num_sms=num_sms))


def test_side_stream(gd):
    import torch
    x = _case([300, 64, 129], [200, 128, 1], 2, 128, 7)
    s = torch.cuda.Stream()
    _assert(compare_full(gd, x, 2, 128, 128 ** -0.5, "silu", "bf16", stream=s))


def test_repeat_calls_identical_forward(gd):
    # the forward has no atomics: repeated launches give identical bytes
    import torch
    x = _case([300, 64, 129, 700], [200, 128, 1, 90], 2, 128, 8)
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, 128)
    o1 = gd.gdpa_fwd(plan, x["q"], x["k"], x["v"])
    o2 = gd.gdpa_fwd(plan, x["q"], x["k"], x["v"])
    plan.check()
    assert torch.equal(o1, o2)
    plan.destroy()


@pytest.mark.parametrize("num_sms", [1, 2, 3, 7])
@pytest.mark.parametrize("sched", ["round_robin", "zigzag"])
def test_multi_block_tiles_on_few_ctas(gd, sched, num_sms):
    """Long queues of forward tiles with 1 to 4 key blocks each (keys up to
    500), in both dealing orders, on a handful of CTAs: every CTA's two tile
    slots take turns on the K and V rings with tiles of different lengths,
    the case where a stage released too early or a barrier phase skipped
    shows up as a wrong output or an abandoned wait."""
    rng = np.random.default_rng(900 + num_sms)
    lq = rng.integers(1, 300, 24).tolist()
    lkv = rng.integers(1, 500, 24).tolist()
    x = _case(lq, lkv, 2, 128, 900 + num_sms)
    _assert(compare_full(gd, x, 2, 128, 128 ** -0.5, "gelu_erf", "bf16", sched=sched,
                         num_sms=num_sms))


@pytest.mark.parametrize("num_sms", [2, 5])
@pytest.mark.parametrize("act,mask,window,split", [
    ("softmax", "none", 0, 0),            # two passes over tiles of several key blocks
    ("silu", "causal_window", 200, 0),    # windowed tiles of 1-3 blocks
    ("gelu_erf", "none", 0, 1),           # key-split tiles of one block, fp32 reduce
])
def test_forward_queues_on_few_ctas(gd, act, mask, window, split, num_sms):
    """The forward's item queue (K, V rings and the S issuer's guards) on long
    per-CTA queues for the softmax variant's two passes, the causal window
    and a key-split plan."""
    rng = np.random.default_rng(950 + num_sms)
    lq = rng.integers(1, 400, 16).tolist()
    lkv = lq if mask != "none" else rng.integers(1, 600, 16).tolist()
    x = _case(lq, lkv, 2, 128, 950 + num_sms)
    _assert(compare_full(gd, x, 2, 128, 128 ** -0.5, act, "bf16", mask, window,
                         backward=act != "softmax", num_sms=num_sms, max_kv_blocks=split))
