"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle
on identical seeded inputs.

Tolerances: float32 inputs max|x - ref| <= 1e-5 max|ref|; bf16 inputs with
float32 accumulation max|x - ref| <= 1e-2 max|ref|; the same bound for O, dQ,
dK and dV separately.  Plans must match the oracle's planner bit for bit.
"""

import numpy as np
import pytest

from gpu_util import TOL, check, compare_full, compare_sampled, max_rel, pick_samples, small_case, to_dev
from oracle import planner as ref_planner
from oracle import ref
from workloads import CONFIGS, get_config, make_inputs

pytestmark = pytest.mark.gpu

ACTS = ["gelu_erf", "gelu_tanh", "silu", "gelu_taylor6", "identity"]
BF16_KERNELS = ["simt", "auto"]


@pytest.fixture(scope="module")
def gd():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import recommender_model_attention_gb300 as g
    g.build()
    return g


def _assert(errs, tol):
    check(errs, tol)


def test_device_plan_matches_oracle(gd):
    w = get_config(1)
    x = make_inputs(w, device="cpu")
    p = gd.Plan(x["q_off"], x["kv_off"], w.H, w.d, mask=w.mask, window=w.window)
    ref = ref_planner.plan(x["q_off"], x["kv_off"], w.H, p.num_sms, mask=w.mask, window=w.window)
    tiles, seg = p.export()
    assert np.array_equal(tiles, ref["fwd"]) and np.array_equal(seg, ref["fwd_seg"])
    p.destroy()


def test_tiny_workload_f32(gd):
    w = get_config(0)
    x = to_dev(make_inputs(w, device="cpu"))
    _assert(compare_full(gd, x, w.H, w.d, w.alpha, w.act, "f32"), TOL["f32"])


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("mask,window", [("none", 0), ("causal_window", 40)])
def test_small_f32_all_activations(gd, act, mask, window):
    c = small_case(21, B=6, H=2, d=64, q_range=(0, 300),
                   kv_range=None if mask != "none" else (0, 200), zero_lengths=True)
    _assert(compare_full(gd, to_dev(c), 2, 64, 0.125, act, "f32", mask, window), TOL["f32"])


@pytest.mark.parametrize("kernel", BF16_KERNELS)
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("d", [64, 128])
def test_small_bf16_no_mask(gd, kernel, act, d):
    c = small_case(7 + d, B=7, H=3, d=d, q_range=(1, 400), kv_range=(1, 300), dtype="bf16",
                   rmsnorm=True)
    _assert(compare_full(gd, to_dev(c), 3, d, d ** -0.5, act, "bf16", kernel=kernel), TOL["bf16"])


@pytest.mark.parametrize("kernel", BF16_KERNELS)
@pytest.mark.parametrize("window", [1, 77, 256])
def test_small_bf16_causal_window(gd, kernel, window):
    c = small_case(30 + window, B=5, H=2, d=128, q_range=(1, 700), dtype="bf16", rmsnorm=True)
    _assert(compare_full(gd, to_dev(c), 2, 128, 128 ** -0.5, "silu", "bf16", "causal_window",
                         window, kernel=kernel), TOL["bf16"])


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_bf16_empty_and_degenerate_samples(gd, kernel):
    # zero-length queries or keys, single keys, a sample of exactly one tile
    from workloads import offsets_from_lengths
    import torch
    lq = np.array([0, 5, 128, 1, 0, 129, 3, 300])
    lkv = np.array([4, 0, 128, 1, 0, 1, 200, 17])
    qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
    g = torch.Generator().manual_seed(3)
    H, d = 2, 128
    x = {"q_off": qo, "kv_off": ko}
    for n, rows in (("q", qo[-1]), ("k", ko[-1]), ("v", ko[-1]), ("do", qo[-1])):
        x[n] = (torch.randn((int(rows), H, d), generator=g) / 4).to(torch.bfloat16)
    _assert(compare_full(gd, to_dev(x), H, d, d ** -0.5, "gelu_erf", "bf16", kernel=kernel),
            TOL["bf16"])


@pytest.mark.parametrize("kernel", BF16_KERNELS)
@pytest.mark.parametrize("idx", [1, 2, 3])
def test_workload_forward_sampled(gd, kernel, idx):
    w = get_config(idx)
    x = make_inputs(w, device="cuda")
    samples = pick_samples(x["q_off"], x["kv_off"], seed=idx)
    _assert(compare_sampled(gd, x, samples, w.H, w.d, w.alpha, w.act, w.mask, w.window,
                            kernel=kernel), TOL["bf16"])


@pytest.mark.parametrize("kernel", BF16_KERNELS)
def test_training_workload_fwd_bwd_sampled(gd, kernel):
    w = get_config(4)
    x = make_inputs(w, device="cuda")
    samples = pick_samples(x["q_off"], x["kv_off"], n_random=3, seed=4)
    _assert(compare_sampled(gd, x, samples, w.H, w.d, w.alpha, w.act, w.mask, w.window,
                            kernel=kernel, backward=True), TOL["bf16"])


def test_pma_activation_inputs_bounded(gd):
    # the PMA workload's RMSNorm gain keeps |alpha q.k| <= 2 (up to bf16 rounding)
    import torch
    w = get_config(3)
    x = make_inputs(w, device="cuda")
    kv_off = torch.from_numpy(x["kv_off"].astype(np.int64))
    b = int(np.argmax(np.diff(x["kv_off"])))
    q = x["q"][32 * b:32 * (b + 1)].float()
    k = x["k"][int(kv_off[b]):int(kv_off[b + 1])].float()
    s = torch.einsum("ihc,jhc->hij", q, k) * w.alpha
    assert float(s.abs().max()) <= 2.0 * (1 + 2 ** -7)


def test_output_guard_regions_untouched(gd):
    # canaries before and after O, dQ, dK, dV catch writes past jagged ends
    import torch
    c = to_dev(small_case(99, B=5, H=2, d=128, q_range=(1, 260), kv_range=(1, 140),
                          dtype="bf16", rmsnorm=True))
    plan = gd.Plan(c["q_off"], c["kv_off"], 2, 128)
    Tq, Tkv, pad = int(c["q_off"][-1]), int(c["kv_off"][-1]), 300
    for kernel in ("simt", "auto"):
        plan.set_kernel(kernel)
        ob = torch.full((Tq + 2 * pad, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        gb = [torch.full((n + 2 * pad, 2, 128), 7.0, device="cuda") for n in (Tq, Tkv, Tkv)]
        o = ob[pad:pad + Tq]
        gd.gdpa_fwd(plan, c["q"], c["k"], c["v"], o=o, act="gelu_tanh")
        gd.gdpa_bwd(plan, c["q"], c["k"], c["v"], c["do"], *[g[pad:pad + n] for g, n in
                                                            zip(gb, (Tq, Tkv, Tkv))], act="gelu_tanh")
        plan.check()
        for buf, n in [(ob, Tq)] + list(zip(gb, (Tq, Tkv, Tkv))):
            assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + n:] == 7.0)
    plan.destroy()


def test_launch_counter_and_timing(gd):
    import torch
    w = get_config(2)
    x = make_inputs(w, device="cuda")
    plan = gd.Plan(x["q_off"], x["kv_off"], w.H, w.d)
    plan.set_timing(True)
    n0 = plan.launches
    gd.gdpa_fwd(plan, x["q"], x["k"], x["v"], act=w.act)
    plan.check()
    assert plan.launches == n0 + 1
    torch.cuda.synchronize()
    se, sm = plan.sm_times("fwd")
    assert np.all(se[:, 1] >= se[:, 0])
    plan.destroy()


def test_pma_workload_as_benchmarked_sampled(gd):
    # the pooling workload in the launch configuration the benchmark times:
    # the seed rows passed once (shared-query mode) and the planner's key
    # split; sampled outputs against the oracle on the materialised queries
    import torch
    w = get_config("pma_pooling")
    x = make_inputs(w, device="cuda")
    plan = gd.Plan(x["q_off"], x["kv_off"], w.H, w.d, mask=w.mask, window=w.window,
                   max_kv_blocks="auto")
    plan.set_shared_q(w.shared_q)
    o = gd.gdpa_fwd(plan, x["q_seeds"], x["k"], x["v"], alpha=w.alpha, act=w.act)
    plan.check()
    torch.cuda.synchronize()
    samples = pick_samples(x["q_off"], x["kv_off"], seed=3)
    sq, skv, qi, kvi = ref.sub_batch(x["q_off"], x["kv_off"], samples)
    qi_t = torch.from_numpy(qi).to(o.device)
    kvi_t = torch.from_numpy(kvi).to(o.device)
    want = ref.fwd(sq, skv, x["q"].index_select(0, qi_t), x["k"].index_select(0, kvi_t),
                   x["v"].index_select(0, kvi_t), w.alpha, w.act, w.mask, w.window)
    _assert({"o": max_rel(ref.to_f64(o.index_select(0, qi_t)), want)}, TOL["bf16"])
    plan.destroy()
