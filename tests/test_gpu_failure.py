"""Failure path of the tensor-core kernels, without a GPU fault.

Every barrier wait in the kernels is bounded.  The plan's test hook shortens
the limit to 20 ms and makes CTA 0's loader skip its first query-tile load,
so one wait is never satisfied: the kernel must record a timeout, unwind
(its copies and MMAs in flight finish, TMEM is freed) and return, gdpa_check
must report GDPA_ERR_TIMEOUT, and the next normal launch on the same plan
must match the oracle.  Host-side refusals (a plan used with another device
current) are checked where the box has a second device.
"""

import time

import numpy as np
import pytest

from gpu_util import TOL, check, max_rel, small_case, to_dev
from oracle import ref

pytestmark = pytest.mark.gpu

TIMEOUT = 5   # GDPA_ERR_TIMEOUT


@pytest.fixture(scope="module")
def gd():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import recommender_model_attention_gb300 as g
    g.build()
    return g


def _case(d):
    # enough tiles and units that every CTA (CTA 0 included) has work
    return to_dev(small_case(71, B=64, H=4, d=d, q_range=(100, 300), kv_range=(50, 200),
                             dtype="bf16", rmsnorm=True))


@pytest.mark.parametrize("which", ["fwd", "bwd"])
@pytest.mark.parametrize("d", [128, 64])
def test_expired_wait_reports_timeout_and_plan_recovers(gd, which, d):
    import torch
    c = _case(d)
    alpha = d ** -0.5
    plan = gd.Plan(c["q_off"], c["kv_off"], 4, d)
    plan.set_kernel("tcgen05")
    nf, nb, S = plan.sizes()
    assert min(nf, nb) >= S
    plan.set_wait_test(limit_us=20000, stall=True)
    t0 = time.time()
    if which == "fwd":
        gd.gdpa_fwd(plan, c["q"], c["k"], c["v"], alpha=alpha, act="gelu_erf")
    else:
        gd.gdpa_bwd(plan, c["q"], c["k"], c["v"], c["do"], alpha=alpha, act="gelu_erf")
    with pytest.raises(gd.GdpaError) as e:
        plan.check()
    assert e.value.status == TIMEOUT
    # where: an abandoned wait (device code 1) at one of this kernel's wait
    # sites, first given up by the stalled CTA 0
    code, site, cta, _ = plan.error_detail()
    assert code == 1 and cta == 0, plan.error_detail()
    assert (1 <= site <= 16) if which == "fwd" else (21 <= site <= 50), site
    # the kernel returned well inside the default limit (2 s per wait)
    assert time.time() - t0 < 10.0
    # the flag is cleared and the device is usable: a normal launch on the
    # same plan matches the oracle
    plan.set_wait_test(0, False)
    args = (c["q_off"], c["kv_off"], c["q"], c["k"], c["v"])
    if which == "fwd":
        o = gd.gdpa_fwd(plan, c["q"], c["k"], c["v"], alpha=alpha, act="gelu_erf")
        plan.check()
        check({"o": max_rel(ref.to_f64(o), ref.fwd(*args, alpha, "gelu_erf"))}, TOL["bf16"])
    else:
        grads = gd.gdpa_bwd(plan, c["q"], c["k"], c["v"], c["do"], alpha=alpha, act="gelu_erf")
        plan.check()
        want = ref.bwd(*args, c["do"], alpha, "gelu_erf")
        check({name: max_rel(ref.to_f64(g), w) for name, g, w in zip(("dq", "dk", "dv"), grads, want)},
              TOL["bf16"])
    plan.check()
    plan.destroy()
    torch.cuda.synchronize()


def test_plan_refused_on_another_device(gd):
    import torch
    if torch.cuda.device_count() < 2:
        pytest.skip("needs a second device")
    c = _case(128)
    plan = gd.Plan(c["q_off"], c["kv_off"], 4, 128)
    with torch.cuda.device(1):
        st = gd.lib().gdpa_check(plan.handle, None)
        assert st == 1   # GDPA_ERR_INVALID_ARG, refused before touching the device
    plan.check()
    plan.destroy()


def test_destroy_does_not_wait_for_other_streams(gd):
    """Destroying a plan waits (on the device) for the plan's own launches
    only: the outputs of a launch queued just before destroy are complete and
    correct, and a long kernel on an unrelated stream does not block it."""
    import torch
    c = _case(128)
    alpha = 128 ** -0.5
    plan = gd.Plan(c["q_off"], c["kv_off"], 4, 128)
    o = gd.gdpa_fwd(plan, c["q"], c["k"], c["v"], alpha=alpha, act="silu")
    plan.destroy()   # returns at once; the forward still reads the plan
    torch.cuda.synchronize()
    check({"o": max_rel(ref.to_f64(o), ref.fwd(c["q_off"], c["kv_off"], c["q"], c["k"], c["v"],
                                                 alpha, "silu"))}, TOL["bf16"])
    side = torch.cuda.Stream()
    big = torch.randn(4096, 4096, device="cuda")
    torch.cuda.synchronize()
    plan = gd.Plan(c["q_off"], c["kv_off"], 4, 128)
    gd.gdpa_fwd(plan, c["q"], c["k"], c["v"], alpha=alpha, act="silu")
    with torch.cuda.stream(side):
        # float32 products on an unrelated stream: well over 100 ms of work
        for _ in range(60):
            big = big @ big.T
            big = big / big.norm()
    t0 = time.perf_counter()
    plan.destroy()
    dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    assert np.isfinite(dt) and dt < 0.05, dt
