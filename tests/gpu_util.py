"""Helpers shared by the GPU parity tests: run the library through its C ABI
and compare with the float64 oracle on the same inputs."""

from __future__ import annotations

import os

import numpy as np

from oracle import ref
from workloads import make_inputs, small_case

TOL = {"f32": 1e-5, "bf16": 1e-2}

# Every checked error with its tolerance, for the end-of-run margin summary
# (tests/conftest.py): (test id, quantity, max relative error, tolerance).
MARGINS = []


def record(errs, tol):
    """Note each error of `errs` ({name: max relative error}) against `tol`."""
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    for name, e in errs.items():
        MARGINS.append((test, name, float(e), float(tol)))


def check(errs, tol):
    """Record, then assert every error is within `tol`."""
    record(errs, tol)
    for name, e in errs.items():
        assert e <= tol, "%s: max rel err %.3e > %.1e (%s)" % (name, e, tol, errs)


def max_rel(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if want.size == 0:
        return 0.0
    scale = float(np.max(np.abs(want)))
    err = float(np.max(np.abs(got - want)))
    if scale == 0.0:
        return err
    return err / scale


def to_dev(case, device="cuda"):
    out = dict(case)
    for n in ("q", "k", "v", "do"):
        if out.get(n) is not None:
            out[n] = out[n].to(device).contiguous()
    return out


def run_gpu(gd, x, H, d, alpha, act, mask="none", window=0, kernel="auto", backward=True,
            sched="zigzag", num_sms=0, stream=None, max_kv_blocks=0):
    import torch
    plan = gd.Plan(x["q_off"], x["kv_off"], H, d, mask=mask, window=window, sched=sched,
                   num_sms=num_sms, stream=stream, max_kv_blocks=max_kv_blocks)
    plan.set_kernel(kernel)
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())
    o = gd.gdpa_fwd(plan, x["q"], x["k"], x["v"], alpha=alpha, act=act, stream=stream)
    grads = None
    if backward:
        grads = gd.gdpa_bwd(plan, x["q"], x["k"], x["v"], x["do"], alpha=alpha, act=act,
                            stream=stream)
    plan.check(stream)
    torch.cuda.synchronize()
    return plan, o, grads


def compare_full(gd, x, H, d, alpha, act, dtype, mask="none", window=0, kernel="auto",
                 backward=True, **launch):
    """Whole-batch comparison; returns the max relative errors.  `launch` goes
    to run_gpu (sched, num_sms, stream, max_kv_blocks)."""
    plan, o, grads = run_gpu(gd, x, H, d, alpha, act, mask, window, kernel, backward, **launch)
    args = (x["q_off"], x["kv_off"], x["q"], x["k"], x["v"])
    errs = {"o": max_rel(ref.to_f64(o), ref.fwd(*args, alpha, act, mask, window))}
    if backward:
        rg = ref.bwd(*args, x["do"], alpha, act, mask, window)
        for name, g, r in zip(("dq", "dk", "dv"), grads, rg):
            errs[name] = max_rel(ref.to_f64(g), r)
    plan.destroy()
    return errs


def compare_sampled(gd, x, samples, H, d, alpha, act, mask="none", window=0, kernel="auto",
                    backward=False):
    """Run the whole batch on the GPU, check the listed samples with the oracle."""
    import torch
    plan, o, grads = run_gpu(gd, x, H, d, alpha, act, mask, window, kernel, backward)
    sq, skv, qi, kvi = ref.sub_batch(x["q_off"], x["kv_off"], samples)
    qi_t = torch.from_numpy(qi).to(x["q"].device)
    kvi_t = torch.from_numpy(kvi).to(x["q"].device)
    sub = [x["q"].index_select(0, qi_t), x["k"].index_select(0, kvi_t),
           x["v"].index_select(0, kvi_t)]
    errs = {"o": max_rel(ref.to_f64(o.index_select(0, qi_t)),
                         ref.fwd(sq, skv, *sub, alpha, act, mask, window))}
    if backward:
        dsub = x["do"].index_select(0, qi_t)
        rg = ref.bwd(sq, skv, *sub, dsub, alpha, act, mask, window)
        for name, g, r, idx in zip(("dq", "dk", "dv"), grads, rg, (qi_t, kvi_t, kvi_t)):
            errs[name] = max_rel(ref.to_f64(g.index_select(0, idx)), r)
    plan.destroy()
    return errs


def pick_samples(q_off, kv_off, n_random=4, seed=0):
    """Longest / shortest query and key samples plus a few seeded random ones."""
    lq = np.diff(np.asarray(q_off, dtype=np.int64))
    lkv = np.diff(np.asarray(kv_off, dtype=np.int64))
    picks = [int(np.argmax(lq)), int(np.argmin(lq)), int(np.argmax(lkv)), int(np.argmin(lkv)),
             len(lq) - 1]
    rng = np.random.Generator(np.random.PCG64(seed))
    picks += [int(i) for i in rng.integers(0, len(lq), size=n_random)]
    return sorted(set(picks))


__all__ = ["MARGINS", "TOL", "check", "compare_full", "record", "compare_sampled", "make_inputs", "max_rel", "pick_samples",
           "small_case", "to_dev"]
