"""gdpa_fwd_noalloc, the forward for callers that cannot allocate device
memory (code inside a device allocator or memory pool, plugins given one
fixed arena, processes that reserve all memory up front), against the
planned forward gdpa_fwd on the same inputs, through the C ABI.

pytest collects this file last, so that a run stopping at its first failure
has run every other test before it; it sets up its own inputs and passes
alone in a fresh process as well.
"""

import ctypes

import numpy as np
import pytest

from gpu_util import TOL, check, max_rel, small_case, to_dev
from oracle import ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gd():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import recommender_model_attention_gb300 as g
    g.build()
    return g


def _call(gd, c, H, d, act, mask, window, o):
    import torch
    L = gd.lib()
    qo = np.ascontiguousarray(c["q_off"], dtype=np.int32)
    ko = np.ascontiguousarray(c["kv_off"], dtype=np.int32)
    i32p = ctypes.POINTER(ctypes.c_int32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return L.gdpa_fwd_noalloc(qo.ctypes.data_as(i32p), ko.ctypes.data_as(i32p), len(qo) - 1, H, d,
                              gd.MASK[mask], window, p(c["q"]), p(c["k"]), p(c["v"]), p(o),
                              ctypes.c_float(d ** -0.5), gd.ACT[act],
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    dict(seed=41, B=6, H=2, d=128, q_range=(1, 600), kv_range=None, act="silu",
         mask="causal_window", window=200),
    dict(seed=42, B=9, H=3, d=64, q_range=(1, 300), kv_range=(1, 200), act="gelu_erf",
         mask="none", window=0),
]


def _case(case):
    return to_dev(small_case(case["seed"], B=case["B"], H=case["H"], d=case["d"],
                             q_range=case["q_range"], kv_range=case["kv_range"], dtype="bf16",
                             rmsnorm=True))


def _planned(gd, c, case):
    plan = gd.Plan(c["q_off"], c["kv_off"], case["H"], case["d"], mask=case["mask"],
                   window=case["window"])
    want = gd.gdpa_fwd(plan, c["q"], c["k"], c["v"], act=case["act"])
    plan.check()
    plan.destroy()
    return want


def test_noalloc_matches_planned_forward_on_consecutive_calls(gd):
    """Same kernel, same zigzag plan over the same SMs, no atomics: the two
    entry points give the same bytes, and so the same oracle margin."""
    import torch
    for case in CASES:
        c = _case(case)
        want = _planned(gd, c, case)
        ref_err = max_rel(want.double().cpu().numpy(),
                          ref.fwd(c["q_off"], c["kv_off"], c["q"], c["k"], c["v"],
                                  case["d"] ** -0.5, case["act"], case["mask"], case["window"]))
        check({"o": ref_err}, TOL["bf16"])
        for _ in range(2):
            o = torch.full_like(c["q"], float("nan"))
            st = _call(gd, c, case["H"], case["d"], case["act"], case["mask"], case["window"], o)
            assert st == 0, gd.STATUS.get(st, st)
            torch.cuda.synchronize()
            assert torch.equal(o, want)


def test_noalloc_rejects_batch_beyond_scratch(gd):
    import torch
    H, d = 8, 64
    lq = np.ones(4200, dtype=np.int64)             # 4200 samples x 8 heads > 32768 tiles
    off = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    x = torch.zeros((int(off[-1]), H, d), dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(x, 3.0)
    c = {"q_off": off, "kv_off": off, "q": x, "k": x, "v": x}
    st = _call(gd, c, H, d, "gelu_erf", "none", 0, o)
    assert st == 7  # GDPA_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(o == 3.0)
    # a refused call leaves nothing behind that holds back the next one
    case = CASES[1]
    c = _case(case)
    want = _planned(gd, c, case)
    o = torch.full_like(c["q"], float("nan"))
    st = _call(gd, c, case["H"], case["d"], case["act"], case["mask"], case["window"], o)
    assert st == 0, gd.STATUS.get(st, st)
    torch.cuda.synchronize()
    assert torch.equal(o, want)
