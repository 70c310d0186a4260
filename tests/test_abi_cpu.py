"""CPU-side checks of the C-ABI library: it loads, exports every function
that include/gdpa.h declares, and its C++ planner reproduces the oracle's
plan bit for bit (host-only plans, no GPU needed)."""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import planner as ref_planner
from workloads import CONFIGS, draw_lengths, offsets_from_lengths, small_case

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gd():
    import recommender_model_attention_gb300 as g
    g.build()
    return g


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(gdpa_[a-z0-9_]+)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function(gd):
    names = _declared_functions()
    assert "gdpa_fwd" in names and "gdpa_bwd" in names and "gdpa_plan_create" in names
    L = ctypes.CDLL(gd.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def _compare(gd, qo, ko, H, S, mask, window, sched, max_kvb=0):
    p = gd.Plan(qo, ko, H, 128, mask=mask, window=window, sched=sched, num_sms=S,
                max_kv_blocks=max_kvb, host_only=True)
    ref = ref_planner.plan(qo, ko, H, S, mask=mask, window=window, policy=sched,
                           max_kv_blocks=max_kvb)
    tiles, seg = p.export()
    assert np.array_equal(tiles, ref["fwd"].reshape(-1, 6))
    assert np.array_equal(seg, ref["fwd_seg"])
    units, useg, zero_dq = p.export_bwd()
    assert np.array_equal(units, ref["bwd"].reshape(-1, 7))
    assert np.array_equal(useg, ref["bwd_seg"])
    assert zero_dq == ref["zero_dq"]
    p.destroy()


@pytest.mark.parametrize("cfg", CONFIGS, ids=[c.name for c in CONFIGS])
@pytest.mark.parametrize("sched", ["zigzag", "round_robin", "zigzag_timed"])
def test_planner_matches_oracle_on_workloads(gd, cfg, sched):
    lq, lkv = draw_lengths(cfg)
    qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
    if cfg.index == 4 and sched == "round_robin":
        pytest.skip("same enumeration already covered by zigzag on this workload")
    _compare(gd, qo, ko, cfg.H, 152, cfg.mask, cfg.window, sched)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("S", [1, 5, 152])
def test_planner_matches_oracle_random(gd, seed, S):
    mask = "causal_window" if seed % 2 else "none"
    c = small_case(seed, B=9, H=1, d=1, q_range=(0, 700),
                   kv_range=None if mask == "causal_window" else (0, 400), zero_lengths=True)
    for sched in ("zigzag", "round_robin", "zigzag_timed"):
        _compare(gd, c["q_off"], c["kv_off"], 3, S, mask, 1 + 37 * seed, sched,
                 max_kvb=(seed % 3))


@pytest.mark.parametrize("mask,window", [("none", 0), ("causal_window", 300),
                                         ("causal_window", 1200)])
def test_planner_automatic_key_split(gd, mask, window):
    # "auto" resolves to 2-block chunks when some query tile's key hull has
    # 8 or more blocks, else to no split: compare with the explicit plans
    for lkv_max, seed in ((1000, 1), (1100, 2), (3000, 3)):
        rng = np.random.default_rng(seed)
        lq = rng.integers(1, 400, size=7)
        lkv = rng.integers(0, lkv_max, size=7) if mask == "none" else lq
        if mask == "causal_window":
            lq = lkv = rng.integers(1, lkv_max, size=7)
        qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
        widest = 0
        for t in ref_planner.fwd_tiles(qo, ko, 1, 128, 128, mask, window):
            widest = max(widest, t[4] - t[3])
        want = 2 if widest >= 8 else 0
        auto = gd.Plan(qo, ko, 2, 128, mask=mask, window=window, num_sms=19,
                       max_kv_blocks="auto", host_only=True)
        expl = gd.Plan(qo, ko, 2, 128, mask=mask, window=window, num_sms=19,
                       max_kv_blocks=want, host_only=True)
        for a, b in zip(auto.export(), expl.export()):
            assert np.array_equal(a, b)
        auto.destroy()
        expl.destroy()


def test_planner_rejects_bad_arguments(gd):
    from recommender_model_attention_gb300 import GdpaError
    good = offsets_from_lengths([3, 4])
    bad = np.array([0, 5, 4], dtype=np.int32)
    with pytest.raises(GdpaError) as e:
        gd.Plan(bad, good, 1, 64, num_sms=4, host_only=True)
    assert e.value.status == 1
    with pytest.raises(GdpaError) as e:
        gd.Plan(np.array([1, 3, 4], np.int32), good, 1, 64, num_sms=4, host_only=True)
    assert e.value.status == 1
    with pytest.raises(GdpaError) as e:
        gd.Plan(good, good, 1, 130, num_sms=4, host_only=True)
    assert e.value.status == 2
    with pytest.raises(GdpaError) as e:
        gd.Plan(good, good, 1, 64, mask="causal_window", window=0, num_sms=4, host_only=True)
    assert e.value.status == 1
    with pytest.raises(GdpaError) as e:
        gd.Plan(good, good, 1, 64, num_sms=0, host_only=True)
    assert e.value.status == 1
    with pytest.raises(GdpaError) as e:
        gd.Plan(good, good, 1, 64, num_sms=4, max_kv_blocks=-2, host_only=True)
    assert e.value.status == 1


def test_shared_q_needs_enough_seeds(gd):
    from recommender_model_attention_gb300 import GdpaError
    qo = offsets_from_lengths([32, 5, 0])
    p = gd.Plan(qo, qo, 1, 128, num_sms=4, host_only=True)
    with pytest.raises(GdpaError) as e:
        p.set_shared_q(31)          # a sample has 32 queries
    assert e.value.status == 1
    with pytest.raises(GdpaError) as e:
        p.set_shared_q(-1)
    assert e.value.status == 1
    p.set_shared_q(32)
    assert p.q_rows == 32
    p.set_shared_q(0)
    assert p.q_rows == 37
    p.destroy()


def test_host_only_plan_cannot_launch(gd):
    off = offsets_from_lengths([3, 4])
    p = gd.Plan(off, off, 1, 64, num_sms=4, host_only=True)
    L = gd.lib()
    st = L.gdpa_fwd(p.handle, 0, None, None, None, None, ctypes.c_float(1.0), 0, None)
    assert st == 1
    p.destroy()


def test_empty_batch_plan(gd):
    off = np.zeros(1, dtype=np.int32)
    p = gd.Plan(off, off, 2, 64, num_sms=4, host_only=True)
    tiles, seg = p.export()
    assert tiles.shape == (0, 6) and np.all(seg == 0)
    p.destroy()


def test_shard_batch_hand_worked(gd):
    # worked by hand from the rule in include/gdpa.h (H = 2, two ranks):
    # sample 0: Lq 300 -> 3 query tiles x 1 key block (Lkv 100), work 3 x 2 = 6
    # sample 1: Lq 5 -> 1 tile x 3 key blocks (Lkv 300), work 3 x 2 = 6
    # sample 2: Lq 0 -> no tile, work 0
    # sample 3: Lq 129 -> 2 tiles x 1 block, work 2 x 2 = 4
    # sorted (stable, descending): 0, 1, 3, 2; ranks 0, 1 (round 0), then 1, 0
    qo = offsets_from_lengths([300, 5, 0, 129])
    ko = offsets_from_lengths([100, 300, 10, 1])
    rank, work = gd.shard_batch(qo, ko, 2, 2)
    assert list(rank) == [0, 1, 0, 1]
    assert list(work) == [6, 10]


@pytest.mark.parametrize("cfg", CONFIGS, ids=[c.name for c in CONFIGS])
@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_shard_batch_matches_oracle(gd, cfg, R):
    lq, lkv = draw_lengths(cfg)
    qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
    rank, work = gd.shard_batch(qo, ko, cfg.H, R, cfg.mask, cfg.window)
    want_rank, want_work = ref_planner.shard_samples(qo, ko, cfg.H, R, mask=cfg.mask,
                                                     window=cfg.window)
    assert list(rank) == list(want_rank)
    assert list(work) == list(want_work)
    # every sample's work lands on some rank, and every rank gets work when
    # there are enough samples
    assert work.sum() == sum(want_work)
    if len(lq) >= R:
        assert work.min() > 0


def test_shard_rows_partition(gd):
    c = small_case(5, B=11, H=1, d=1, q_range=(0, 90), kv_range=(0, 70), zero_lengths=True)
    rank, _ = gd.shard_batch(c["q_off"], c["kv_off"], 1, 3)
    seen_q, seen_k = [], []
    for r in range(3):
        lo, lk, qi, ki, mine = gd.shard_rows(c["q_off"], c["kv_off"], rank, r)
        assert list(np.diff(lo)) == [int(c["q_off"][b + 1] - c["q_off"][b]) for b in mine]
        assert list(np.diff(lk)) == [int(c["kv_off"][b + 1] - c["kv_off"][b]) for b in mine]
        assert len(qi) == lo[-1] and len(ki) == lk[-1]
        seen_q += list(qi)
        seen_k += list(ki)
    assert sorted(seen_q) == list(range(int(c["q_off"][-1])))
    assert sorted(seen_k) == list(range(int(c["kv_off"][-1])))


def test_shard_batch_refuses_bad_arguments(gd):
    qo = offsets_from_lengths([3, 4])
    with pytest.raises(gd.GdpaError):
        gd.shard_batch(qo, qo, 1, 0)
    with pytest.raises(gd.GdpaError):
        gd.shard_batch(np.array([1, 2, 3]), qo, 1, 2)


def test_qk_norm_argument_checks(gd):
    qo = offsets_from_lengths([3, 4])
    p = gd.Plan(qo, qo, 2, 64, num_sms=4, host_only=True)
    p.set_qk_norm(1.0, 1e-6)
    p.set_qk_norm(0.0, 0.0)          # off
    for gain, eps in ((-1.0, 1e-6), (1.0, 0.0), (1.0, -1e-3), (float("nan"), 1e-6)):
        with pytest.raises(gd.GdpaError):
            p.set_qk_norm(gain, eps)
    p.destroy()


def test_mx_argument_checks_on_the_host(gd):
    # the MXFP8 entry points refuse bad sizes and pointers before touching a
    # device: counts that are not a multiple of the 32-value block, NULL or
    # misaligned buffers; n = 0 is a no-op
    import ctypes
    L = gd.lib()
    vp = ctypes.c_void_p
    a = vp(1 << 20)   # an aligned address that is never dereferenced
    assert L.gdpa_mx_quantise(a, 48, a, a, None) == 1
    assert L.gdpa_mx_quantise(a, -32, a, a, None) == 1
    assert L.gdpa_mx_quantise(None, 32, a, a, None) == 1
    assert L.gdpa_mx_quantise(vp((1 << 20) + 8), 32, a, a, None) == 1
    assert L.gdpa_mx_dequantise(a, a, 31, a, None) == 1
    assert L.gdpa_mx_dequantise(vp((1 << 20) + 4), a, 32, a, None) == 1
    assert L.gdpa_mx_quantise(None, 0, None, None, None) == 0
    assert L.gdpa_mx_dequantise(None, None, 0, None, None) == 0
    # the plan forms: a NULL plan, and a host-only plan, are refused
    assert L.gdpa_fwd_mx(None, a, a, a, a, a, a, ctypes.c_float(1.0), 0, None) == 1
    qo = offsets_from_lengths([3, 4])
    p = gd.Plan(qo, qo, 2, 64, num_sms=4, host_only=True)
    assert L.gdpa_fwd_mx(p.handle, a, a, a, a, a, a, ctypes.c_float(1.0), 0, None) == 1
    assert L.gdpa_bwd_mx(p.handle, a, a, a, a, a, a, a, a, a, ctypes.c_float(1.0), 0, None) == 1
    p.destroy()


def test_act_eval_argument_checks_on_the_host(gd):
    # the activation test hook refuses an unknown activation or form, a
    # negative count and NULL arrays before touching a device; n = 0 is a
    # no-op
    import ctypes
    L = gd.lib()
    vp = ctypes.c_void_p
    a = vp(1 << 20)   # never dereferenced
    n = ctypes.c_int64
    assert L.gdpa_act_eval(0, 3, a, a, a, n(8), None) == 1
    assert L.gdpa_act_eval(0, -1, a, a, a, n(8), None) == 1
    assert L.gdpa_act_eval(5, 1, a, a, a, n(8), None) == 1   # softmax is a row operation
    assert L.gdpa_act_eval(0, 2, a, a, a, n(-1), None) == 1
    assert L.gdpa_act_eval(0, 2, None, a, a, n(8), None) == 1
    assert L.gdpa_act_eval(0, 2, None, None, None, n(0), None) == 0


def test_error_detail_on_the_host(gd):
    # the last-failure record is a host-side copy: zeros before any failure,
    # and refused for a NULL plan or output
    import ctypes
    L = gd.lib()
    d = (ctypes.c_int32 * 4)(9, 9, 9, 9)
    assert L.gdpa_error_detail(None, d) == 1
    qo = offsets_from_lengths([3, 4])
    p = gd.Plan(qo, qo, 2, 64, num_sms=4, host_only=True)
    assert L.gdpa_error_detail(p.handle, None) == 1
    assert p.error_detail() == (0, 0, 0, 0)
    p.destroy()
