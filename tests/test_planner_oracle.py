"""Pins of the oracle's tile planner (CPU only): a hand-worked dealing, brute
force over all (query, key) pairs for the tile and unit ranges, and the
invariants of the dealing policies."""

import os

import numpy as np
import pytest

from oracle import planner
from workloads import draw_lengths, get_config, offsets_from_lengths, small_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                out[k] = [int(x) for x in v]
    return out


def test_zigzag_hand_worked_example():
    g = _read("zigzag_worked_example.txt")
    S = g["S"][0]
    costs = g["costs"]
    sm, queues = planner.deal(costs, S, "zigzag")
    assert sm == g["zigzag_sm"]
    for s in range(S):
        assert queues[s] == g["zigzag_queue%d" % s]
    assert [sum(costs[i] for i in q) for q in queues] == g["zigzag_work"]
    sm, queues = planner.deal(costs, S, "round_robin")
    assert sm == g["round_robin_sm"]
    assert [sum(costs[i] for i in q) for q in queues] == g["round_robin_work"]


def _valid(i, j, lq, lkv, mask, W):
    if i >= lq or j >= lkv:
        return False
    return (j <= i and j > i - W) if mask == "causal_window" else True


CASES = [
    dict(seed=0, B=6, q_range=(1, 300), kv_range=(1, 300), mask="none", W=0),
    dict(seed=1, B=6, q_range=(1, 400), kv_range=None, mask="causal_window", W=100),
    dict(seed=2, B=5, q_range=(1, 600), kv_range=None, mask="causal_window", W=256),
    dict(seed=3, B=8, q_range=(0, 300), kv_range=(0, 200), mask="none", W=0),
    dict(seed=4, B=4, q_range=(100, 500), kv_range=(1, 130), mask="causal_window", W=20),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("BM,BN", [(128, 128), (64, 128), (128, 64)])
def test_tiles_cover_exactly_the_valid_pairs(case, BM, BN):
    c = small_case(case["seed"], B=case["B"], H=1, d=1, q_range=case["q_range"],
                   kv_range=case["kv_range"], zero_lengths=True)
    qo, ko = c["q_off"], c["kv_off"]
    mask, W = case["mask"], case["W"]
    H = 2
    tiles = planner.fwd_tiles(qo, ko, H, BM, BN, mask, W)
    units, zero_dq = planner.bwd_units(qo, ko, H, BM, BN, mask, W)
    # brute force: which key blocks hold a valid pair for each query tile,
    # which query tiles hold one for each key block
    expect_tiles = []
    expect_units = []
    need_zero = False
    for b in range(len(qo) - 1):
        lq, lkv = qo[b + 1] - qo[b], ko[b + 1] - ko[b]
        i = np.arange(lq)[:, None]
        j = np.arange(lkv)[None, :]
        V = np.ones((lq, lkv), bool) if mask == "none" else ((j <= i) & (j > i - W))
        nm, nk = -(-lq // BM), -(-lkv // BN)
        blk = np.zeros((nm, nk), bool)
        for m in range(nm):
            for kb in range(nk):
                blk[m, kb] = V[m * BM:(m + 1) * BM, kb * BN:(kb + 1) * BN].any()
        per_tile_units = blk.sum(axis=1)
        atomic = bool((per_tile_units > 1).any())
        if atomic or (per_tile_units == 0).any():
            need_zero = True
        for h in range(H):
            for m in range(nm):
                ks = np.nonzero(blk[m])[0]
                if len(ks) == 0:
                    expect_tiles.append((b, h, m, 0, 0))
                else:
                    assert np.all(np.diff(ks) == 1)
                    expect_tiles.append((b, h, m, int(ks[0]), int(ks[-1]) + 1))
            for kb in range(nk):
                ms = np.nonzero(blk[:, kb])[0]
                if len(ms) == 0:
                    expect_units.append((b, h, kb, 0, 0, int(atomic)))
                else:
                    assert np.all(np.diff(ms) == 1)
                    expect_units.append((b, h, kb, int(ms[0]), int(ms[-1]) + 1, int(atomic)))
    assert tiles == expect_tiles
    assert units == expect_units
    assert zero_dq == need_zero


def test_kv_split_chunks():
    qo = offsets_from_lengths([32, 32])
    ko = offsets_from_lengths([1000, 129])
    tiles = planner.fwd_tiles(qo, ko, 1, 128, 128, "none", 0, max_kv_blocks=3)
    assert tiles == [(0, 0, 0, 0, 3), (0, 0, 0, 3, 6), (0, 0, 0, 6, 8), (1, 0, 0, 0, 2)]


def test_timed_costs_hand_worked_example():
    g = _read("timed_costs_worked_example.txt")
    qo, ko = offsets_from_lengths(g["q_lengths"]), offsets_from_lengths(g["kv_lengths"])
    units, _ = planner.bwd_units(qo, ko, 1)
    assert [planner.bwd_time(u, qo, ko) for u in units] == g["bwd_costs"]


def test_timed_costs_grow_with_work():
    # more keys or more query rows never cost less, and a unit of one query
    # tile costs more than the tile alone (its fixed part)
    for lq in (1, 100, 128, 129, 1000):
        for lkv in (1, 16, 17, 64, 112):
            qo = offsets_from_lengths([lq, lq, lq + 32])
            ko = offsets_from_lengths([lkv, lkv + 16, lkv])
            u, _ = planner.bwd_units(qo, ko, 1)
            c = [planner.bwd_time(x, qo, ko) for x in u]
            assert c[1] >= c[0] and c[2] >= c[0]
            assert c[0] > 40 * len(range(u[0][3], u[0][4]))


@pytest.mark.parametrize("policy", ["zigzag", "round_robin", "zigzag_timed"])
@pytest.mark.parametrize("S", [1, 7, 152])
def test_dealing_invariants(policy, S):
    rng = np.random.Generator(np.random.PCG64(S))
    for trial in range(20):
        costs = list(rng.integers(0, 40, size=int(rng.integers(0, 2000))))
        sm, queues = planner.deal(costs, S, policy)
        flat = sorted(i for q in queues for i in q)
        assert flat == list(range(len(costs)))
        for s, q in enumerate(queues):
            assert all(sm[i] == s for i in q)
            assert (q == sorted(q, key=lambda i: (-costs[i], i)) if policy != "round_robin"
                    else q == sorted(q))
        work = [sum(costs[i] for i in q) for q in queues]
        assert sum(work) == sum(costs)
        if policy != "round_robin" and costs:
            # snake dealing of a descending list: spread at most the largest item
            assert max(work) - min(work) <= max(costs)


def test_plan_export_layout():
    w = get_config("jagged_selfattn_window256")
    lq, lkv = draw_lengths(w)
    qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
    p = planner.plan(qo, ko, w.H, 152, mask=w.mask, window=w.window)
    assert p["fwd"].shape[1] == 6 and p["bwd"].shape[1] == 7
    for name in ("fwd", "bwd"):
        seg = p[name + "_seg"]
        assert seg[0] == 0 and seg[-1] == len(p[name]) and np.all(np.diff(seg) >= 0)
        for s in range(152):
            assert np.all(p[name][seg[s]:seg[s + 1], -1] == s)
    zz = p["fwd_work"]
    rr = planner.plan(qo, ko, w.H, 152, mask=w.mask, window=w.window, policy="round_robin")["fwd_work"]
    assert zz.sum() == rr.sum()
    assert zz.max() - zz.min() <= rr.max() - rr.min()
