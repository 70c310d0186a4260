"""The host tile plan, restated in plain Python (TEST INFRASTRUCTURE ONLY).

The GDPA page ("범용 내적 어텐션(GDPA) ...", aitrends.kr) says, in the
paragraph on jagged inputs and the zigzag-scheduling diagram after it, that
the CPU precomputes the valid tiles from the jagged lengths and assigns them
to SMs in a zigzag pattern after sorting them, instead of round robin.  The
page gives no further detail; the rules below are this project's reading,
and the library's C++ planner must reproduce them bit for bit.

Forward tiles, one per (sample b, head h, query tile m), enumerated b -> h -> m:
  query rows [m*BM, min((m+1)*BM, Lq)); the key range is the hull of the valid
  keys of those rows: [0, Lkv) without a mask, and with a causal window W
  [max(0, m*BM - W + 1), min(Lkv, (m+1)*BM, Lq)).  An empty range gives a
  zero tile (kb0 = kb1 = 0, its rows are written as zeros); otherwise the key
  blocks are [lo // BN, ceil(hi / BN)), optionally cut into chunks of at most
  ``max_kv_blocks`` blocks (enumerated in increasing kb0).

Backward units, one per (b, h, key block j), enumerated b -> h -> j:
  key rows [j*BN, min((j+1)*BN, Lkv)); query hull [0, Lq) without a mask,
  [j*BN, min(Lq, min((j+1)*BN, Lkv) - 1 + W)) with the window; query tiles
  [lo // BM, ceil(hi / BM)), or a zero unit (m0 = m1 = 0) if empty.  Flag bit 0
  (dQ by atomic add) is set on every unit of a sample in which some query
  tile is covered by more than one unit of the same head.

Cost w = number of blocks on the inner loop (kb1 - kb0 forward, m1 - m0
backward).  Zigzag: stable sort by w descending, the r-th tile goes to round
r // S, position p = r % S, SM p on even rounds and S - 1 - p on odd ones.
Round robin: the r-th tile in enumeration order goes to SM r % S.  Each SM's
queue keeps the dealing order.

Timed zigzag (the library's GDPA_SCHED_ZIGZAG_TIMED) deals like zigzag, with
the backward units' w from an integer time model (50 ns units) of the
tensor-core backward: 36 + 22 K/128 plus 40 + 34 q/128 + 24 K/128 for each of
the unit's query tiles, where q is a query tile's rows rounded up to 32 and K
the unit's keys rounded up to 16, every division an integer one; an empty
unit costs 1.  Forward tiles keep w = key blocks.
"""

from __future__ import annotations

import numpy as np


def _cdiv(a, b):
    return -(-a // b)


def fwd_tiles(q_off, kv_off, H, BM=128, BN=128, mask="none", window=0, max_kv_blocks=0):
    q_off = [int(x) for x in q_off]
    kv_off = [int(x) for x in kv_off]
    out = []
    for b in range(len(q_off) - 1):
        lq = q_off[b + 1] - q_off[b]
        lkv = kv_off[b + 1] - kv_off[b]
        for h in range(H):
            for m in range(_cdiv(lq, BM)):
                r0, r1 = m * BM, min((m + 1) * BM, lq)
                if mask == "causal_window":
                    lo, hi = max(0, r0 - window + 1), min(lkv, r1)
                else:
                    lo, hi = 0, lkv
                if lo >= hi:
                    out.append((b, h, m, 0, 0))
                    continue
                k0, k1 = lo // BN, _cdiv(hi, BN)
                if max_kv_blocks <= 0:
                    out.append((b, h, m, k0, k1))
                else:
                    for s in range(k0, k1, max_kv_blocks):
                        out.append((b, h, m, s, min(s + max_kv_blocks, k1)))
    return out


def bwd_units(q_off, kv_off, H, BM=128, BN=128, mask="none", window=0):
    """Returns (units, zero_dq): units are (b, h, j, m0, m1, flags)."""
    q_off = [int(x) for x in q_off]
    kv_off = [int(x) for x in kv_off]
    out = []
    zero_dq = False
    for b in range(len(q_off) - 1):
        lq = q_off[b + 1] - q_off[b]
        lkv = kv_off[b + 1] - kv_off[b]
        ranges = []
        for j in range(_cdiv(lkv, BN)):
            c0, c1 = j * BN, min((j + 1) * BN, lkv)
            if mask == "causal_window":
                lo, hi = c0, min(lq, c1 - 1 + window)
            else:
                lo, hi = 0, lq
            ranges.append((lo // BM, _cdiv(hi, BM)) if lo < hi else (0, 0))
        nonempty = [r for r in ranges if r[1] > r[0]]
        atomic = any(nonempty[i][1] > nonempty[i + 1][0] for i in range(len(nonempty) - 1))
        covered = set()
        for r in nonempty:
            covered.update(range(r[0], r[1]))
        if atomic or len(covered) != _cdiv(lq, BM):
            zero_dq = True
        for h in range(H):
            for j, (m0, m1) in enumerate(ranges):
                out.append((b, h, j, m0, m1, 1 if atomic else 0))
    return out, zero_dq


def _round_up(a, m):
    return _cdiv(a, m) * m


def bwd_time(unit, q_off, kv_off, BM=128, BN=128):
    """Timed-zigzag cost of a backward unit (b, h, j, m0, m1, flags)."""
    b, _, j, m0, m1 = unit[:5]
    if m1 <= m0:
        return 1
    lq = int(q_off[b + 1]) - int(q_off[b])
    lkv = int(kv_off[b + 1]) - int(kv_off[b])
    keys = _round_up(min(BN, lkv - j * BN), 16)
    cost = 36 + (22 * keys) // 128
    for m in range(m0, m1):
        rows = _round_up(min(BM, lq - m * BM), 32)
        cost += 40 + (34 * rows) // 128 + (24 * keys) // 128
    return cost


def deal(costs, S, policy="zigzag"):
    """SM of every item (by item index) and the per-SM queues (lists of item indices)."""
    n = len(costs)
    if policy in ("zigzag", "zigzag_timed"):
        order = sorted(range(n), key=lambda i: (-costs[i], i))
    elif policy == "round_robin":
        order = list(range(n))
    else:
        raise ValueError(policy)
    sm = [0] * n
    queues = [[] for _ in range(S)]
    for r, i in enumerate(order):
        p = r % S
        if policy in ("zigzag", "zigzag_timed") and (r // S) % 2 == 1:
            p = S - 1 - p
        sm[i] = p
        queues[p].append(i)
    return sm, queues


def plan(q_off, kv_off, H, S, BM=128, BN=128, mask="none", window=0,
         policy="zigzag", max_kv_blocks=0):
    """The full plan as NumPy arrays in the layout the library exports.

    ``fwd``: int32 [n, 6] rows (b, h, m, kb0, kb1, sm) in queue order (SM 0's
    queue first); ``fwd_seg``: int32 [S + 1] queue starts.  ``bwd``: int32
    [n, 7] rows (b, h, j, m0, m1, flags, sm); ``bwd_seg`` likewise.
    """
    ft = fwd_tiles(q_off, kv_off, H, BM, BN, mask, window, max_kv_blocks)
    bu, zero_dq = bwd_units(q_off, kv_off, H, BM, BN, mask, window)
    res = {"zero_dq": zero_dq}
    fcost = lambda t: t[4] - t[3]  # noqa: E731
    if policy == "zigzag_timed":
        bcost = lambda u: bwd_time(u, q_off, kv_off, BM, BN)  # noqa: E731
    else:
        bcost = lambda u: u[4] - u[3]  # noqa: E731
    for name, items, cost_of in (("fwd", ft, fcost), ("bwd", bu, bcost)):
        costs = [cost_of(t) for t in items]
        sm, queues = deal(costs, S, policy)
        rows, seg = [], [0]
        for s in range(S):
            for i in queues[s]:
                rows.append(tuple(items[i]) + (s,))
            seg.append(len(rows))
        width = 6 if name == "fwd" else 7
        res[name] = np.array(rows, dtype=np.int32).reshape(-1, width)
        res[name + "_seg"] = np.array(seg, dtype=np.int32)
        res[name + "_work"] = np.array([sum(costs[i] for i in queues[s]) for s in range(S)],
                                       dtype=np.int64)
    return res


def shard_samples(q_off, kv_off, H, R, BM=128, BN=128, mask="none", window=0):
    """Samples of one batch dealt to R ranks (the library's gdpa_shard_batch):
    a sample's work is H times the key blocks of its forward tiles (the
    forward tile cost, summed over the sample); stable sort by work,
    descending, then snake dealing over the ranks.  Returns (rank of each
    sample, work of each rank)."""
    q_off = [int(x) for x in q_off]
    B = len(q_off) - 1
    work = [0] * B
    for t in fwd_tiles(q_off, kv_off, 1, BM, BN, mask, window):
        work[t[0]] += (t[4] - t[3]) * H
    rank, queues = deal(work, R, "zigzag")
    return rank, [sum(work[b] for b in q) for q in queues]
