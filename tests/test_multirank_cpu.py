"""The benchmark's multi-rank logic on CPU with gloo, world size 2.

Each rank draws its own batch of the same shape (seeded by rank), plans it on
the host with the C++ planner (no GPU), and the job's time is the maximum
over ranks while its work is the sum: the only cross-rank steps of the path,
which otherwise has no data exchange.
"""

import json
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import recommender_model_attention_gb300 as gd
    from workloads import draw_lengths, get_config, make_inputs
    w = get_config("training_cross_fwd_bwd")
    lq, lkv = draw_lengths(w)
    lq, lkv = np.minimum(lq[:6], 300), lkv[:6]
    x = make_inputs(w, device="cpu", seed=bench.rank_seed(w, rank), lengths=(lq, lkv))
    plan = gd.Plan(x["q_off"], x["kv_off"], w.H, w.d, num_sms=152, host_only=True)
    n_fwd, n_bwd, _ = plan.sizes()
    pairs = bench.useful_pairs(x["q_off"], x["kv_off"], w.mask, w.window)
    ms, flops = bench.reduce_across_ranks(10.0 + 5.0 * rank, 12.0 * w.d * w.H * pairs, "cpu")
    sums = [None] * world
    dist.all_gather_object(sums, float(x["q"].float().sum()))
    with open(os.path.join(outdir, "rank%d.json" % rank), "w") as f:
        json.dump({"ms": ms, "flops": flops, "n_fwd": n_fwd, "n_bwd": n_bwd, "pairs": pairs,
                   "q_sums": sums}, f)
    dist.destroy_process_group()


def test_two_ranks_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    pytest.importorskip("torch.distributed")
    import recommender_model_attention_gb300 as gd
    gd.build()
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    r = [json.load(open(tmp_path / ("rank%d.json" % k))) for k in range(2)]
    # same shape on both ranks (same plan sizes and work), different data
    assert r[0]["n_fwd"] == r[1]["n_fwd"] and r[0]["n_bwd"] == r[1]["n_bwd"]
    assert r[0]["q_sums"][0] != r[0]["q_sums"][1]
    # job time = slowest rank, job work = sum over ranks, identical on every rank
    for k in range(2):
        assert r[k]["ms"] == 15.0
        assert r[k]["flops"] == pytest.approx(2 * 12.0 * 128 * 8 * r[0]["pairs"])
