"""The benchmark's multi-rank logic on CPU with gloo, world size 2.

Each rank draws its own batch of the same shape (seeded by rank), plans it on
the host with the C++ planner (no GPU), and the job's time is the maximum
over ranks while its work is the sum: the only cross-rank steps of the path,
which otherwise has no data exchange.  The one exchange of the sharded
path, the shared seeds' gradient of pooling attention, is checked too: each
rank's share (from the oracle) summed by the library's all-reduce equals the
gradient of the whole batch.
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


def _seed_worker(rank, world, port, outdir):
    # shared-query pooling sharded by sample: every rank holds the same seeds
    # and its own samples; the oracle gives each rank's share of the seeds'
    # gradient, summed over ranks by the library's one all-reduce
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import recommender_model_attention_gb300 as gd
    from oracle import ref
    seeds, ks, vs, dos, qos, kos = _seed_batches(world)
    qt = ref.shared_q_tokens(seeds, qos[rank])
    dq, _, _ = ref.bwd(qos[rank], kos[rank], qt, ks[rank], vs[rank], dos[rank], 0.3, "gelu_erf")
    g = torch.from_numpy(ref.shared_q_grad(dq, qos[rank], seeds.shape[0])).float()
    gd.allreduce_seed_grad(g)
    np.save(os.path.join(outdir, "seed%d.npy" % rank), g.numpy())
    dist.destroy_process_group()


def _seed_batches(world):
    from workloads import offsets_from_lengths
    g = np.random.default_rng(17)
    seeds = g.standard_normal((4, 2, 8))
    out = ([], [], [], [], [])
    for r in range(world):
        lq = np.array([4, 2, 3]) if r == 0 else np.array([1, 4])
        lkv = np.array([5, 9, 1]) if r == 0 else np.array([7, 3])
        qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
        for lst, t in zip(out, (g.standard_normal((ko[-1], 2, 8)), g.standard_normal((ko[-1], 2, 8)),
                                g.standard_normal((qo[-1], 2, 8)), qo, ko)):
            lst.append(t)
    return (seeds,) + out


def test_shared_seed_gradient_all_reduce_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    from oracle import ref
    from workloads import offsets_from_lengths
    port = _free_port()
    mp.spawn(_seed_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [np.load(tmp_path / ("seed%d.npy" % k)) for k in range(2)]
    assert np.array_equal(got[0], got[1])
    # the whole batch on one process
    seeds, ks, vs, dos, qos, kos = _seed_batches(2)
    lq = np.concatenate([np.diff(q) for q in qos])
    lkv = np.concatenate([np.diff(k) for k in kos])
    qo, ko = offsets_from_lengths(lq), offsets_from_lengths(lkv)
    dq, _, _ = ref.bwd(qo, ko, ref.shared_q_tokens(seeds, qo), np.concatenate(ks),
                       np.concatenate(vs), np.concatenate(dos), 0.3, "gelu_erf")
    want = ref.shared_q_grad(dq, qo, seeds.shape[0])
    assert np.allclose(got[0], want, rtol=1e-5, atol=1e-6)
