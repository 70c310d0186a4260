"""The multi-rank path on CPU with gloo, world size 2.

One batch is sharded over the ranks by the library's gdpa_shard_batch (its
samples dealt by work in zigzag order); each rank runs its own samples as a
batch of their own (here through the float64 oracle, the GPU kernels' stand-
in on a CPU machine) and the outputs and gradients gathered from the ranks equal
those of the whole batch exactly, because samples share nothing.  The job's
time is the slowest rank's measured time and its work the sum of the ranks'
(the benchmark's reduction).  The one exchange of the sharded path, the
shared seeds' gradient of pooling attention, is checked too: each rank's share
(from the oracle) summed by the library's all-reduce equals the gradient of
the whole batch.
"""

import json
import os
import socket
import sys
import time

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    """A jagged batch with the training workload's length mix, small enough
    for the float64 oracle."""
    from workloads import draw_lengths, get_config, make_inputs
    w = get_config("training_cross_fwd_bwd")
    lq, lkv = draw_lengths(w)
    lq, lkv = np.minimum(lq[:24], 300), lkv[:24]
    x = make_inputs(w, device="cpu", seed=77, lengths=(lq, lkv))
    return w, x


def _shard_worker(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import recommender_model_attention_gb300 as gd
    from oracle import ref
    w, x = _batch()
    owner, work = gd.shard_batch(x["q_off"], x["kv_off"], w.H, world)
    lo, lk, qi, ki, mine = gd.shard_rows(x["q_off"], x["kv_off"], owner, rank)
    sub = [x[n].index_select(0, torch.from_numpy(idx)) for n, idx in
           (("q", qi), ("k", ki), ("v", ki), ("do", qi))]
    t0 = time.perf_counter()
    o = ref.fwd(lo, lk, sub[0], sub[1], sub[2], w.alpha, w.act)
    dq, dk, dv = ref.bwd(lo, lk, sub[0], sub[1], sub[2], sub[3], w.alpha, w.act)
    ms = (time.perf_counter() - t0) * 1e3
    flops = 12.0 * w.d * w.H * bench.useful_pairs(lo, lk, w.mask, w.window)
    job_ms, job_flops = bench.reduce_across_ranks(ms, flops, "cpu")
    times = [None] * world
    dist.all_gather_object(times, (ms, flops))
    np.savez(os.path.join(outdir, "shard%d.npz" % rank), o=o, dq=dq, dk=dk, dv=dv, qi=qi, ki=ki,
             mine=mine)
    with open(os.path.join(outdir, "rank%d.json" % rank), "w") as f:
        json.dump({"job_ms": job_ms, "job_flops": job_flops, "times": times,
                   "work": [int(v) for v in work]}, f)
    dist.destroy_process_group()


def test_sharded_batch_equals_whole_batch_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    pytest.importorskip("torch.distributed")
    import recommender_model_attention_gb300 as gd
    from oracle import planner, ref
    gd.build()
    port = _free_port()
    mp.spawn(_shard_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    w, x = _batch()
    args = (x["q_off"], x["kv_off"], x["q"], x["k"], x["v"])
    want_o = ref.fwd(*args, w.alpha, w.act)
    want = ref.bwd(*args, x["do"], w.alpha, w.act)
    got = {n: np.full_like(t, np.nan) for n, t in zip(("o", "dq", "dk", "dv"), (want_o,) + want)}
    owners = []
    for r in range(2):
        z = np.load(tmp_path / ("shard%d.npz" % r))
        owners.append(z["mine"])
        for n, idx in (("o", "qi"), ("dq", "qi"), ("dk", "ki"), ("dv", "ki")):
            got[n][z[idx]] = z[n]
    # every sample on exactly one rank, both ranks busy, as the oracle deals
    allb = np.sort(np.concatenate(owners))
    assert np.array_equal(allb, np.arange(len(x["q_off"]) - 1))
    assert all(len(o) > 0 for o in owners)
    rank_ref, work_ref = planner.shard_samples(x["q_off"], x["kv_off"], w.H, 2)
    assert all(rank_ref[b] == r for r in range(2) for b in owners[r])
    # the gathered shards are the whole batch's result, bit for bit
    for n, ref_t in zip(("o", "dq", "dk", "dv"), (want_o,) + want):
        assert np.array_equal(got[n], ref_t), n
    # job time = slowest rank, job work = sum of the ranks', on every rank
    meta = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    times = meta[0]["times"]
    for m in meta:
        assert m["job_ms"] == max(t[0] for t in times)
        assert m["job_flops"] == pytest.approx(sum(t[1] for t in times))
        assert m["work"] == work_ref


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
