"""GDPA benchmark: one step = forward + backward over one jagged batch.

Default workload: the training step (jagged user-ad cross-attention, B=2048,
H=8, d=128, bf16 inputs, Lq ~ Zipf(1.2) clipped to [1, 4096], Lkv ~ U[8, 128],
GELU-erf, dO ~ N(0, 1)), inputs resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own batch of the same shape (different
seed): the work shards by sample with no exchange, so scaling is weak.  With
``--scaling strong`` every rank draws the same batch and runs the samples that
gdpa_shard_batch deals to it (by work, zigzag order), so the total work is
fixed as the rank count grows.
``--impl reference`` times the float64 CPU oracle on a bounded sample.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "GDPA fwd/bwd useful TFLOP/s on jagged batches; % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM bytes per algorithmic byte of the two tensor-core kernels, from the
# ncu captures summarised in profiles/ (first 256 sequences of the training
# workload; traffic grows with the rows processed, so it is scaled to a full
# launch by algorithmic bytes).  Valid only for the kernel sources they were
# measured on (hash of the kernel's source files), the training workload and
# the unsplit softmax-free kernels without the fused RMSNorm; otherwise
# reported null.
TRAFFIC_WORKLOAD = "training_cross_fwd_bwd"
TRAFFIC_RATIO = {
    "gdpa_fwd": ("2451a965b2c28742", 0.9602),
    "gdpa_bwd": ("583aee4f29bf51c3", 1.0463),
}
KERNEL_SOURCES = {
    "gdpa_fwd": ("gdpa_tc_fwd.cu", "tc_common.cuh", "tc_drain.cuh", "act.cuh", "f2.cuh"),
    "gdpa_bwd": ("gdpa_tc_bwd.cu", "tc_common.cuh", "tc_drain.cuh", "act.cuh", "f2.cuh"),
}


def kernel_source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "recommender_model_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel, algorithmic_bytes, workload, key_split, softmax, qk_norm):
    """DRAM bytes of one launch of `kernel` from its captured ratio, or None
    where the capture does not apply (other kernel sources, another
    workload, the key-split, softmax or fused-RMSNorm kernels)."""
    src_hash, ratio = TRAFFIC_RATIO[kernel]
    if (kernel_source_hash(kernel) != src_hash or workload != TRAFFIC_WORKLOAD or key_split
            or softmax or qk_norm):
        return None
    return ratio * algorithmic_bytes


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(w, rank):
    """Tensor seed of a rank: every rank draws its own batch of the same shape."""
    return 1000 + w.index + 7919 * rank


def reduce_across_ranks(ms, flops, device):
    """(max of `ms`, sum of `flops`) over the process group; identity when the
    job is not distributed.  Whole-job throughput = summed work / slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms), float(flops)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    f = torch.tensor([float(flops)], dtype=torch.float64, device=device)
    dist.all_reduce(f, op=dist.ReduceOp.SUM)
    return float(t.item()), float(f.item())


def useful_pairs(q_off, kv_off, mask, window):
    """Valid (query, key) pairs summed over samples (per head), closed form."""
    lq = np.diff(np.asarray(q_off, dtype=np.int64))
    lkv = np.diff(np.asarray(kv_off, dtype=np.int64))
    if mask == "none":
        return int(np.sum(lq * lkv))
    # causal window on self-attention: sum_i min(i + 1, W) for i < min(Lq, Lkv)
    n = 0
    for a, b in zip(lq, lkv):
        L = min(int(a), int(b))
        W = window
        n += W * (W + 1) // 2 + (L - W) * W if L >= W else L * (L + 1) // 2
    return n


DEFAULT_WORKLOAD = "training_cross_fwd_bwd"
POLICIES = ("zigzag", "round_robin", "zigzag_timed")
OTHER_WORKLOADS = ("jagged_selfattn_window256", "user_ad_cross", "pma_pooling")


def busy_spread(start_end):
    """Max/min and (max - min)/mean of the per-CTA busy times."""
    busy = (start_end[:, 1] - start_end[:, 0]).astype(np.float64)
    return {"max_over_min": float(busy.max() / max(busy.min(), 1.0)),
            "max_minus_min_over_mean": float((busy.max() - busy.min()) / busy.mean())}


def forward_workload(name, gd, pk, pk_kind, sched="zigzag_timed", reps=20, warmup=3):
    """One forward-only workload at its full size, timed launch by launch
    with CUDA events on the launching stream, L2 flushed (a 256 MB write)
    before each timed launch; planner's key split, shared seeds for pooling.
    Returns its line: ms, useful TFLOP/s, % of bf16 peak, GB/s, HBM fraction,
    the attainable roofline and the SM spread of both dealing policies."""
    import torch
    from workloads import get_config, make_inputs
    w = get_config(name)
    x = make_inputs(w, device="cuda", seed=rank_seed(w, 0))
    n_seeds = w.shared_q
    q_in = x["q_seeds"] if n_seeds else x["q"]

    def plan_for(pol):
        p = gd.Plan(x["q_off"], x["kv_off"], w.H, w.d, mask=w.mask, window=w.window,
                    sched=pol, max_kv_blocks="auto")
        if n_seeds:
            p.set_shared_q(n_seeds)
        return p

    plan = plan_for(sched)
    o = torch.empty_like(x["q"])
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(warmup):
        gd.gdpa_fwd(plan, q_in, x["k"], x["v"], o=o, alpha=w.alpha, act=w.act)
    plan.check()
    evs = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        gd.gdpa_fwd(plan, q_in, x["k"], x["v"], o=o, alpha=w.alpha, act=w.act)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    plan.check()
    times = [a.elapsed_time(b) for a, b in evs]
    ms = float(np.median(times))
    Tq, Tkv = int(x["q_off"][-1]), int(x["kv_off"][-1])
    pairs = useful_pairs(x["q_off"], x["kv_off"], w.mask, w.window)
    flops = 4.0 * w.d * w.H * pairs
    row = w.H * w.d
    nbytes = (int(q_in.shape[0]) + Tq + 2 * Tkv) * row * 2
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    attainable = min(pk["bf16_tflops"], flops / nbytes * pk["hbm_gbs"] / 1e3)
    spread = {}
    for pol in POLICIES:
        pp = plan_for(pol)
        pp.set_timing(True)
        gd.gdpa_fwd(pp, q_in, x["k"], x["v"], o=o, alpha=w.alpha, act=w.act)
        pp.check()
        spread[pol] = busy_spread(pp.sm_times("fwd")[0])
        pp.destroy()
    n_tiles = plan.sizes()[0]
    plan.destroy()
    return {"ms": ms, "ms_min": float(min(times)), "tflops": tflops,
            "pct_of_bf16_peak": 100.0 * tflops / pk["bf16_tflops"], "gbs": gbs,
            "hbm_frac": gbs / pk["hbm_gbs"], "peak_kind": pk_kind,
            "attainable_tflops": attainable, "pct_of_attainable": 100.0 * tflops / attainable,
            "algorithmic_bytes": nbytes, "useful_pairs": pairs, "fwd_tiles": int(n_tiles),
            "B": w.B, "H": w.H, "act": w.act, "mask": w.mask, "window": w.window,
            "shared_q": n_seeds, "sched": sched,
            "timing": "median of %d launches, L2 flushed before each" % reps,
            "sm_spread": spread}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    @staticmethod
    def _epoch(stamp):
        # nvidia-smi's local-time stamp, "YYYY/MM/DD HH:MM:SS.mmm"
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, region=None):
        """Summary of the samples; with region = (t0, t1) (time.time() around
        the timed region) only the samples taken inside it, when there are
        any (else all, and "in_region" says so)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((self._epoch(f[0]), float(f[1]), float(f[2]),
                             {n for n, v in zip(names, f[5:9]) if v.lower() == "active"}))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if region and r[0] is not None and
                  region[0] - 0.03 <= r[0] <= region[1] + 0.03]
        use = inside or rows
        return {"sm_mhz": float(np.median([r[1] for r in use])),
                "sm_max_mhz": float(max(r[2] for r in use)),
                "reasons": sorted(set().union(*[r[3] for r in use])), "samples": len(use),
                "in_region": bool(inside)}


def cpu_baseline(w, x, budget_s=15.0):
    """Time the float64 oracle (forward + backward) on a prefix of the batch.

    A small calibration prefix is timed first; the rest of the sample is
    sized from it so that the whole measurement takes about ``budget_s``
    seconds.  ``x`` holds the batch (device or host tensors); only the rows
    of the sampled sequences are copied to the host.
    """
    from oracle import ref
    ref.build()
    q_off = np.asarray(x["q_off"], dtype=np.int64)
    kv_off = np.asarray(x["kv_off"], dtype=np.int64)
    backward = x.get("do") is not None
    nb = len(q_off) - 1
    per = np.diff(q_off) * np.diff(kv_off) * w.H * w.d * (12 if backward else 4)

    def host(t, a, b):
        return t[a:b].float().cpu().numpy()

    def run(s0, s1):
        qa, qb, ka, kb = q_off[s0], q_off[s1], kv_off[s0], kv_off[s1]
        sq = (q_off[s0:s1 + 1] - qa).astype(np.int32)
        skv = (kv_off[s0:s1 + 1] - ka).astype(np.int32)
        q, k, v = host(x["q"], qa, qb), host(x["k"], ka, kb), host(x["v"], ka, kb)
        t0 = time.perf_counter()
        ref.fwd(sq, skv, q, k, v, w.alpha, w.act, w.mask, w.window)
        if backward:
            ref.bwd(sq, skv, q, k, v, host(x["do"], qa, qb), w.alpha, w.act, w.mask, w.window)
        dt = time.perf_counter() - t0
        flops = (12 if backward else 4) * w.d * w.H * useful_pairs(sq, skv, w.mask, w.window)
        return flops, dt

    n0 = int(min(nb, max(1, np.searchsorted(np.cumsum(per), 2e8) + 1)))
    f0, t0 = run(0, n0)
    rate = per[:n0].sum() / max(t0, 1e-9)
    n1 = int(min(nb, n0 + np.searchsorted(np.cumsum(per[n0:]), rate * max(budget_s - t0, 0.0))))
    f1, t1 = run(n0, n1) if n1 > n0 else (0, 0.0)
    total_t = t0 + t1
    return {"value": (f0 + f1) / total_t / 1e12, "unit": UNIT, "cores": ref.threads(),
            "kind": "oracle",
            "sample": "first %d of %d sequences of the same batch, %s, float64 loops "
                      "(%.1f s)" % (n1 if n1 > n0 else n0, w.B,
                                    "forward + backward" if backward else "forward", total_t)}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from workloads import draw_lengths, make_inputs
    lq, lkv = draw_lengths(w)
    # a prefix of the batch with about 4e10 double flops is plenty for a
    # bounded sample; the tensors are drawn on the host for it alone
    per = lq * lkv * w.H * w.d * 12
    n = int(min(w.B, np.searchsorted(np.cumsum(per), 4e10) + 1))
    xh = make_inputs(w, device="cpu", lengths=(lq[:n], lkv[:n]))
    budget = 20.0 / max(1, args.steps + args.warmup)
    vals = []
    base = None
    for s in range(args.warmup + args.steps):
        r = cpu_baseline(w, xh, budget_s=budget)
        if s >= args.warmup:
            vals.append(r["value"])
            base = r
    value = float(np.median(vals))
    base["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, same shapes as the GPU arm)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "d": w.d, "act": w.act,
                       "mask": w.mask, "window": w.window},
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--samples", type=int, default=0,
                    help="use only the first N sequences of the workload (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--scaling", default="weak", choices=["weak", "strong"],
                    help="N > 1: each rank its own batch (weak) or one batch sharded over "
                         "the ranks by gdpa_shard_batch (strong)")
    ap.add_argument("--sched", default="zigzag_timed", choices=list(POLICIES),
                    help="dealing policy of the timed plans")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the forward-only lines of the other jagged workloads")
    ap.add_argument("--max-kv-blocks", default="auto",
                    help="key-split plans: at most this many 128-row key blocks per forward "
                         "tile (0 = whole key range per tile; 'auto' = the planner's choice, "
                         "no split for the softmax variant, which refuses split plans)")
    ap.add_argument("--materialise-q", action="store_true",
                    help="shared-query workloads: pass Q replicated per sample instead of "
                         "the seed rows (shared-query mode)")
    ap.add_argument("--qk-norm", type=float, default=0.0,
                    help="fused RMSNorm of the Q and K rows inside the kernels with this gain "
                         "(eps 1e-6); 0 = off")
    ap.add_argument("--act", default=None,
                    help="override the workload's activation; 'softmax' times the softmax "
                         "variant (Jagged Flash Attention) on the same batch")
    args = ap.parse_args()

    import dataclasses
    from workloads import get_config, make_inputs
    w = get_config(args.workload)
    if args.act:
        w = dataclasses.replace(w, act=args.act)
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import torch.distributed as dist
    import recommender_model_attention_gb300 as gd

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    gd.lib()
    pk, pk_kind = peaks()

    lengths = None
    if args.samples:
        from workloads import draw_lengths
        lq, lkv = draw_lengths(w)
        lengths = (lq[:args.samples], lkv[:args.samples])
    strong = args.scaling == "strong" and world > 1
    if strong:
        # one batch for the whole job; this rank keeps the samples dealt to it
        full = make_inputs(w, device="cuda", seed=rank_seed(w, 0), lengths=lengths)
        owner, _ = gd.shard_batch(full["q_off"], full["kv_off"], w.H, world, w.mask, w.window)
        lo, lk, qi, ki, _ = gd.shard_rows(full["q_off"], full["kv_off"], owner, rank)
        qi_t = torch.from_numpy(qi).cuda()
        ki_t = torch.from_numpy(ki).cuda()
        x = dict(full)
        x["q_off"], x["kv_off"] = lo, lk
        for n, idx in (("q", qi_t), ("k", ki_t), ("v", ki_t), ("do", qi_t)):
            if full.get(n) is not None:
                x[n] = full[n].index_select(0, idx).contiguous()
        del full
        torch.cuda.empty_cache()
    else:
        x = make_inputs(w, device="cuda", seed=rank_seed(w, rank), lengths=lengths)
    stream = torch.cuda.current_stream()
    mkb = args.max_kv_blocks if args.max_kv_blocks == "auto" else int(args.max_kv_blocks)
    if w.act == "softmax" and mkb == "auto":
        mkb = 0

    # shared-query workloads (pooling): Q is the seed rows, unless asked to
    # materialise it per sample
    n_seeds = w.shared_q if (w.shared_q and not args.materialise_q) else 0
    q_in = x["q_seeds"] if n_seeds else x["q"]

    def make_plan(**kw):
        kw.setdefault("sched", args.sched)
        p = gd.Plan(x["q_off"], x["kv_off"], w.H, w.d, mask=w.mask, window=w.window,
                    max_kv_blocks=mkb, **kw)
        if n_seeds:
            p.set_shared_q(n_seeds)
        if args.qk_norm > 0:
            p.set_qk_norm(args.qk_norm, 1e-6)
        return p

    plan = make_plan()
    # host planning + upload of one batch's plan (it synchronises on its upload)
    plan_times = []
    for _ in range(3):
        t0 = time.perf_counter()
        make_plan().destroy()
        plan_times.append((time.perf_counter() - t0) * 1e3)
    n_fwd_tiles, n_bwd_units, plan_sms = plan.sizes()
    whole = gd.Plan(x["q_off"], x["kv_off"], w.H, w.d, mask=w.mask, window=w.window,
                    num_sms=plan_sms, host_only=True)
    key_split = whole.sizes()[0] != n_fwd_tiles   # the plan cut some key ranges
    whole.destroy()
    f32 = torch.float32
    o = torch.empty_like(x["q"])
    dq = torch.empty(q_in.shape, dtype=f32, device="cuda")
    dk = torch.empty(x["k"].shape, dtype=f32, device="cuda")
    dv = torch.empty(x["v"].shape, dtype=f32, device="cuda")
    backward = x["do"] is not None
    # the softmax variant goes through its own calls (its backward needs O
    # and the row log-sum-exp, kept per output buffer)
    softmax = w.act == "softmax"
    lse_of = {}

    def fwd_call(p, q, k, v, o_):
        if softmax:
            lse = lse_of.setdefault(o_.data_ptr(), torch.empty((o_.shape[0], w.H), dtype=f32,
                                                               device=q.device))
            gd.gdpa_softmax_fwd(p, q, k, v, o=o_, lse=lse, alpha=w.alpha)
        else:
            gd.gdpa_fwd(p, q, k, v, o=o_, alpha=w.alpha, act=w.act)

    def bwd_call(p, q, k, v, o_, do_, dq_, dk_, dv_):
        if softmax:
            gd.gdpa_softmax_bwd(p, q, k, v, o_, do_, lse_of[o_.data_ptr()], dq_, dk_, dv_,
                                alpha=w.alpha)
        else:
            gd.gdpa_bwd(p, q, k, v, do_, dq_, dk_, dv_, alpha=w.alpha, act=w.act)

    def step():
        fwd_call(plan, q_in, x["k"], x["v"], o)
        if backward:
            bwd_call(plan, q_in, x["k"], x["v"], o, x["do"], dq, dk, dv)

    Tq, Tkv = int(x["q_off"][-1]), int(x["kv_off"][-1])
    pairs = useful_pairs(x["q_off"], x["kv_off"], w.mask, w.window)
    fwd_flops = 4.0 * w.d * w.H * pairs
    bwd_flops = 8.0 * w.d * w.H * pairs if backward else 0.0
    row = w.H * w.d
    Rq = int(q_in.shape[0])   # Q and dQ rows (the seeds in shared-query mode)
    fwd_bytes = (Rq + Tq + 2 * Tkv) * row * 2
    bwd_bytes = (Rq + Tq + 2 * Tkv) * row * 2 + (Rq + 2 * Tkv) * row * 4 if backward else 0
    if backward and softmax:
        bwd_bytes += Tq * row * 2   # O, read for the dO.O rows
    input_bytes = sum(t.numel() * t.element_size() for t in (q_in, x["k"], x["v"], x["do"])
                      if t is not None)

    for _ in range(args.warmup):
        step()
    plan.check()
    torch.cuda.synchronize()

    # timed region: K steps, per-phase events on the launching stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = Clocks(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = plan.launches
    t_region0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in range(args.steps):
        ev[s][0].record(stream)
        fwd_call(plan, q_in, x["k"], x["v"], o)
        ev[s][1].record(stream)
        if backward:
            bwd_call(plan, q_in, x["k"], x["v"], o, x["do"], dq, dk, dv)
        ev[s][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_region1 = time.time()
    clk = clocks.stop((t_region0, t_region1))
    launches = plan.launches - launches0
    plan.check()
    elapsed_ms, job_flops = reduce_across_ranks(start.elapsed_time(end),
                                                (fwd_flops + bwd_flops) * args.steps, "cuda")
    ms_step = elapsed_ms / args.steps
    fwd_ms = float(np.mean([a.elapsed_time(b) for a, b, _ in ev]))
    bwd_ms = float(np.mean([b.elapsed_time(c) for _, b, c in ev])) if backward else 0.0
    value = job_flops / (elapsed_ms * 1e-3) / 1e12

    # roofline of the dominant phase (kernel time measured live above)
    if bwd_ms > fwd_ms:
        dom, dom_ms, dom_bytes = "gdpa_bwd", bwd_ms, bwd_bytes
    else:
        dom, dom_ms, dom_bytes = "gdpa_fwd", fwd_ms, fwd_bytes
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = dram_traffic(dom, dom_bytes, w.name, key_split, softmax, args.qk_norm > 0)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                "algorithmic_bytes": dom_bytes, "peak_kind": pk_kind}

    # end to end through the public API: pinned host inputs in, the step's
    # metric out (the L2 norms of O, dQ, dK, dV, as a training loop logs
    # them; reduced by torch on the device), and separately with every output
    # copied back.  Steps are pipelined the way a training loader runs them:
    # step k's inputs go up on one stream while step k-1 computes, and its
    # results come down on another; two device buffer sets alternate.
    e2e = None
    if not args.no_e2e:
        hq = q_in.cpu().pin_memory()
        hk = x["k"].cpu().pin_memory()
        hv = x["v"].cpu().pin_memory()
        hdo = x["do"].cpu().pin_memory() if backward else None
        ho, hgrads = None, []   # full-readback buffers, pinned when that run comes
        sets = []
        for _ in range(2):
            ins = [torch.empty_like(t) for t in (q_in, x["k"], x["v"])]
            ins.append(torch.empty_like(x["do"]) if backward else None)
            outs = [torch.empty_like(o)] + ([torch.empty_like(t) for t in (dq, dk, dv)]
                                            if backward else [])
            sets.append((ins, outs))
        up, down, plan_stream = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "done", "out")}
        n_out = len(sets[0][1])
        metric_d = [torch.empty(n_out, dtype=f32, device="cuda") for _ in range(2)]
        metric_h = torch.empty(n_out, dtype=f32, pin_memory=True)

        def bf16_compute(p, ins, outs):
            q_d, k_d, v_d, do_d = ins
            fwd_call(p, q_d, k_d, v_d, outs[0])
            if backward:
                bwd_call(p, q_d, k_d, v_d, outs[0], do_d, *outs[1:])

        def e2e_run(n, replan=False, full=False, hosts=None, dsets=None, compute=bf16_compute):
            hosts = (hq, hk, hv, hdo) if hosts is None else hosts
            dsets = sets if dsets is None else dsets
            plans = []
            for k in range(n):
                sl = k % 2
                ins, outs = dsets[sl]
                if k >= 2:
                    up.wait_event(ev["done"][sl])      # step k-2 has read this set
                with torch.cuda.stream(up):
                    for dst, src in zip(ins, hosts):
                        if dst is not None:
                            dst.copy_(src, non_blocking=True)
                    ev["in"][sl].record(up)
                p = plan
                if replan:   # each step's batch planned afresh, as in training
                    p = make_plan(stream=plan_stream)
                    plans.append(p)
                stream.wait_event(ev["in"][sl])
                if k >= 2:
                    stream.wait_event(ev["out"][sl])   # step k-2's results are down
                compute(p, ins, outs)
                if not full:
                    for j, t in enumerate(outs):
                        metric_d[sl][j] = torch.linalg.vector_norm(t, dtype=f32)
                ev["done"][sl].record(stream)
                down.wait_event(ev["done"][sl])
                with torch.cuda.stream(down):
                    if full:
                        for h, d_ in zip([ho] + hgrads, outs):
                            h.copy_(d_, non_blocking=True)
                    else:
                        metric_h.copy_(metric_d[sl], non_blocking=True)
                    ev["out"][sl].record(down)
            for sl in range(2):
                stream.wait_event(ev["out"][sl])
            return plans

        # newly pinned host pages copy slowly for their first passes (the
        # first 8 GB of copies measured 175 GB/s, later ones 211): warm the
        # pipeline up over two full rounds before timing one
        n_e2e = max(3, min(args.steps, 6))
        e2e_run(2 * n_e2e)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_run(n_e2e)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_total, e2e_flops = reduce_across_ranks(a.elapsed_time(b),
                                                   (fwd_flops + bwd_flops) * n_e2e, "cuda")
        e2e_ms = e2e_total / n_e2e
        h2d = input_bytes
        d2h = n_out * 4
        d2h_full = o.numel() * o.element_size() + (sum(t.numel() * 4 for t in (dq, dk, dv))
                                                   if backward else 0)
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hgrads = [torch.empty(t.shape, dtype=f32, pin_memory=True) for t in (dq, dk, dv)]
        e2e_run(2 * n_e2e, full=True)
        torch.cuda.synchronize()
        a.record(stream)
        e2e_run(n_e2e, full=True)
        b.record(stream)
        torch.cuda.synchronize()
        full_total, _ = reduce_across_ranks(a.elapsed_time(b), 0.0, "cuda")
        # the same with each step's batch planned afresh (host planning and plan
        # upload inside the timed region)
        a.record(stream)
        plans = e2e_run(n_e2e, replan=True)
        b.record(stream)
        torch.cuda.synchronize()
        for p in plans:
            p.destroy()
        replan_total, _ = reduce_across_ranks(a.elapsed_time(b), 0.0, "cuda")
        e2e = {"value": e2e_flops / (e2e_total * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms, "readback": "L2 norms of O, dQ, dK, dV (float32)",
               "ms_per_step_with_planning": replan_total / n_e2e,
               "full_readback": {"value": e2e_flops / (full_total * 1e-3) / 1e12,
                                 "d2h_bytes_per_step": int(d2h_full),
                                 "ms_per_step": full_total / n_e2e},
               "pipelining": "inputs up, compute, results down on three streams, "
                             "two buffer sets",
               "warmup_steps": 2 * n_e2e, "timed_steps": n_e2e}

    # the same step with Q and K arriving in MXFP8 (E4M3 elements, one E8M0
    # scale per 32 values along d): gdpa_fwd_mx / gdpa_bwd_mx expand them to
    # bf16 on the device, then run the bf16 kernels; on device and end to end
    mxfp8 = None
    if rank == 0 and world == 1 and not args.no_workloads and not softmax and not args.samples:
        qm, km = gd.mx_quantise(q_in), gd.mx_quantise(x["k"])

        def mx_step(p, q_m, k_m, v_, do_, o_, dq_, dk_, dv_):
            gd.gdpa_fwd_mx(p, q_m, k_m, v_, o=o_, alpha=w.alpha, act=w.act)
            if backward:   # reuses the forward's expansion of Q and K
                gd.gdpa_bwd_mx(p, None, None, v_, do_, dq_, dk_, dv_, alpha=w.alpha, act=w.act)

        for _ in range(args.warmup):
            mx_step(plan, qm, km, x["v"], x["do"], o, dq, dk, dv)
        torch.cuda.synchronize()
        mev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for s in range(args.steps):
            mev[s][0].record(stream)
            gd.gdpa_fwd_mx(plan, qm, km, x["v"], o=o, alpha=w.alpha, act=w.act)
            mev[s][1].record(stream)
            if backward:
                gd.gdpa_bwd_mx(plan, None, None, x["v"], x["do"], dq, dk, dv, alpha=w.alpha,
                               act=w.act)
            mev[s][2].record(stream)
        torch.cuda.synchronize()
        plan.check()
        m_fwd = float(np.mean([a.elapsed_time(b) for a, b, _ in mev]))
        m_bwd = float(np.mean([b.elapsed_time(c) for _, b, c in mev])) if backward else 0.0
        m_ms = float(np.mean([a.elapsed_time(c) for a, _, c in mev]))
        mx_in = (qm.elements, qm.scales, km.elements, km.scales, x["v"], x["do"])
        mx_bytes = sum(t.numel() * t.element_size() for t in mx_in if t is not None)
        mxfp8 = {"ms_per_step": m_ms, "fwd_ms": m_fwd, "bwd_ms": m_bwd,
                 "tflops": (fwd_flops + bwd_flops) / (m_ms * 1e-3) / 1e12,
                 "input_bytes": int(mx_bytes), "input_bytes_bf16": int(input_bytes),
                 "what": "Q and K in MXFP8, expanded to bf16 on the device by the forward "
                         "(two launches) and reused by the backward; V, dO, O bf16, "
                         "gradients float32"}
        if e2e is not None:
            h_mx = [t.cpu().pin_memory() if t is not None else None for t in mx_in]
            mx_sets = [([torch.empty_like(t) if t is not None else None for t in mx_in], outs)
                       for _, outs in sets]

            def mx_compute(p, ins, outs):
                mx_step(p, gd.MX(ins[0], ins[1]), gd.MX(ins[2], ins[3]), ins[4], ins[5], *outs)

            e2e_run(2 * n_e2e, hosts=h_mx, dsets=mx_sets, compute=mx_compute)
            torch.cuda.synchronize()
            a.record(stream)
            e2e_run(n_e2e, hosts=h_mx, dsets=mx_sets, compute=mx_compute)
            b.record(stream)
            torch.cuda.synchronize()
            mx_e2e_ms = a.elapsed_time(b) / n_e2e
            mxfp8["e2e"] = {"value": (fwd_flops + bwd_flops) / (mx_e2e_ms * 1e-3) / 1e12,
                            "unit": UNIT, "ms_per_step": mx_e2e_ms,
                            "h2d_bytes_per_step": int(mx_bytes), "d2h_bytes_per_step": int(d2h)}
            del h_mx, mx_sets
        del qm, km
        torch.cuda.empty_cache()

    # SM busy-time spread of each policy, forward and backward (separate,
    # untimed launches)
    spread, spread_bwd = {}, {}
    try:
        for pol in POLICIES:
            pp = make_plan(sched=pol)
            pp.set_timing(True)
            fwd_call(pp, q_in, x["k"], x["v"], o)
            if backward:
                bwd_call(pp, q_in, x["k"], x["v"], o, x["do"], dq, dk, dv)
            pp.check()
            spread[pol] = busy_spread(pp.sm_times("fwd")[0])
            if backward:
                spread_bwd[pol] = busy_spread(pp.sm_times("bwd")[0])
            pp.destroy()
    except Exception as e:  # timing is a report, not the measurement
        spread["error"] = str(e)

    # the other jagged workloads, forward only, in the same run
    others = None
    if rank == 0 and world == 1 and not args.no_workloads and args.workload == DEFAULT_WORKLOAD \
            and not args.samples and not args.act:
        others = {}
        for name in OTHER_WORKLOADS:
            try:
                others[name] = forward_workload(name, gd, pk, pk_kind, sched=args.sched)
            except Exception as e:  # a report beside the headline
                others[name] = {"error": str(e)}
            torch.cuda.synchronize()
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, x)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "strong" if strong else "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded lengths and RMSNorm'd N(0,1) inputs, random dO)",
            "config": {"workload": w.name, "B": len(x["q_off"]) - 1, "H": w.H, "d": w.d,
                       "act": w.act, "max_kv_blocks": mkb, "sched": args.sched,
                       "qk_norm": args.qk_norm,
                       "key_split": key_split, "shared_q": n_seeds,
                       "Tq": Tq, "Tkv": Tkv, "useful_pairs": pairs,
                       "l2": "inputs larger than L2 (%.1f GB resident)" % (input_bytes / 1e9),
                       "parallelism": ("one batch's samples dealt to ranks by gdpa_shard_batch, "
                                       "no exchange" if strong else
                                       "each rank its own batch, no exchange") if world > 1
                       else "single GPU"},
            "pct_of_bf16_peak": 100.0 * value / world / pk["bf16_tflops"],
            "fwd": {"ms": fwd_ms, "tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12,
                    "gbs": fwd_bytes / (fwd_ms * 1e-3) / 1e9},
            "bwd": ({"ms": bwd_ms, "tflops": bwd_flops / (bwd_ms * 1e-3) / 1e12,
                     "gbs": bwd_bytes / (bwd_ms * 1e-3) / 1e9} if backward else None),
            "roofline": roofline,
            "gpu_launches": int(launches),
            "clocks": clk,
            "e2e": e2e,
            "mxfp8": mxfp8,
            "sm_spread_fwd": spread,
            "sm_spread_bwd": spread_bwd if backward else None,
            "workloads": others,
            "plan": {"host_ms_median": float(np.median(plan_times)), "fwd_tiles": int(n_fwd_tiles),
                     "bwd_units": int(n_bwd_units)},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    plan.destroy()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
