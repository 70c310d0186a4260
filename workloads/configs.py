"""The five seeded GDPA workloads and a generator for small random cases.

Lengths are drawn with NumPy's PCG64 (seed = the workload's index), so the
offset arrays are identical on every machine.  Tensors are drawn with a seeded
``torch.Generator`` on the device that will hold them; the oracle receives a
host copy of exactly the same tensors.

Readings of the workload descriptions that the source pages leave open:

* "lognormal (median m)" uses sigma = 1: L = clip(rint(exp(ln m + z)), lo, hi).
* "Zipf (s) clipped to [1, N]" is NumPy's ``Generator.zipf(s)`` clipped to N.
* "RMSNorm'd N(0,1)" normalises every (token, head) row of length d to unit
  mean square, x / sqrt(mean(x^2) + 1e-6), then multiplies by a gain (1 unless
  stated).  The PMA workload uses the gain sqrt(2) * d**-0.25 on Q and K, so
  Cauchy-Schwarz bounds |alpha * q.k| by 2 (before rounding to bf16).
* The PMA workload's 32 seed queries are shared by every sample; they are
  materialised as a [32 * B, H, d] tensor with q_off[b] = 32 * b.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

ACTS = ("gelu_erf", "gelu_tanh", "silu", "gelu_taylor6", "identity")
MASKS = ("none", "causal_window")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int            # also the length-draw seed
    B: int
    H: int
    d: int
    dtype: str            # "f32" or "bf16"
    q_len: tuple          # ("uniform", lo, hi) | ("lognormal", median, lo, hi) | ("zipf", s, lo, hi) | ("const", n)
    kv_len: Optional[tuple]  # None = same lengths as Q (self-attention)
    mask: str
    window: int
    act: str
    backward: bool
    qk_gain: float = 1.0  # RMSNorm gain on Q and K (1.0 = plain RMSNorm)
    rmsnorm: bool = True  # False: N(0,1)/sqrt(d) without normalisation
    shared_q: int = 0     # >0: that many seed queries shared by all samples

    @property
    def alpha(self) -> float:
        return 1.0 / math.sqrt(self.d)


CONFIGS = (
    Workload("tiny_selfattn_f32", 0, B=4, H=2, d=32, dtype="f32",
             q_len=("uniform", 1, 64), kv_len=None, mask="none", window=0,
             act="gelu_erf", backward=True, rmsnorm=False),
    Workload("jagged_selfattn_window256", 1, B=256, H=4, d=128, dtype="bf16",
             q_len=("lognormal", 200, 1, 2048), kv_len=None,
             mask="causal_window", window=256, act="silu", backward=False),
    Workload("user_ad_cross", 2, B=512, H=8, d=128, dtype="bf16",
             q_len=("lognormal", 500, 1, 4096), kv_len=("uniform", 8, 64),
             mask="none", window=0, act="gelu_tanh", backward=False),
    Workload("pma_pooling", 3, B=1024, H=4, d=128, dtype="bf16",
             q_len=("const", 32), kv_len=("zipf", 1.1, 1, 8192),
             mask="none", window=0, act="gelu_taylor6", backward=False,
             qk_gain=math.sqrt(2.0) * 128 ** -0.25, shared_q=32),
    Workload("training_cross_fwd_bwd", 4, B=2048, H=8, d=128, dtype="bf16",
             q_len=("zipf", 1.2, 1, 4096), kv_len=("uniform", 8, 128),
             mask="none", window=0, act="gelu_erf", backward=True),
)


def get_config(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return CONFIGS[name_or_index]
    for c in CONFIGS:
        if c.name == name_or_index:
            return c
    raise KeyError(name_or_index)


def _draw(rng: np.random.Generator, spec: tuple, B: int) -> np.ndarray:
    kind = spec[0]
    if kind == "uniform":
        _, lo, hi = spec
        return rng.integers(lo, hi + 1, size=B, dtype=np.int64)
    if kind == "lognormal":
        _, median, lo, hi = spec
        z = rng.standard_normal(B)
        return np.clip(np.rint(np.exp(math.log(median) + z)), lo, hi).astype(np.int64)
    if kind == "zipf":
        _, s, lo, hi = spec
        return np.clip(rng.zipf(s, size=B), lo, hi).astype(np.int64)
    if kind == "const":
        return np.full(B, spec[1], dtype=np.int64)
    raise ValueError(spec)


def draw_lengths(w: Workload):
    """Per-sample (Lq, Lkv) as int64 arrays, seeded by the workload index."""
    rng = np.random.Generator(np.random.PCG64(w.index))
    lq = _draw(rng, w.q_len, w.B)
    lkv = lq.copy() if w.kv_len is None else _draw(rng, w.kv_len, w.B)
    return lq, lkv


def offsets_from_lengths(lengths) -> np.ndarray:
    """Exclusive prefix sum as int32, checked to fit."""
    lengths = np.asarray(lengths, dtype=np.int64)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    if off[-1] >= 2 ** 31:
        raise OverflowError("total length does not fit int32 offsets")
    return off.astype(np.int32)


def _rmsnorm_rows(x, gain: float):
    import torch
    ms = x.pow(2).mean(dim=-1, keepdim=True)
    return x * torch.rsqrt(ms + 1e-6) * gain


def _torch_dtype(name: str):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None,
                lengths=None, chunk_rows: int = 1 << 20):
    """Draw Q, K, V (and dO when the workload has a backward pass).

    Returns a dict with int32 numpy offsets ``q_off``/``kv_off`` and torch
    tensors ``q``, ``k``, ``v`` ([T, H, d], contiguous) and ``do`` (or None),
    all in the workload's dtype on ``device``; for shared-query workloads also
    ``q_seeds`` ([shared_q, H, d]; ``q`` is then the seeds repeated per
    sample), else ``q_seeds`` is None.
    """
    import torch

    lq, lkv = draw_lengths(w) if lengths is None else lengths
    q_off = offsets_from_lengths(lq)
    kv_off = offsets_from_lengths(lkv)
    tq, tkv = int(q_off[-1]), int(kv_off[-1])
    dt = _torch_dtype(w.dtype)
    g = torch.Generator(device=device)
    g.manual_seed(1000 + w.index if seed is None else seed)

    def rows(n, gain):
        out = torch.empty((n, w.H, w.d), dtype=dt, device=device)
        for s in range(0, n, chunk_rows):
            e = min(n, s + chunk_rows)
            x = torch.randn((e - s, w.H, w.d), generator=g, device=device,
                            dtype=torch.float32)
            if w.rmsnorm:
                x = _rmsnorm_rows(x, gain)
            else:
                x = x / math.sqrt(w.d)
            out[s:e] = x.to(dt)
        return out

    seeds = None
    if w.shared_q:
        seeds = rows(w.shared_q, w.qk_gain)
        nb = len(lq)   # w.B, or fewer when a prefix of the batch is drawn
        assert tq == w.shared_q * nb
        q = seeds.repeat(nb, 1, 1).contiguous()
    else:
        q = rows(tq, w.qk_gain)
    k = rows(tkv, w.qk_gain)
    v = rows(tkv, 1.0)
    do = None
    if w.backward:
        do = torch.empty((tq, w.H, w.d), dtype=dt, device=device)
        for s in range(0, tq, chunk_rows):
            e = min(tq, s + chunk_rows)
            do[s:e] = torch.randn((e - s, w.H, w.d), generator=g, device=device,
                                  dtype=torch.float32).to(dt)
    return dict(q_off=q_off, kv_off=kv_off, q=q, k=k, v=v, do=do, q_seeds=seeds)


def small_case(seed: int, B: int, H: int, d: int, q_range=(1, 64), kv_range=None,
               dtype: str = "f32", rmsnorm: bool = False, zero_lengths: bool = False):
    """A random jagged case with explicit sizes, drawn with NumPy PCG64.

    ``kv_range=None`` makes it self-attention (Lkv = Lq).  With
    ``zero_lengths`` a quarter of the samples get Lq = 0 or Lkv = 0.
    Returns the same dict as :func:`make_inputs`, with CPU tensors.
    """
    import torch

    rng = np.random.Generator(np.random.PCG64(seed))
    lq = rng.integers(q_range[0], q_range[1] + 1, size=B, dtype=np.int64)
    if kv_range is None:
        lkv = lq.copy()
    else:
        lkv = rng.integers(kv_range[0], kv_range[1] + 1, size=B, dtype=np.int64)
    if zero_lengths and B > 0:
        z = rng.random(B)
        lq[z < 0.125] = 0
        lkv[(z >= 0.125) & (z < 0.25)] = 0
    q_off = offsets_from_lengths(lq)
    kv_off = offsets_from_lengths(lkv)
    tq, tkv = int(q_off[-1]), int(kv_off[-1])
    dt = _torch_dtype(dtype)

    def rows(n):
        x = torch.from_numpy(rng.standard_normal((n, H, d)).astype(np.float32))
        if rmsnorm:
            x = _rmsnorm_rows(x, 1.0)
        else:
            x = x / math.sqrt(d)
        return x.to(dt).contiguous()

    q, k, v = rows(tq), rows(tkv), rows(tkv)
    do = torch.from_numpy(rng.standard_normal((tq, H, d)).astype(np.float32)).to(dt).contiguous()
    return dict(q_off=q_off, kv_off=kv_off, q=q, k=k, v=v, do=do)
