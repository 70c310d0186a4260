"""Thin ctypes binding of the GDPA C ABI (``include/gdpa.h``).

Argument marshalling only: every step of planning and of the forward and
backward passes runs in the C++/CUDA library.  There is no fallback: if the
library has not been built, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import NamedTuple

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdpa_gb300.so")

ACT = {"gelu_erf": 0, "gelu_tanh": 1, "silu": 2, "gelu_taylor6": 3, "identity": 4,
       "softmax": 5}
MASK = {"none": 0, "causal_window": 1}
SCHED = {"zigzag": 0, "round_robin": 1, "zigzag_timed": 2}
KERNEL = {"auto": 0, "tcgen05": 1, "simt": 2}
KV_SPLIT_AUTO = -1   # max_kv_blocks_per_tile: the planner chooses
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
          4: "allocation failed", 5: "kernel barrier wait timed out",
          6: "kernel reported an internal error",
          7: "batch exceeds the static scratch of gdpa_fwd_noalloc"}
BLOCK_M = 128
BLOCK_N = 128

_lib = None


class GdpaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s (status %d)" % (what, STATUS.get(status, "?"), status))
        self.status = status


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("GDPA CUDA library missing (%s); build it with "
                               "recommender_model_attention_gb300.build()" % LIB_PATH)
        try:
            import torch  # noqa: F401  (loads the CUDA runtime the library links)
        except ImportError:
            pass
        L = ctypes.CDLL(LIB_PATH)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        vp = ctypes.c_void_p
        st = ctypes.c_int
        sig = {
            "gdpa_plan_create": [i32p, i32p, st, st, st, st, st, st, st, st, vp, ctypes.POINTER(vp)],
            "gdpa_plan_create_host": [i32p, i32p, st, st, st, st, st, st, st, st, ctypes.POINTER(vp)],
            "gdpa_plan_sizes": [vp, i64p, i64p, ctypes.POINTER(ctypes.c_int)],
            "gdpa_plan_export": [vp, i32p, ctypes.c_int64, i64p, i32p],
            "gdpa_plan_export_bwd": [vp, i32p, ctypes.c_int64, i64p, i32p, ctypes.POINTER(ctypes.c_int)],
            "gdpa_plan_set_kernel": [vp, st],
            "gdpa_plan_set_timing": [vp, st],
            "gdpa_plan_set_shared_q": [vp, st],
            "gdpa_plan_set_wait_test": [vp, st, st],
            "gdpa_plan_set_qk_norm": [vp, ctypes.c_float, ctypes.c_float],
            "gdpa_fwd": [vp, st, vp, vp, vp, vp, ctypes.c_float, st, vp],
            "gdpa_bwd": [vp, st, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, st, vp],
            "gdpa_check": [vp, vp],
            "gdpa_error_detail": [vp, i32p],
            "gdpa_sm_times": [vp, st, ctypes.POINTER(ctypes.c_uint64), i32p],
            "gdpa_fwd_noalloc": [i32p, i32p, st, st, st, st, st, vp, vp, vp, vp, ctypes.c_float,
                                 st, vp],
            "gdpa_act_eval": [st, st, vp, vp, vp, ctypes.c_int64, vp],
            "gdpa_shard_batch": [i32p, i32p, st, st, st, st, st, i32p, i64p],
            "gdpa_softmax_fwd": [vp, st, vp, vp, vp, vp, vp, ctypes.c_float, vp],
            "gdpa_softmax_bwd": [vp, st, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp],
            "gdpa_mx_quantise": [vp, ctypes.c_int64, vp, vp, vp],
            "gdpa_mx_dequantise": [vp, vp, ctypes.c_int64, vp, vp],
            "gdpa_fwd_mx": [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, st, vp],
            "gdpa_bwd_mx": [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, st, vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.gdpa_plan_launches.argtypes = [vp]
        L.gdpa_plan_launches.restype = ctypes.c_int64
        L.gdpa_plan_destroy.argtypes = [vp]
        L.gdpa_plan_destroy.restype = None
        L.gdpa_status_str.argtypes = [ctypes.c_int]
        L.gdpa_status_str.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ok(status: int, what: str):
    if status != 0:
        raise GdpaError(status, what)


def _i32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """A GDPA tile plan (forward tiles and backward units dealt to SMs).

    max_kv_blocks: 0 = one forward tile per query tile; k > 0 = key ranges
    cut into chunks of at most k 128-row key blocks; "auto" = the planner's
    choice (2-block chunks when some query tile reaches 8 key blocks).
    """

    def __init__(self, q_off, kv_off, H: int, d: int, mask: str = "none", window: int = 0,
                 sched: str = "zigzag", num_sms: int = 0, max_kv_blocks: int = 0,
                 stream=None, host_only: bool = False):
        L = lib()
        qo, qp = _i32(q_off)
        ko, kp = _i32(kv_off)
        if len(qo) != len(ko) or len(qo) < 1:
            raise ValueError("offset arrays must both have B + 1 entries")
        self.B, self.H, self.d = len(qo) - 1, int(H), int(d)
        self.mask, self.window = mask, int(window)
        self.Tq, self.Tkv = int(qo[-1]), int(ko[-1])
        self.q_off, self.kv_off = qo.copy(), ko.copy()
        self.shared_q = 0
        self.q_rows = self.Tq   # rows of q and dq (the seeds in shared-query mode)
        mkb = KV_SPLIT_AUTO if max_kv_blocks == "auto" else int(max_kv_blocks)
        h = ctypes.c_void_p()
        if host_only:
            _ok(L.gdpa_plan_create_host(qp, kp, self.B, self.H, self.d, MASK[mask], int(window),
                                        SCHED[sched], int(num_sms), mkb,
                                        ctypes.byref(h)), "gdpa_plan_create_host")
        else:
            _ok(L.gdpa_plan_create(qp, kp, self.B, self.H, self.d, MASK[mask], int(window),
                                   SCHED[sched], int(num_sms), mkb,
                                   _stream_ptr(stream), ctypes.byref(h)), "gdpa_plan_create")
        self._h = h

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan destroyed")
        return self._h

    def sizes(self):
        nf, nb, s = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int()
        _ok(lib().gdpa_plan_sizes(self.handle, ctypes.byref(nf), ctypes.byref(nb), ctypes.byref(s)),
            "gdpa_plan_sizes")
        return nf.value, nb.value, s.value

    @property
    def num_sms(self) -> int:
        return self.sizes()[2]

    def export(self):
        """(tiles int32 [n, 6] = b, h, m, kb0, kb1, sm;  seg int32 [S + 1])."""
        nf, _, S = self.sizes()
        tiles = np.zeros((max(nf, 1), 6), dtype=np.int32)
        seg = np.zeros(S + 1, dtype=np.int32)
        n = ctypes.c_int64()
        _ok(lib().gdpa_plan_export(self.handle, tiles.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                   nf, ctypes.byref(n),
                                   seg.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))), "gdpa_plan_export")
        return tiles[:n.value], seg

    def export_bwd(self):
        """(units int32 [n, 7] = b, h, j, m0, m1, flags, sm;  seg [S + 1];  zero_dq)."""
        _, nb, S = self.sizes()
        units = np.zeros((max(nb, 1), 7), dtype=np.int32)
        seg = np.zeros(S + 1, dtype=np.int32)
        n, z = ctypes.c_int64(), ctypes.c_int()
        _ok(lib().gdpa_plan_export_bwd(self.handle, units.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       nb, ctypes.byref(n),
                                       seg.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       ctypes.byref(z)), "gdpa_plan_export_bwd")
        return units[:n.value], seg, bool(z.value)

    def set_kernel(self, kernel: str):
        _ok(lib().gdpa_plan_set_kernel(self.handle, KERNEL[kernel]), "gdpa_plan_set_kernel")

    def set_shared_q(self, n_seeds: int):
        """Shared-query mode: q (and the backward's dq) hold n_seeds seed rows
        shared by every sample, sample b's queries being seeds 0 .. Lq_b - 1;
        0 restores per-token queries."""
        _ok(lib().gdpa_plan_set_shared_q(self.handle, int(n_seeds)), "gdpa_plan_set_shared_q")
        self.shared_q = int(n_seeds)
        self.q_rows = self.shared_q if self.shared_q > 0 else self.Tq

    def set_timing(self, enable: bool):
        _ok(lib().gdpa_plan_set_timing(self.handle, 1 if enable else 0), "gdpa_plan_set_timing")

    def set_qk_norm(self, gain: float = 1.0, eps: float = 1e-6):
        """Fused RMSNorm of the Q and K rows inside the kernels (gain > 0);
        gain = 0 turns it off."""
        _ok(lib().gdpa_plan_set_qk_norm(self.handle, ctypes.c_float(gain), ctypes.c_float(eps)),
            "gdpa_plan_set_qk_norm")

    def set_wait_test(self, limit_us: int = 0, stall: bool = False):
        """Failure-path test hook: bounded-wait limit (microseconds, 0 = the
        default) and whether CTA 0's loader skips its first query-tile load on
        the next tensor-core launches, so that a wait expires."""
        _ok(lib().gdpa_plan_set_wait_test(self.handle, int(limit_us), 1 if stall else 0),
            "gdpa_plan_set_wait_test")

    def sm_times(self, which: str = "fwd"):
        """(start_end uint64 [S, 2] in ns, smid int32 [S]) of the last timed launch."""
        S = self.num_sms
        se = np.zeros((S, 2), dtype=np.uint64)
        sm = np.zeros(S, dtype=np.int32)
        _ok(lib().gdpa_sm_times(self.handle, 0 if which == "fwd" else 1,
                                se.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                sm.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))), "gdpa_sm_times")
        return se, sm

    def check(self, stream=None):
        status = lib().gdpa_check(self.handle, _stream_ptr(stream))
        if status != 0:
            code, site, cta, word = self.error_detail()
            raise GdpaError(status, "gdpa_check (device code %d, wait site %d, CTA %d, %d)"
                            % (code, site, cta, word))

    def error_detail(self):
        """(device code, wait site, CTA, word) of the last failure that
        check() reported for this plan; zeros if none."""
        d = (ctypes.c_int32 * 4)()
        _ok(lib().gdpa_error_detail(self.handle, d), "gdpa_error_detail")
        return tuple(int(v) for v in d)

    @property
    def launches(self) -> int:
        return int(lib().gdpa_plan_launches(self.handle))

    def destroy(self):
        if getattr(self, "_h", None) is not None:
            lib().gdpa_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _dtype_id(t):
    import torch
    if t.dtype == torch.bfloat16:
        return 0
    if t.dtype == torch.float32:
        return 1
    raise TypeError("GDPA takes bfloat16 or float32 tensors, got %s" % t.dtype)


def _check(t, rows, plan, name, dtype=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if tuple(t.shape) != (rows, plan.H, plan.d):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), (rows, plan.H, plan.d)))
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s" % (name, dtype))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)


def gdpa_fwd(plan: Plan, q, k, v, o=None, alpha=None, act: str = "gelu_erf", stream=None):
    """O = act(alpha Q K^T) V per sample and head; returns O ([Tq, H, d], dtype of q)."""
    import torch
    _check(q, plan.q_rows, plan, "q")
    _check(k, plan.Tkv, plan, "k", q.dtype)
    _check(v, plan.Tkv, plan, "v", q.dtype)
    if o is None:
        o = torch.empty((plan.Tq, plan.H, plan.d), dtype=q.dtype, device=q.device)
    _check(o, plan.Tq, plan, "o", q.dtype)
    alpha = plan.d ** -0.5 if alpha is None else float(alpha)
    _ok(lib().gdpa_fwd(plan.handle, _dtype_id(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                       ctypes.c_float(alpha), ACT[act], _stream_ptr(stream)), "gdpa_fwd")
    return o


def gdpa_bwd(plan: Plan, q, k, v, do, dq=None, dk=None, dv=None, alpha=None,
             act: str = "gelu_erf", stream=None):
    """(dQ, dK, dV) as float32 tensors given the upstream gradient dO (dQ per
    seed row, summed over the samples, in shared-query mode)."""
    import torch
    _check(q, plan.q_rows, plan, "q")
    _check(k, plan.Tkv, plan, "k", q.dtype)
    _check(v, plan.Tkv, plan, "v", q.dtype)
    _check(do, plan.Tq, plan, "do", q.dtype)
    f32 = torch.float32
    dq = torch.empty(q.shape, dtype=f32, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=f32, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=f32, device=v.device) if dv is None else dv
    _check(dq, plan.q_rows, plan, "dq", f32)
    _check(dk, plan.Tkv, plan, "dk", f32)
    _check(dv, plan.Tkv, plan, "dv", f32)
    alpha = plan.d ** -0.5 if alpha is None else float(alpha)
    _ok(lib().gdpa_bwd(plan.handle, _dtype_id(q), _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq),
                       _ptr(dk), _ptr(dv), ctypes.c_float(alpha), ACT[act], _stream_ptr(stream)),
        "gdpa_bwd")
    return dq, dk, dv


class MX(NamedTuple):
    """An MXFP8 tensor: E4M3 codes (uint8, the values' shape) and one E8M0
    scale byte (exponent + 127) per 32 values along the last axis."""
    elements: "object"
    scales: "object"


def mx_quantise(x, stream=None) -> MX:
    """bf16 CUDA tensor (last axis a multiple of 32) -> its MXFP8 encoding."""
    import torch
    if not x.is_cuda or not x.is_contiguous() or x.dtype != torch.bfloat16:
        raise ValueError("mx_quantise takes a contiguous bfloat16 CUDA tensor")
    if x.shape[-1] % 32:
        raise ValueError("the last axis must be a multiple of 32")
    el = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    sc = torch.empty(x.shape[:-1] + (x.shape[-1] // 32,), dtype=torch.uint8, device=x.device)
    _ok(lib().gdpa_mx_quantise(_ptr(x), x.numel(), _ptr(el), _ptr(sc), _stream_ptr(stream)),
        "gdpa_mx_quantise")
    return MX(el, sc)


def mx_dequantise(m: MX, stream=None):
    """The bf16 values an MXFP8 tensor stands for."""
    import torch
    el, sc = m
    _mx_check(el, sc, 0, None, "x")
    x = torch.empty(el.shape, dtype=torch.bfloat16, device=el.device)
    _ok(lib().gdpa_mx_dequantise(_ptr(el), _ptr(sc), el.numel(), _ptr(x), _stream_ptr(stream)),
        "gdpa_mx_dequantise")
    return x


def _mx_check(el, sc, rows, plan, name):
    import torch
    for t, what in ((el, "elements"), (sc, "scales")):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.uint8:
            raise ValueError("%s %s must be a contiguous uint8 CUDA tensor" % (name, what))
    if tuple(sc.shape) != tuple(el.shape[:-1]) + (el.shape[-1] // 32,) or el.shape[-1] % 32:
        raise ValueError("%s: scales must have one byte per 32 elements" % name)
    if plan is not None and tuple(el.shape) != (rows, plan.H, plan.d):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(el.shape),
                                                           (rows, plan.H, plan.d)))


def gdpa_fwd_mx(plan: Plan, q: MX, k: MX, v, o=None, alpha=None, act: str = "gelu_erf",
                stream=None):
    """gdpa_fwd with Q and K in MXFP8 (``mx_quantise``); V and O bf16."""
    import torch
    _mx_check(q.elements, q.scales, plan.q_rows, plan, "q")
    _mx_check(k.elements, k.scales, plan.Tkv, plan, "k")
    _check(v, plan.Tkv, plan, "v", torch.bfloat16)
    if o is None:
        o = torch.empty((plan.Tq, plan.H, plan.d), dtype=torch.bfloat16, device=v.device)
    _check(o, plan.Tq, plan, "o", torch.bfloat16)
    alpha = plan.d ** -0.5 if alpha is None else float(alpha)
    _ok(lib().gdpa_fwd_mx(plan.handle, _ptr(q.elements), _ptr(q.scales), _ptr(k.elements),
                          _ptr(k.scales), _ptr(v), _ptr(o), ctypes.c_float(alpha), ACT[act],
                          _stream_ptr(stream)), "gdpa_fwd_mx")
    return o


def gdpa_bwd_mx(plan: Plan, q, k, v, do, dq=None, dk=None, dv=None, alpha=None,
                act: str = "gelu_erf", stream=None):
    """gdpa_bwd with Q and K in MXFP8: float32 (dQ, dK, dV) with respect to the
    values the MXFP8 tensors stand for.  q = k = None reuses the bf16
    expansion of the plan's previous MXFP8 call (the forward's)."""
    import torch
    reuse = q is None and k is None
    if not reuse:
        _mx_check(q.elements, q.scales, plan.q_rows, plan, "q")
        _mx_check(k.elements, k.scales, plan.Tkv, plan, "k")
        ptrs = [_ptr(q.elements), _ptr(q.scales), _ptr(k.elements), _ptr(k.scales)]
    else:
        ptrs = [ctypes.c_void_p(0)] * 4
    _check(v, plan.Tkv, plan, "v", torch.bfloat16)
    _check(do, plan.Tq, plan, "do", torch.bfloat16)
    f32 = torch.float32
    dq = torch.empty((plan.q_rows, plan.H, plan.d), dtype=f32, device=v.device) if dq is None else dq
    dk = torch.empty(v.shape, dtype=f32, device=v.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=f32, device=v.device) if dv is None else dv
    _check(dq, plan.q_rows, plan, "dq", f32)
    _check(dk, plan.Tkv, plan, "dk", f32)
    _check(dv, plan.Tkv, plan, "dv", f32)
    alpha = plan.d ** -0.5 if alpha is None else float(alpha)
    _ok(lib().gdpa_bwd_mx(plan.handle, *ptrs, _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                          ctypes.c_float(alpha), ACT[act], _stream_ptr(stream)), "gdpa_bwd_mx")
    return dq, dk, dv


def shard_batch(q_off, kv_off, H: int, num_ranks: int, mask: str = "none", window: int = 0):
    """(rank of each sample int32 [B], work of each rank int64 [R]): the
    samples of one batch dealt to ranks by work in zigzag order
    (gdpa_shard_batch)."""
    qo, qp = _i32(q_off)
    ko, kp = _i32(kv_off)
    if len(qo) != len(ko) or len(qo) < 1:
        raise ValueError("offset arrays must both have B + 1 entries")
    B = len(qo) - 1
    rank = np.zeros(max(B, 1), dtype=np.int32)
    work = np.zeros(int(num_ranks), dtype=np.int64)
    _ok(lib().gdpa_shard_batch(qp, kp, B, int(H), MASK[mask], int(window), int(num_ranks),
                               rank.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                               work.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))),
        "gdpa_shard_batch")
    return rank[:B], work


def shard_rows(q_off, kv_off, rank_of_sample, rank: int):
    """The local batch of one rank: (local q_off, local kv_off, query row
    indices, key row indices, sample indices) of the samples dealt to
    ``rank``, in their batch order; the index arrays gather the rank's rows
    from (or scatter its results to) the whole batch's token-major tensors."""
    q_off = np.asarray(q_off, dtype=np.int64)
    kv_off = np.asarray(kv_off, dtype=np.int64)
    mine = np.nonzero(np.asarray(rank_of_sample) == rank)[0]
    lq = q_off[mine + 1] - q_off[mine]
    lkv = kv_off[mine + 1] - kv_off[mine]
    qi = np.concatenate([np.arange(q_off[b], q_off[b + 1]) for b in mine] or [np.zeros(0, np.int64)])
    ki = np.concatenate([np.arange(kv_off[b], kv_off[b + 1]) for b in mine] or [np.zeros(0, np.int64)])
    lo = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    lk = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    return lo, lk, qi.astype(np.int64), ki.astype(np.int64), mine


def allreduce_seed_grad(dq, group=None):
    """Shared-query mode over several ranks, each with its own samples: each
    rank's ``dq`` ([n_seeds, H, d] float32 from gdpa_bwd) holds its samples'
    share of the seeds' gradient, and the sum over ranks, one all-reduce of
    that small tensor, is the gradient of the whole batch (the only exchange
    the sharded path has).  In place; returns ``dq``."""
    import torch.distributed as dist
    dist.all_reduce(dq, op=dist.ReduceOp.SUM, group=group)
    return dq


def gdpa_fwd_noalloc(q_off, kv_off, q, k, v, o, alpha=None, act: str = "gelu_erf",
                     mask: str = "none", window: int = 0, stream=None):
    """Forward into a caller-provided ``o`` with no allocation by the library.

    For callers that cannot allocate device memory themselves (see
    ``gdpa_fwd_noalloc`` in include/gdpa.h): bf16, d in {64, 128}, at most
    GDPA_NOALLOC_MAX_TILES (32768) forward tiles.
    """
    qo, qp = _i32(q_off)
    ko, kp = _i32(kv_off)
    B = len(qo) - 1
    H, d = int(q.shape[1]), int(q.shape[2])
    alpha = d ** -0.5 if alpha is None else float(alpha)
    _ok(lib().gdpa_fwd_noalloc(qp, kp, B, H, d, MASK[mask], int(window), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(o), ctypes.c_float(alpha), ACT[act], _stream_ptr(stream)),
        "gdpa_fwd_noalloc")
    return o


def act_eval(x, act: str = "gelu_erf", fast=True, stream=None):
    """(act(x), act'(x)) element-wise with the kernels' device functions
    (``fast``: the tensor-core flavour, one element at a time; ``fast=2``:
    the same in the f32x2 pair form those kernels evaluate it in; false: the
    float32 CUDA-core one).  ``x``: a contiguous float32 CUDA tensor."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    y = torch.empty_like(x)
    dy = torch.empty_like(x)
    mode = 2 if fast == 2 else (1 if fast else 0)
    _ok(lib().gdpa_act_eval(ACT[act], mode, _ptr(x), _ptr(y), _ptr(dy),
                            ctypes.c_int64(x.numel()), _stream_ptr(stream)), "gdpa_act_eval")
    return y, dy


def gdpa_softmax_fwd(plan: Plan, q, k, v, o=None, lse=None, alpha=None, stream=None):
    """Softmax variant (Jagged Flash Attention): (O, lse), lse the row
    log-sum-exp [Tq, H] float32 the backward needs."""
    import torch
    _check(q, plan.q_rows, plan, "q")
    _check(k, plan.Tkv, plan, "k", q.dtype)
    _check(v, plan.Tkv, plan, "v", q.dtype)
    if o is None:
        o = torch.empty((plan.Tq, plan.H, plan.d), dtype=q.dtype, device=q.device)
    _check(o, plan.Tq, plan, "o", q.dtype)
    if lse is None:
        lse = torch.empty((plan.Tq, plan.H), dtype=torch.float32, device=q.device)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (plan.Tq, plan.H) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [Tq, H] tensor")
    alpha = plan.d ** -0.5 if alpha is None else float(alpha)
    _ok(lib().gdpa_softmax_fwd(plan.handle, _dtype_id(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                               _ptr(lse), ctypes.c_float(alpha), _stream_ptr(stream)),
        "gdpa_softmax_fwd")
    return o, lse


def gdpa_softmax_bwd(plan: Plan, q, k, v, o, do, lse, dq=None, dk=None, dv=None, alpha=None,
                     stream=None):
    """(dQ, dK, dV) of the softmax variant from its forward's O and lse."""
    import torch
    f32 = torch.float32
    _check(q, plan.q_rows, plan, "q")
    _check(k, plan.Tkv, plan, "k", q.dtype)
    _check(v, plan.Tkv, plan, "v", q.dtype)
    _check(o, plan.Tq, plan, "o", q.dtype)
    _check(do, plan.Tq, plan, "do", q.dtype)
    if lse.dtype != f32 or tuple(lse.shape) != (plan.Tq, plan.H) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [Tq, H] tensor")
    dq = torch.empty(q.shape, dtype=f32, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=f32, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=f32, device=v.device) if dv is None else dv
    for t, n, rows in ((dq, "dq", plan.q_rows), (dk, "dk", plan.Tkv), (dv, "dv", plan.Tkv)):
        _check(t, rows, plan, n, f32)
    alpha = plan.d ** -0.5 if alpha is None else float(alpha)
    _ok(lib().gdpa_softmax_bwd(plan.handle, _dtype_id(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                               _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                               ctypes.c_float(alpha), _stream_ptr(stream)), "gdpa_softmax_bwd")
    return dq, dk, dv
