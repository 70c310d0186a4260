"""ctypes front end of the float64 GDPA loops in ``gdpa_ref.c``.

TEST INFRASTRUCTURE ONLY (see the package docstring).  ``build()`` compiles
the C file with the host gcc (OpenMP over (sample, head)); the functions below
take NumPy arrays, upcast them to float64 and return float64 arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import ACT_IDS, MASK_IDS

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdpa_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgdpa_ref.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the reference loops; returns the shared-library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i32p = ctypes.POINTER(ctypes.c_int32)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdpa_ref_act.restype = ctypes.c_double
        lib.gdpa_ref_act.argtypes = [ctypes.c_int, ctypes.c_double]
        lib.gdpa_ref_dact.restype = ctypes.c_double
        lib.gdpa_ref_dact.argtypes = [ctypes.c_int, ctypes.c_double]
        lib.gdpa_ref_threads.restype = ctypes.c_int
        lib.gdpa_ref_pairs.restype = ctypes.c_int64
        lib.gdpa_ref_pairs.argtypes = [ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int]
        lib.gdpa_ref_fwd.restype = None
        lib.gdpa_ref_fwd.argtypes = [ctypes.c_int] * 3 + [i32p, i32p] + [dp] * 4 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.gdpa_ref_bwd.restype = None
        lib.gdpa_ref_bwd.argtypes = [ctypes.c_int] * 3 + [i32p, i32p] + [dp] * 7 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.gdpa_ref_lse.restype = None
        lib.gdpa_ref_lse.argtypes = [ctypes.c_int] * 3 + [i32p, i32p] + [dp] * 3 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_int]
        lib.gdpa_ref_softmax_bwd.restype = None
        lib.gdpa_ref_softmax_bwd.argtypes = [ctypes.c_int] * 3 + [i32p, i32p] + [dp] * 7 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_int]
        _lib = lib
    return _lib


def _i32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _f64(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def to_f64(t) -> np.ndarray:
    """torch tensor (any float dtype, any device) or array -> float64 ndarray."""
    if hasattr(t, "detach"):
        import torch
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def threads() -> int:
    return int(_load().gdpa_ref_threads())


def act(kind: str, x: float) -> float:
    return float(_load().gdpa_ref_act(ACT_IDS[kind], float(x)))


def dact(kind: str, x: float) -> float:
    return float(_load().gdpa_ref_dact(ACT_IDS[kind], float(x)))


def pairs(q_off, kv_off, mask: str = "none", window: int = 0) -> int:
    qo, qp = _i32(q_off)
    ko, kp = _i32(kv_off)
    return int(_load().gdpa_ref_pairs(len(qo) - 1, qp, kp, MASK_IDS[mask], int(window)))


def fwd(q_off, kv_off, q, k, v, alpha: float, act: str, mask: str = "none",
        window: int = 0) -> np.ndarray:
    """O for a jagged batch; q/k/v are [T, H, d] (any float type)."""
    qo, qp = _i32(q_off)
    ko, kp = _i32(kv_off)
    Q, Qp = _f64(to_f64(q))
    K, Kp = _f64(to_f64(k))
    V, Vp = _f64(to_f64(v))
    T, H, d = Q.shape
    O = np.zeros_like(Q)
    _load().gdpa_ref_fwd(len(qo) - 1, H, d, qp, kp, Qp, Kp, Vp,
                         O.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                         float(alpha), ACT_IDS[act], MASK_IDS[mask], int(window))
    return O


def bwd(q_off, kv_off, q, k, v, do, alpha: float, act: str, mask: str = "none",
        window: int = 0):
    """(dQ, dK, dV) for a jagged batch given the upstream gradient dO."""
    qo, qp = _i32(q_off)
    ko, kp = _i32(kv_off)
    Q, Qp = _f64(to_f64(q))
    K, Kp = _f64(to_f64(k))
    V, Vp = _f64(to_f64(v))
    dO, dOp = _f64(to_f64(do))
    T, H, d = Q.shape
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dp = ctypes.POINTER(ctypes.c_double)
    if act == "softmax":
        _load().gdpa_ref_softmax_bwd(len(qo) - 1, H, d, qp, kp, Qp, Kp, Vp, dOp,
                                     dQ.ctypes.data_as(dp), dK.ctypes.data_as(dp),
                                     dV.ctypes.data_as(dp), float(alpha), MASK_IDS[mask],
                                     int(window))
        return dQ, dK, dV
    _load().gdpa_ref_bwd(len(qo) - 1, H, d, qp, kp, Qp, Kp, Vp, dOp,
                         dQ.ctypes.data_as(dp), dK.ctypes.data_as(dp), dV.ctypes.data_as(dp),
                         float(alpha), ACT_IDS[act], MASK_IDS[mask], int(window))
    return dQ, dK, dV


def lse(q_off, kv_off, q, k, alpha: float, mask: str = "none", window: int = 0):
    """Row log-sum-exp [T, H] of the softmax variant (-inf for a row without
    a valid key)."""
    qo, qp = _i32(q_off)
    ko, kp = _i32(kv_off)
    Q, Qp = _f64(to_f64(q))
    K, Kp = _f64(to_f64(k))
    T, H, d = Q.shape
    out = np.zeros((T, H), dtype=np.float64)
    _load().gdpa_ref_lse(len(qo) - 1, H, d, qp, kp, Qp, Kp,
                         out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), float(alpha),
                         MASK_IDS[mask], int(window))
    return out


def sub_batch(q_off, kv_off, samples):
    """Offsets and token index arrays of the listed samples, in order.

    Used to run the oracle on a few samples of a batch too large to check in
    full: the returned ``q_idx``/``kv_idx`` select those samples' rows.
    """
    q_off = np.asarray(q_off, dtype=np.int64)
    kv_off = np.asarray(kv_off, dtype=np.int64)
    lq = [int(q_off[b + 1] - q_off[b]) for b in samples]
    lkv = [int(kv_off[b + 1] - kv_off[b]) for b in samples]
    sq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    skv = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    q_idx = np.concatenate([np.arange(q_off[b], q_off[b + 1]) for b in samples] or [np.zeros(0)]).astype(np.int64)
    kv_idx = np.concatenate([np.arange(kv_off[b], kv_off[b + 1]) for b in samples] or [np.zeros(0)]).astype(np.int64)
    return sq, skv, q_idx, kv_idx


def shared_q_tokens(seeds, q_off) -> np.ndarray:
    """Shared-query mode (pooling attention: learned seed queries attend to
    each sample's sequence; GEM page, section on the asymmetric attention
    shapes).  Sample b's queries are seed rows 0 .. Lq_b - 1, so the
    per-token Q [Tq, H, d] is the seeds repeated per sample; the forward and
    backward of shared-query mode are the ordinary ones on this Q."""
    seeds = to_f64(seeds)
    q_off = np.asarray(q_off, dtype=np.int64)
    rows = [seeds[: q_off[b + 1] - q_off[b]] for b in range(len(q_off) - 1)]
    if not rows:
        return np.zeros((0,) + seeds.shape[1:])
    return np.concatenate(rows, axis=0)


def shared_q_grad(dq_tokens, q_off, n_seeds: int) -> np.ndarray:
    """Gradient of the seeds: a parameter used by every sample receives the
    sum of its per-use gradients, i.e. seed i gets the dQ rows of position i
    of all samples."""
    dq_tokens = to_f64(dq_tokens)
    q_off = np.asarray(q_off, dtype=np.int64)
    out = np.zeros((n_seeds,) + dq_tokens.shape[1:])
    for b in range(len(q_off) - 1):
        n = q_off[b + 1] - q_off[b]
        out[:n] += dq_tokens[q_off[b]:q_off[b + 1]]
    return out
