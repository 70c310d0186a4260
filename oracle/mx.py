"""MXFP8 (E4M3 elements, E8M0 block scales) quantisation, restated in float64.
TEST INFRASTRUCTURE ONLY (see the package docstring).

The GEM page ("GEM 트레이닝: Meta가 LLM 규모의 광고 파운데이션 모델 효율성을
두 배로 높인 방법", techlist.io, section "GPU 연산 효율을 높인 맞춤형 커널과
정밀도") says attention and MLP train in mixed ultra-low precision that
includes MXFP8, with the precision chosen per operation.  The format itself is
the OCP Microscaling (MX) one: blocks of 32 consecutive elements share one
power-of-two scale (an E8M0 exponent), and each element is an FP8 E4M3 number:

* E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
  holds the subnormals m/8 * 2^-6; field 15 with mantissa 7 is NaN (no
  infinities), so the largest finite magnitude is 1.75 * 2^8 = 448.
* Block scale: X = 2^(floor(log2(max|x|)) - 8), 8 being the exponent of
  E4M3's largest normal; an all-zero block takes X = 2^-127.  Elements are
  x / X rounded to the nearest E4M3 value (ties to the even mantissa) and
  clamped to +-448 (the block maximum can land in (448, 512)).  The value a
  block stands for is element * X.

Reading taken for GDPA (the pages give no more than the format's name): Q and
K are quantised along the head dimension d (the contraction of S = Q K^T), so
the scores see the dequantised Q and K; V, P and the output stay as in the
bf16 path.  The oracle of that variant is the ordinary float64 GDPA applied
to ``dequantise(quantise(Q))`` and the same for K.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal
E4M3_EMIN = -6         # exponent of the smallest normal
MANT_BITS = 3
BLOCK = 32


def e4m3_value(code: int) -> float:
    """The number an 8-bit E4M3 code stands for (NaN for the two NaN codes)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** E4M3_EMIN
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def round_e4m3(x) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to the even mantissa, clamped to
    +-448.  Works element-wise on float64 arrays."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # spacing of the representable values around a: 2^(e - 3) for a normal
    # a in [2^e, 2^(e+1)), 2^-9 in the subnormal range
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, E4M3_EMIN)
    step = 2.0 ** (e - MANT_BITS)
    q = a / step
    r = np.floor(q)
    frac = q - r
    up = (frac > 0.5) | ((frac == 0.5) & (np.fmod(r, 2.0) == 1.0))
    r = r + up
    out = np.minimum(r * step, E4M3_MAX)
    return np.copysign(out, x)


def block_exponents(x, block: int = BLOCK) -> np.ndarray:
    """E8M0 exponent of each block of ``block`` consecutive elements along the
    last axis (its length must be a multiple of ``block``)."""
    x = np.asarray(x, dtype=np.float64)
    if x.shape[-1] % block:
        raise ValueError("last axis must be a multiple of the block size")
    b = x.reshape(x.shape[:-1] + (x.shape[-1] // block, block))
    amax = np.max(np.abs(b), axis=-1)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - E4M3_EMAX
    e = np.where(amax > 0, e, -127.0)
    return np.clip(e, -127, 127).astype(np.int32)


def quantise(x, block: int = BLOCK):
    """(elements, exponents): E4M3 values (as float64) of x / 2^exponent per
    block, and the blocks' E8M0 exponents."""
    x = np.asarray(x, dtype=np.float64)
    ex = block_exponents(x, block)
    scale = np.repeat(2.0 ** ex.astype(np.float64), block, axis=-1)
    return round_e4m3(x / scale), ex


def dequantise(elements, exponents, block: int = BLOCK) -> np.ndarray:
    """The values the blocks stand for: element * 2^exponent."""
    scale = np.repeat(2.0 ** np.asarray(exponents, dtype=np.float64), block, axis=-1)
    return np.asarray(elements, dtype=np.float64) * scale


def mx_round_trip(x, block: int = BLOCK) -> np.ndarray:
    """dequantise(quantise(x)): what an MXFP8 operand contributes."""
    el, ex = quantise(x, block)
    return dequantise(el, ex, block)
