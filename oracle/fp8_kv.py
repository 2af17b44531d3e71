"""fp8 (e4m3) KV cache for the oracle -- TEST INFRASTRUCTURE.

The pages' deployment runs vLLM with an fp8 KV cache ("P-EAGLE: Faster LLM
Inference with Parallel Speculative Decoding in vLLM", experiment setup:
software and system configuration, --kv-cache-dtype fp8).  The pages fix no
more than that; the readings here follow the usual form of such a cache:

  F1 format: OCP FP8 E4M3 -- 1 sign bit, 4 exponent bits (bias 7), 3
     mantissa bits; exponent field 0 is subnormal (m / 8 * 2^-6); no
     infinities; S.1111.111 is NaN, so the largest finite value is
     1.75 * 2^8 = 448.
  F2 quantisation: k / k_scale (v / v_scale) rounded to the nearest e4m3
     value, ties to the even code, saturating to +-448; one scale per layer
     and per K or V (a per-tensor scale, 1.0 unless calibrated).
  F3 attention reads code * scale.

Only the tests may import it (the library shares no code with it).
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_value(code: int) -> float:
    """Value of one e4m3 code from the format definition (F1)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


# the non-negative finite codes in increasing order of value (0x00 .. 0x7E)
_POS_VALUES = E4M3_TABLE[:0x7F]


def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3 code to each value, ties to the even code, saturating to
    +-448, NaN to 0x7F (F2): the two neighbours of |x| among the 127
    non-negative values, the nearer one, the even code on a tie."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)
    n = len(_POS_VALUES)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, n - 1)  # first value >= a
    lo = np.clip(hi - 1, 0, n - 1)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    c = np.where(_POS_VALUES[hi] == a, hi,
                 np.where(d_lo < d_hi, lo,
                          np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi))))
    sign = (x < 0) | ((x == 0) & np.signbit(x))
    code = (c | np.where(sign, 0x80, 0)).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), code).astype(np.uint8)


def quantize(x, scale: float) -> np.ndarray:
    """Codes of x / scale (F2)."""
    return e4m3_encode(np.asarray(x, dtype=np.float64) / scale)


def dequantize(codes, scale: float) -> np.ndarray:
    """Values the attention reads: code * scale (F3)."""
    return e4m3_decode(codes) * scale
