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
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = E4M3_TABLE[:0x7F]


def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3 code to each value, ties to the even code, saturating to
    +-448, NaN to 0x7F (F2).  Plain search over the 127 non-negative values."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    flat, res = x.reshape(-1), out.reshape(-1)
    for i, v in enumerate(flat):
        if np.isnan(v):
            res[i] = 0x7F
            continue
        sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
        a = min(abs(v), E4M3_MAX)
        hi = int(np.searchsorted(_POS_VALUES, a, side="left"))   # first value >= a
        if hi < len(_POS_VALUES) and _POS_VALUES[hi] == a:
            c = hi
        else:
            lo = hi - 1
            d_lo, d_hi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
            if d_lo < d_hi:
                c = lo
            elif d_hi < d_lo:
                c = hi
            else:
                c = lo if lo % 2 == 0 else hi      # tie: the even code
        res[i] = sign | int(_POS_CODES[c])
    return out


def quantize(x, scale: float) -> np.ndarray:
    """Codes of x / scale (F2)."""
    return e4m3_encode(np.asarray(x, dtype=np.float64) / scale)


def dequantize(codes, scale: float) -> np.ndarray:
    """Values the attention reads: code * scale (F3)."""
    return e4m3_decode(codes) * scale
