"""Exact float64 values of stored fp16, bf16 and e4m3 codes, from the format definitions.

Test infrastructure only (see ``oracle/__init__``).

Every code is decoded bit by bit: sign, biased exponent, mantissa, with the
subnormal and special cases of each format.  Tables of all codes are built once.

* binary16 (fp16): 1 sign, 5 exponent bits (bias 15), 10 mantissa bits, IEEE specials.
* bfloat16: 1 sign, 8 exponent bits (bias 127), 7 mantissa bits, IEEE specials.
* e4m3 ("fn" variant, the fp8 KV-cache format): 1 sign, 4 exponent bits (bias 7),
  3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448.

``encode_e4m3`` is round-to-nearest-even with saturation to ±448 ("satfinite"),
written as a search over the finite code values — the quantisation rule a fp8
KV write uses.
"""
from __future__ import annotations

import numpy as np

_F16_TABLE = None
_BF16_TABLE = None
_E4M3_TABLE = None


def _ieee_value(sign: int, exp: int, man: int, exp_bits: int, man_bits: int) -> float:
    bias = (1 << (exp_bits - 1)) - 1
    if exp == (1 << exp_bits) - 1:
        if man == 0:
            return -np.inf if sign else np.inf
        return np.nan
    if exp == 0:
        mag = man * 2.0 ** (1 - bias - man_bits)
    else:
        mag = (1.0 + man / float(1 << man_bits)) * 2.0 ** (exp - bias)
    return -mag if sign else mag


def f16_table() -> np.ndarray:
    global _F16_TABLE
    if _F16_TABLE is None:
        t = np.empty(1 << 16, dtype=np.float64)
        for c in range(1 << 16):
            t[c] = _ieee_value(c >> 15, (c >> 10) & 0x1F, c & 0x3FF, 5, 10)
        _F16_TABLE = t
    return _F16_TABLE


def bf16_table() -> np.ndarray:
    global _BF16_TABLE
    if _BF16_TABLE is None:
        t = np.empty(1 << 16, dtype=np.float64)
        for c in range(1 << 16):
            t[c] = _ieee_value(c >> 15, (c >> 7) & 0xFF, c & 0x7F, 8, 7)
        _BF16_TABLE = t
    return _BF16_TABLE


def e4m3_value(code: int) -> float:
    sign, exp, man = code >> 7, (code >> 3) & 0xF, code & 0x7
    if exp == 0xF and man == 0x7:
        return np.nan
    if exp == 0:
        mag = man * 2.0 ** (1 - 7 - 3)          # subnormal: m/8 * 2^-6
    else:
        mag = (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return -mag if sign else mag


def e4m3_table() -> np.ndarray:
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
    return _E4M3_TABLE


def to_f64(codes: np.ndarray, dtype: str) -> np.ndarray:
    """Decode an array of stored codes (uint16 for f16/bf16, uint8 for e4m3) to float64."""
    codes = np.asarray(codes)
    if dtype == "f16":
        return f16_table()[codes.view(np.uint16) if codes.dtype != np.uint16 else codes]
    if dtype == "bf16":
        return bf16_table()[codes.view(np.uint16) if codes.dtype != np.uint16 else codes]
    if dtype == "e4m3":
        return e4m3_table()[codes.view(np.uint8) if codes.dtype != np.uint8 else codes]
    raise ValueError(f"unknown dtype {dtype}")


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """Round float64 values to e4m3 codes: nearest, ties to even mantissa, saturate to ±448."""
    x = np.asarray(x, dtype=np.float64)
    table = e4m3_table()
    pos_codes = np.array([c for c in range(0x7F)], dtype=np.int64)   # +0 .. +448, ascending
    pos_vals = table[pos_codes]
    out = np.empty(x.shape, dtype=np.uint8)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for i, v in enumerate(flat_in):
        if np.isnan(v):
            flat_out[i] = 0x7F
            continue
        sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
        a = min(abs(v), 448.0)
        k = int(np.searchsorted(pos_vals, a))          # pos_vals[k-1] < a <= pos_vals[k]
        if k < len(pos_vals) and pos_vals[k] == a:
            code = int(pos_codes[k])
        else:
            lo, hi = int(pos_codes[k - 1]), int(pos_codes[k])
            dlo, dhi = a - table[lo], table[hi] - a
            if dlo < dhi:
                code = lo
            elif dhi < dlo:
                code = hi
            else:                                        # tie: even mantissa
                code = lo if (lo & 1) == 0 else hi
        flat_out[i] = sign | code
    return out
