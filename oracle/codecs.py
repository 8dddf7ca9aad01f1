"""Output-cast codecs for the oracle, written from the number formats' definitions.

bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored mantissa bits; the
same exponent range as IEEE binary32, subnormals down to 2**-133.

FP8 e4m3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
bits, no infinities, largest finite magnitude 448 = 1.75 * 2**8, the all-ones
pattern S.1111.111 is NaN, subnormals m/8 * 2**-6 down to 2**-9.

Both encoders round to nearest, ties to even, directly from the float64 value
(no intermediate float32 rounding). The e4m3 encoder saturates to +-448
("satfinite"), which is the cast the FlashMLA PR #25 epilogue and the combine
perform when they emit FP8 ("What changes": the FP8 cast moves to the combine).
"""
from __future__ import annotations

import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
E4M3_MAX = 448.0


def _round_to_grid(x: np.ndarray, mant_bits: int, min_normal_exp: int) -> np.ndarray:
    """Round float64 x to the nearest value with `mant_bits` stored mantissa bits.

    Exponents below `min_normal_exp` use the subnormal quantum
    2**(min_normal_exp - mant_bits). np.rint rounds half to even.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    # exponent e with 2**e <= |x| < 2**(e+1)
    with np.errstate(divide="ignore"):
        _, e = np.frexp(ax)          # ax = f * 2**e, f in [0.5, 1)
    e = e.astype(np.int64) - 1
    e = np.maximum(e, min_normal_exp)
    quantum = np.ldexp(1.0, (e - mant_bits).astype(np.int64))
    return np.rint(x / quantum) * quantum


def bf16_round(x) -> np.ndarray:
    """Float64 -> nearest bf16 value (returned as float64), +-inf on overflow."""
    x = np.asarray(x, dtype=np.float64)
    r = _round_to_grid(x, 7, -126)
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)
    return np.where(np.isnan(x), np.nan, r)


def bf16_bits(x) -> np.ndarray:
    """Float64 -> bf16 bit pattern (uint16) after RNE rounding."""
    r = bf16_round(x).astype(np.float32)       # exact: every bf16 value is a float32
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def bf16_decode(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """uint8 e4m3 codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = np.ldexp(1.0 + man / 8.0, exp - 7)
    sub = np.ldexp(man / 8.0, -6)
    val = sign * np.where(exp == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_round(y) -> np.ndarray:
    """Float64 -> nearest e4m3 value, ties to even, saturating to +-448."""
    y = np.asarray(y, dtype=np.float64)
    r = _round_to_grid(y, 3, -6)
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def e4m3_encode(y) -> np.ndarray:
    """Float64 -> uint8 e4m3 code (RNE, satfinite). NaN maps to 0x7F."""
    y = np.asarray(y, dtype=np.float64)
    r = e4m3_round(y)
    ar = np.abs(r)
    sign = np.where(np.signbit(r), 0x80, 0).astype(np.int64)
    with np.errstate(divide="ignore"):
        _, e = np.frexp(ar)
    e = e.astype(np.int64) - 1                      # 2**e <= ar < 2**(e+1)
    is_sub = ar < 2.0 ** -6
    exp_field = np.where(is_sub, 0, e + 7)
    man_normal = np.rint((ar / np.ldexp(1.0, e) - 1.0) * 8.0)
    man_sub = np.rint(ar / 2.0 ** -9)
    man = np.where(is_sub, man_sub, man_normal).astype(np.int64)
    code = sign | (exp_field << 3) | man
    code = np.where(ar == 0, sign, code)
    code = np.where(np.isnan(y), 0x7F, code)
    return code.astype(np.uint8)
