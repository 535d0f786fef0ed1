"""Number-format emulation for the oracle (test infrastructure only).

Written from the format definitions, not from any library routine:

* E4M3 (OCP FP8, "E4M3FN" variant): 1 sign bit, 4 exponent bits with bias 7,
  3 mantissa bits; no infinities; exponent 15 with mantissa 7 is NaN, so the
  largest finite magnitude is 2^8 * 1.75 = 448; subnormals have spacing 2^-9.
  Conversion is round-to-nearest-even with saturation to +-448 (the
  "satfinite" behaviour the pages' static-scale FP8 convert needs: a static
  scale cannot guarantee |x| <= 448, and clamping keeps the value finite).
* BF16: float32 with the low 16 mantissa bits dropped (8 significant bits),
  round-to-nearest-even.
* E2M1 (NVFP4 element): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit:
  magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; round-to-nearest-even, saturating
  at 6.
* fp32: IEEE binary32 round-to-nearest-even (numpy's float32 cast).

All functions take and return float64 arrays of *values* (codes are exposed
separately where a test needs them).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _round_to_grid(x: np.ndarray, mant_bits: int, min_exp: int, max_val: float) -> np.ndarray:
    """Round |x| to the nearest value of a binary float grid, ties to even.

    mant_bits: explicit mantissa bits; min_exp: exponent of the smallest normal
    binade (values below 2^min_exp use the subnormal spacing 2^(min_exp-mant_bits)).
    Saturates to max_val. NaN propagates.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # exponent e with 2^e <= a < 2^(e+1); frexp gives a = f * 2^E with 0.5 <= f < 1
    _, E = np.frexp(a)
    e = np.maximum(E - 1, min_exp)
    spacing = np.ldexp(1.0, e - mant_bits)
    q = a / spacing                       # exact: power-of-two division
    r = np.round(q)                       # numpy rounds half to even
    out = r * spacing
    out = np.minimum(out, max_val)
    out = np.where(np.isnan(a), np.nan, out)
    return np.copysign(out, x)


def e4m3(x) -> np.ndarray:
    """Round to E4M3 (RNE, saturate to +-448); returns the represented values."""
    return _round_to_grid(x, mant_bits=3, min_exp=-6, max_val=E4M3_MAX)


def e2m1(x) -> np.ndarray:
    """Round to E2M1 (RNE, saturate to +-6); returns the represented values."""
    return _round_to_grid(x, mant_bits=1, min_exp=0, max_val=E2M1_MAX)


def bf16(x) -> np.ndarray:
    """Round to bf16 (RNE); exponent range as float32 (no saturation needed here)."""
    x = np.asarray(x, dtype=np.float64)
    return _round_to_grid(x, mant_bits=7, min_exp=-126, max_val=np.inf)


def fp32(x) -> np.ndarray:
    """Round to IEEE binary32 (RNE) and return as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ---- codes (bit patterns), for exhaustive checks and for reading GPU buffers ----

def e4m3_decode_code(code) -> np.ndarray:
    """Decode E4M3 byte codes (uint8) to values, from the format definition."""
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3_encode_code(x) -> np.ndarray:
    """Values -> E4M3 byte codes (after RNE/saturation). -0.0 maps to 0x80."""
    v = e4m3(x)
    a = np.abs(v)
    _, E = np.frexp(a)
    e = np.maximum(E - 1, -6)
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e + 7, 0)
    mant = np.where(normal, a / np.ldexp(1.0, e) - 1.0, a / 2.0 ** -6) * 8.0
    mant = np.rint(mant).astype(np.int64)
    code = (exp_field.astype(np.int64) << 3) | mant
    code = np.where(np.signbit(v), code | 0x80, code)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def e2m1_decode_code(code) -> np.ndarray:
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, e - 1))
    return np.where(s == 1, -mag, mag)


def e2m1_encode_code(x) -> np.ndarray:
    v = e2m1(x)
    table = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
    a = np.abs(v)
    code = np.zeros(a.shape, np.int64)
    for val, c in table.items():
        code = np.where(a == val, c, code)
    code = np.where(np.signbit(v), code | 0x8, code)
    return code.astype(np.uint8)


def bf16_decode_bits(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
