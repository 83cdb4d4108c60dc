"""8-bit floating-point codecs, written from the format definitions.

Test infrastructure only (see ``oracle/__init__``).

* E4M3fn (Flax guide section 1 ``float8_e4m3fn``; nanochat module "实现",
  ``FP8_MAX = 448``): sign, 4 exponent bits with bias 7, 3 mantissa bits, no
  infinities, ``S.1111.111`` is NaN; largest finite 1.75 * 2**8 = 448,
  smallest normal 2**-6, subnormals m * 2**-9.
* E5M2 (nanochat module "实现", gradients with max 57344): bias 15, 2
  mantissa bits, IEEE-style inf/NaN at exponent 31; largest finite
  1.75 * 2**15 = 57344, smallest normal 2**-14, subnormals m * 2**-16.
* UE8M0 / E8M0 (Transformers fine-grained FP8 section 四 ``scale_fmt``,
  section 七; MOSS section 4 local factor): one unsigned byte holding a pure
  power of two, value 2**(b - 127); 0xFF is NaN.

``encode`` rounds to nearest, ties to even (the cast the Flax ``quantize``
applies after clipping, section 2.2), and keeps the sign of zero.

Pinned by ``tests/test_oracle_formats.py``: the printed maxima (448, 57344),
torch's own float8 CPU casts over every code and every midpoint, and
encode(decode(c)) == c for every finite code.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Fp8Format:
    name: str
    ebits: int
    mbits: int
    bias: int
    max: float
    ieee_specials: bool  # True: exponent all-ones is inf/NaN (E5M2)

    @property
    def min_normal_exp(self) -> int:
        return 1 - self.bias


E4M3 = Fp8Format("e4m3fn", ebits=4, mbits=3, bias=7, max=448.0, ieee_specials=False)
E5M2 = Fp8Format("e5m2", ebits=5, mbits=2, bias=15, max=57344.0, ieee_specials=True)

FORMATS = {"e4m3": E4M3, "e4m3fn": E4M3, "e5m2": E5M2}


def fmt_of(fmt) -> Fp8Format:
    return fmt if isinstance(fmt, Fp8Format) else FORMATS[fmt]


def decode(codes, fmt) -> np.ndarray:
    """uint8 codes -> float64 values."""
    f = fmt_of(fmt)
    c = np.asarray(codes, dtype=np.int64)
    sign = (c >> 7) & 1
    e = (c >> f.mbits) & ((1 << f.ebits) - 1)
    m = c & ((1 << f.mbits) - 1)
    sub = m * np.ldexp(1.0, f.min_normal_exp - f.mbits)
    nrm = (1.0 + m / float(1 << f.mbits)) * np.ldexp(1.0, e - f.bias)
    mag = np.where(e == 0, sub, nrm)
    emax_field = (1 << f.ebits) - 1
    if f.ieee_specials:
        mag = np.where((e == emax_field) & (m == 0), np.inf, mag)
        mag = np.where((e == emax_field) & (m != 0), np.nan, mag)
    else:
        mag = np.where((e == emax_field) & (m == (1 << f.mbits) - 1), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def encode(y, fmt) -> np.ndarray:
    """Finite values with |y| <= MAX -> uint8 codes, round-to-nearest-even.

    Values must already be clipped to the format's range (the quantizer clips
    before casting); anything else is a caller error.
    """
    f = fmt_of(fmt)
    y = np.asarray(y, dtype=np.float64)
    if not np.all(np.isfinite(y)):
        raise ValueError("encode: non-finite input")
    if np.any(np.abs(y) > f.max):
        raise ValueError("encode: input outside +-MAX (clip first)")
    sign = np.signbit(y).astype(np.int64) << 7
    a = np.abs(y)
    _, ex = np.frexp(a)                   # a = frac * 2**ex, frac in [0.5, 1)
    e_unb = np.maximum(ex - 1, f.min_normal_exp)
    quantum = np.ldexp(1.0, e_unb - f.mbits)
    v = np.rint(a / quantum) * quantum    # exact power-of-two scaling; rint ties to even
    _, exv = np.frexp(v)
    is_sub = v < np.ldexp(1.0, f.min_normal_exp)
    e_field = np.where(is_sub, 0, exv - 1 + f.bias)
    m_norm = (v / np.ldexp(1.0, exv - 1) - 1.0) * (1 << f.mbits)
    m_sub = v / np.ldexp(1.0, f.min_normal_exp - f.mbits)
    m_field = np.where(is_sub, m_sub, m_norm)
    code = sign | (e_field.astype(np.int64) << f.mbits) | m_field.astype(np.int64)
    return code.astype(np.uint8)


# ---------------------------------------------------------------- E8M0 ----

E8M0_BIAS = 127


def e8m0_decode(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.int64)
    return np.where(b == 0xFF, np.nan, np.ldexp(1.0, b - E8M0_BIAS))


def e8m0_encode(exponent) -> np.ndarray:
    """Power-of-two exponent e in [-127, 127] -> byte e + 127."""
    e = np.asarray(exponent, dtype=np.int64)
    if np.any(e < -127) or np.any(e > 127):
        raise ValueError("e8m0_encode: exponent outside [-127, 127]")
    return (e + E8M0_BIAS).astype(np.uint8)


def ceil_log2_f32(s) -> np.ndarray:
    """Exact ceil(log2(s)) of positive float32 values.

    ``s = frac * 2**ex`` with frac in [0.5, 1); s is a power of two exactly when
    frac == 0.5, and then log2(s) = ex - 1; otherwise the ceiling is ex.
    """
    s = np.asarray(s, dtype=np.float32).astype(np.float64)
    if np.any(~(s > 0)) or not np.all(np.isfinite(s)):
        raise ValueError("ceil_log2_f32: needs finite positive values")
    frac, ex = np.frexp(s)
    return np.where(frac == 0.5, ex - 1, ex).astype(np.int64)
