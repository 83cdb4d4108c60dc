"""Pin of reading R1: the quantizer DIVIDES by the scale (Flax FP8 guide,
2.2 ``quantize``: ``x / scale``), it does not multiply by a reciprocal (the
nanochat module, "实现", multiplies by MAX / amax -- the rejected reading).

The two differ only in the last fp32 bit of the quotient, which decides the
FP8 code when the exact quotient sits on an FP8 rounding midpoint.  The
expected codes here come from exact rational arithmetic written in this file
(``fractions.Fraction``, fp32 and FP8 round-to-nearest-even by hand, the FP8
values enumerated with torch's own float8 dtypes), not from the oracle:

    x = m * s exactly (m an FP8 midpoint, s an fp32 scale with few bits), so
    x / s = m exactly, fl32(m) = m, and the FP8 cast breaks the tie to the
    even code; fl32(x * fl32(1 / s)) is m moved by an fp32 ulp for the scales
    chosen, which rounds to the odd neighbour.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import quantize as OQ


def _fp32_rne(q: Fraction) -> Fraction:
    """Round a positive rational to the nearest fp32 value (normal range),
    ties to even."""
    assert q > 0
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    assert -126 <= e <= 127
    unit = Fraction(2) ** (e - 23)
    n = q / unit
    lo = n.numerator // n.denominator
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return lo * unit


def _fp8_values(dtype):
    """(code, exact value) of every finite non-negative FP8 code, from torch."""
    codes = torch.arange(0, 128, dtype=torch.uint8)
    vals = codes.view(dtype).float().tolist()
    return [(c, Fraction(v)) for c, v in zip(range(128), vals) if np.isfinite(v)]


def _fp8_rne(q: Fraction, table):
    """Nearest FP8 code of a non-negative rational, ties to the even code."""
    best = min(table, key=lambda cv: (abs(cv[1] - q), cv[0] % 2))
    return best[0]


def _midpoint_cases(dtype, fmt_max, limit):
    table = _fp8_values(dtype)
    mids = [(table[i][1] + table[i + 1][1]) / 2 for i in range(1, len(table) - 1)
            if table[i + 1][1] <= fmt_max]
    cases = []
    # scales with few significant bits, so that x = m * s is an exact fp32 value
    for num in range(3, 4000, 2):
        s = Fraction(num, 1 << 12)
        for m in mids:
            x = m * s
            if x.denominator & (x.denominator - 1) or _fp32_rne(x) != x:
                continue
            r = _fp32_rne(1 / s)
            p = _fp32_rne(x * r)
            if p == m:
                continue
            want = _fp8_rne(m, table)          # x / s == m exactly: the tie
            recip = _fp8_rne(p, table)         # the rejected reading
            if want != recip:
                cases.append((float(x), float(s), want, recip))
        if len(cases) >= limit:
            break
    return cases


@pytest.mark.parametrize("fmt,dtype,fmt_max", [("e4m3", torch.float8_e4m3fn, 448),
                                               ("e5m2", torch.float8_e5m2, 57344)])
def test_quantize_divides_not_reciprocal(fmt, dtype, fmt_max):
    cases = _midpoint_cases(dtype, fmt_max, limit=24)
    assert len(cases) >= 12, "too few discriminating cases found"
    x = np.array([c[0] for c in cases], dtype=np.float32)
    s = np.array([c[1] for c in cases], dtype=np.float32)
    # the inputs are the exact rationals (fp32 carries them without rounding)
    assert all(Fraction(float(a)) == Fraction(c[0]) for a, c in zip(x, cases))
    got = OQ.quantize_with_scale(x, s, fmt)
    want = np.array([c[2] for c in cases], dtype=np.uint8)
    recip = np.array([c[3] for c in cases], dtype=np.uint8)
    assert np.array_equal(got, want)
    assert np.all(got != recip)
    # negative inputs mirror: the sign bit is the only difference
    got_neg = OQ.quantize_with_scale(-x, s, fmt)
    assert np.array_equal(got_neg, want | 0x80)
