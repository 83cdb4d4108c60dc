"""Pins for the oracle's 8-bit float codecs (oracle/formats.py).

Independent evidence: the maxima the pages print, torch's own float8 CPU casts
(a library routine) over every code and every rounding midpoint, and hand
encodings worked out from the bit layouts.
"""
import numpy as np
import pytest
import torch

from golden.fixtures import load
from oracle import formats as F

CONST = load("format_constants.txt")
TORCH_DT = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def torch_decode(codes, name):
    t = torch.tensor(np.asarray(codes, dtype=np.uint8)).view(TORCH_DT[name])
    return t.to(torch.float64).numpy()


def torch_encode(vals_f32, name):
    t = torch.tensor(np.asarray(vals_f32, dtype=np.float32)).to(TORCH_DT[name])
    return t.view(torch.uint8).numpy()


ALL = np.arange(256, dtype=np.uint8)


def test_printed_maxima():
    e4 = F.decode(ALL, "e4m3")
    e5 = F.decode(ALL, "e5m2")
    assert np.nanmax(e4[np.isfinite(e4)]) == CONST["e4m3_max"] == F.E4M3.max
    assert np.nanmax(e5[np.isfinite(e5)]) == CONST["e5m2_max"] == F.E5M2.max
    assert F.decode(0x7E, "e4m3") == 448.0
    assert F.decode(0x7B, "e5m2") == 57344.0


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_decode_matches_torch_all_codes(name):
    ours = F.decode(ALL, name)
    ref = torch_decode(ALL, name)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))


def test_special_codes_by_hand():
    # E4M3fn: S.1111.111 is NaN, no infinities; smallest subnormal 2^-9, smallest normal 2^-6
    assert np.isnan(F.decode(0x7F, "e4m3")) and np.isnan(F.decode(0xFF, "e4m3"))
    assert F.decode(0x01, "e4m3") == 2.0 ** -9
    assert F.decode(0x08, "e4m3") == 2.0 ** -6
    assert F.decode(0x38, "e4m3") == 1.0
    # E5M2: exponent 31 is inf (m == 0) / NaN; subnormal 2^-16, normal 2^-14
    assert F.decode(0x7C, "e5m2") == np.inf and F.decode(0xFC, "e5m2") == -np.inf
    assert np.isnan(F.decode(0x7D, "e5m2"))
    assert F.decode(0x01, "e5m2") == 2.0 ** -16
    assert F.decode(0x04, "e5m2") == 2.0 ** -14
    assert F.decode(0x3C, "e5m2") == 1.0
    assert np.signbit(F.decode(0x80, "e4m3")) and F.decode(0x80, "e4m3") == 0.0


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_encode_inverts_decode(name):
    vals = F.decode(ALL, name)
    fin = np.isfinite(vals)
    assert np.array_equal(F.encode(vals[fin], name), ALL[fin])


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_midpoints_ties_to_even_and_match_torch(name):
    vals = F.decode(np.arange(0x00, 0x80, dtype=np.uint8), name)
    pos = vals[np.isfinite(vals)]
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2  # exact in fp32: at most mbits + 2 significant bits
    mid32 = mid.astype(np.float32)
    assert np.array_equal(mid32.astype(np.float64), mid)
    codes = F.encode(mid, name)
    # ties go to the code whose mantissa LSB is 0
    assert np.all(codes & 1 == 0)
    assert np.array_equal(codes, torch_encode(mid32, name))
    # one fp32 ulp either side of each midpoint rounds to the neighbours
    below = np.nextafter(mid32, np.float32(0))
    above = np.nextafter(mid32, np.float32(np.inf))
    assert np.array_equal(F.decode(F.encode(below, name), name), lo)
    assert np.array_equal(F.decode(F.encode(above, name), name), hi)
    assert np.array_equal(F.encode(-mid, name), torch_encode(-mid32, name))


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_random_values_match_torch(name):
    mx = F.fmt_of(name).max
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(-mx, mx, 200_000),
        rng.standard_normal(200_000) * 2.0 ** rng.integers(-20, 10, 200_000),
    ]).astype(np.float32)
    x = np.clip(x, -mx, mx)
    assert np.array_equal(F.encode(x, name), torch_encode(x, name))


def test_hand_encodings():
    # 1.0 = 0.0111.000, 0.5 = 0.0110.000, -448 = 1.1111.110, 224 = 0.1110.110
    assert list(F.encode([1.0, 0.5, -448.0, 224.0], "e4m3")) == [0x38, 0x30, 0xFE, 0x76]
    # half the smallest subnormal ties to +0; 3 * 2^-10 ties to the even 2^-8 (m = 2)
    assert list(F.encode([2.0 ** -10, 3 * 2.0 ** -10, -0.0], "e4m3")) == [0x00, 0x02, 0x80]
    # E5M2: 57344 = 0.11110.11, 1.0 = 0.01111.00
    assert list(F.encode([57344.0, 1.0], "e5m2")) == [0x7B, 0x3C]
    # mantissa carry into the next binade: 15.5 is a tie between 15 (m = 7) and 16 -> 16
    assert F.encode([15.5], "e4m3")[0] == 0x58


def test_encode_rejects_unclipped():
    with pytest.raises(ValueError):
        F.encode([449.0], "e4m3")
    with pytest.raises(ValueError):
        F.encode([np.nan], "e4m3")


def test_e8m0():
    assert F.e8m0_decode(127) == 1.0
    assert F.e8m0_decode(0) == 2.0 ** -127
    assert F.e8m0_decode(254) == 2.0 ** 127
    assert np.isnan(F.e8m0_decode(255))
    if hasattr(torch, "float8_e8m0fnu"):
        b = np.arange(255, dtype=np.uint8)
        ref = torch.tensor(b).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert np.array_equal(F.e8m0_decode(b), ref)
    assert list(F.e8m0_encode([-127, 0, 127])) == [0, 127, 254]


def test_ceil_log2_bounds():
    rng = np.random.default_rng(3)
    s = (rng.uniform(0.5, 1.0, 50_000) * 2.0 ** rng.integers(-140, 120, 50_000)).astype(np.float32)
    s = s[s > 0]
    e = F.ceil_log2_f32(s)
    s64 = s.astype(np.float64)
    assert np.all(np.ldexp(1.0, e - 1) < s64) and np.all(s64 <= np.ldexp(1.0, e))
    p = np.ldexp(np.float32(1.0), np.arange(-149, 128)).astype(np.float32)
    assert np.array_equal(F.ceil_log2_f32(p), np.arange(-149, 128))
