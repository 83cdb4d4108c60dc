"""Pins for the float64 dequantized GEMM (oracle/gemm.py) and its tolerance.

Evidence: exact rational arithmetic (fractions.Fraction over values decoded by
torch's float8 dtypes) on tiny shapes, an integer matmul on the E4M3 code grid
for unit scales, and plausible mistakes (a transposed operand, a dropped scale,
a sign flip, a per-group scale applied to the wrong group) each failing the
acceptance check.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads
from oracle import gemm as G
from oracle import quantize as Q

F32 = np.float32


def torch_decode(codes, name):
    dt = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}[name]
    return torch.tensor(np.asarray(codes, dtype=np.uint8)).view(dt).to(torch.float64).numpy()


def finite_codes(rng, shape, name):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    bad = np.isnan(torch_decode(c, name)) | np.isinf(torch_decode(c, name))
    c[bad] = 0x38 if name == "e4m3" else 0x3C
    return c


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (8, 8, 8), (2, 7, 4)])
@pytest.mark.parametrize("names", [("e4m3", "e4m3"), ("e5m2", "e4m3")])
def test_exact_rational_brute_force(shape, names):
    m, n, k = shape
    rng = np.random.default_rng(m * 100 + n * 10 + k)
    qa, qb = finite_codes(rng, (m, k), names[0]), finite_codes(rng, (n, k), names[1])
    sa, sb = F32(rng.uniform(1e-3, 10)), F32(rng.uniform(1e-3, 10))
    c, e = G.gemm(G.dequant_operand(qa, names[0], sa), G.dequant_operand(qb, names[1], sb))
    av, bv = torch_decode(qa, names[0]), torch_decode(qb, names[1])
    for i in range(m):
        for j in range(n):
            exact = sum(Fraction(av[i, t]) * Fraction(bv[j, t]) for t in range(k))
            exact *= Fraction(float(sa)) * Fraction(float(sb))
            mag = sum(abs(Fraction(av[i, t]) * Fraction(bv[j, t])) for t in range(k))
            mag *= Fraction(float(sa)) * Fraction(float(sb))
            assert abs(Fraction(c[i, j]) - exact) <= Fraction(2, 10 ** 15) * (mag + 1)
            assert abs(Fraction(e[i, j]) - mag) <= Fraction(2, 10 ** 15) * (mag + 1)


def test_unit_scale_equals_integer_grid_matmul():
    # every finite E4M3 value is an integer multiple of 2^-9
    rng = np.random.default_rng(1)
    qa, qb = finite_codes(rng, (16, 32), "e4m3"), finite_codes(rng, (64, 32), "e4m3")
    ia = (torch_decode(qa, "e4m3") * 512).astype(np.int64)
    ib = (torch_decode(qb, "e4m3") * 512).astype(np.int64)
    c, _ = G.gemm(G.dequant_operand(qa, "e4m3", 1.0), G.dequant_operand(qb, "e4m3", 1.0))
    assert np.array_equal(c * 512 * 512, (ia @ ib.T).astype(np.float64))


def test_group_scales_brute_force():
    rng = np.random.default_rng(5)
    m, n, k = 3, 130, 256
    qa, qb = finite_codes(rng, (m, k), "e4m3"), finite_codes(rng, (n, k), "e4m3")
    sa = rng.uniform(0.5, 2, (m, 2)).astype(F32)
    sb = rng.uniform(0.5, 2, (2, 2)).astype(F32)
    a = G.dequant_operand(qa, "e4m3", Q.expand(sa, m, k, 1, 128))
    b = G.dequant_operand(qb, "e4m3", Q.expand(sb, n, k, 128, 128))
    c, _ = G.gemm(a, b)
    av, bv = torch_decode(qa, "e4m3"), torch_decode(qb, "e4m3")
    for i in range(m):
        for j in (0, 127, 128, 129):
            ref = 0.0
            for g in range(2):
                part = sum(av[i, t] * bv[j, t] for t in range(128 * g, 128 * g + 128))
                ref += float(sa[i, g]) * float(sb[j // 128, g]) * part
            assert abs(c[i, j] - ref) <= 1e-12 * (abs(ref) + 1)


def test_sampled_matches_full():
    rng = np.random.default_rng(2)
    a = rng.standard_normal((40, 64))
    b = rng.standard_normal((50, 64))
    c, e = G.gemm(a, b)
    rows, cols = rng.integers(0, 40, 30), rng.integers(0, 50, 30)
    cs, es = G.gemm_sampled(a, b, rows, cols)
    assert np.allclose(cs, c[rows, cols], rtol=0, atol=1e-12)
    assert np.allclose(es, e[rows, cols], rtol=0, atol=1e-12)


def test_tolerance_catches_plausible_mistakes():
    x, w, _ = workloads.float8_linear(tokens=64, d_in=256, d_out=48)
    xf, wf = x.float().numpy(), w.float().numpy()
    qa, sa = Q.quantize_tensor(xf, "e4m3")
    qb, sb = Q.quantize_tensor(wf, "e4m3")
    a = G.dequant_operand(qa, "e4m3", sa)
    b = G.dequant_operand(qb, "e4m3", sb)
    c, e = G.gemm(a, b)
    # an fp32-accumulated result passes
    c32 = (a.astype(F32) @ b.astype(F32).T).astype(np.float64)
    assert G.check(c32, c, e, "f32")[0]
    # a dropped scale fails
    assert not G.check(c / float(sb), c, e, "f32")[0]
    # a sign flip fails
    assert not G.check(-c, c, e, "f32")[0]
    # a transposed operand (square case) fails
    sq = b[:48, :48]
    c2, e2 = G.gemm(a[:, :48], sq)
    wrong, _ = G.gemm(a[:, :48], sq.T)
    assert not G.check(wrong, c2, e2, "f32")[0]
    # a group scale applied to the neighbouring group fails
    sg = np.array([[1.0, 4.0]])
    ag = a[:, :256] * Q.expand(np.repeat(sg, 64, 0), 64, 256, 1, 128)
    ag_wrong = a[:, :256] * Q.expand(np.repeat(sg[:, ::-1], 64, 0), 64, 256, 1, 128)
    cg, eg = G.gemm(ag, b[:, :256])
    cw, _ = G.gemm(ag_wrong, b[:, :256])
    assert not G.check(cw, cg, eg, "f32")[0]


def test_bf16_ulp():
    assert G.bf16_ulp(1.0) == 2.0 ** -7
    assert G.bf16_ulp(1.5) == 2.0 ** -7
    assert G.bf16_ulp(-3.0) == 2.0 ** -6
    # one bf16 ulp is exactly the gap torch's bf16 grid has at that value
    v = torch.tensor([1.0, 3.0, 1000.0], dtype=torch.bfloat16)
    nxt = torch.nextafter(v, torch.tensor(float("inf"), dtype=torch.bfloat16))
    assert np.array_equal((nxt - v).double().numpy(), G.bf16_ulp(v.double().numpy()))


# ------------------------------------------------------- expert grouping --

def _expert_case(rng, offsets, n=6, k=5):
    m = offsets[-1]
    qa = finite_codes(rng, (m, k), "e4m3")
    qbs = [finite_codes(rng, (n, k), "e4m3") for _ in range(len(offsets) - 1)]
    a = torch_decode(qa, "e4m3") * 0.5
    bs = [torch_decode(q, "e4m3") * (2.0 ** -e) for e, q in enumerate(qbs)]
    return a, bs


def test_experts_exact_rational_brute_force():
    """Two tiny experts (3 and 2 rows) against a sum of exact rationals,
    written out row by row with each row's own expert."""
    rng = np.random.default_rng(21)
    offsets = [0, 3, 5]
    a, bs = _expert_case(rng, offsets)
    c, e = G.gemm_experts(a, bs, offsets)
    for ex in range(2):
        for m in range(offsets[ex], offsets[ex + 1]):
            for n in range(bs[ex].shape[0]):
                ref = sum(Fraction(float(a[m, kk])) * Fraction(float(bs[ex][n, kk]))
                          for kk in range(a.shape[1]))
                assert Fraction(float(c[m, n])) == ref
                assert e[m, n] == sum(abs(float(a[m, kk]) * float(bs[ex][n, kk]))
                                      for kk in range(a.shape[1]))


def test_one_expert_is_the_plain_product_and_empty_experts_add_nothing():
    rng = np.random.default_rng(22)
    a, bs = _expert_case(rng, [0, 7])
    c1, e1 = G.gemm_experts(a, bs, [0, 7])
    c0, e0 = G.gemm(a, bs[0])
    assert np.array_equal(c1, c0) and np.array_equal(e1, e0)
    # the same rows with empty experts before, between and after
    filler = [np.full_like(bs[0], 3.0)] * 3
    c2, _ = G.gemm_experts(a, [filler[0], bs[0], filler[1], filler[2]], [0, 0, 7, 7, 7])
    assert np.array_equal(c2, c0)


def test_experts_reordered_with_their_rows_permute_the_output():
    rng = np.random.default_rng(23)
    offsets = [0, 2, 6, 9]
    a, bs = _expert_case(rng, offsets)
    c, _ = G.gemm_experts(a, bs, offsets)
    order = [2, 0, 1]
    rows = np.concatenate([np.arange(offsets[i], offsets[i + 1]) for i in order])
    new_off = np.concatenate([[0], np.cumsum([offsets[i + 1] - offsets[i] for i in order])])
    c2, _ = G.gemm_experts(a[rows], [bs[i] for i in order], new_off)
    assert np.array_equal(c2, c[rows])


def test_swapped_expert_weights_fail_the_check():
    rng = np.random.default_rng(24)
    offsets = [0, 4, 8]
    a, bs = _expert_case(rng, offsets, n=16, k=32)
    c, e = G.gemm_experts(a, bs, offsets)
    wrong, _ = G.gemm_experts(a, bs[::-1], offsets)
    assert not G.check(wrong, c, e, "f32")[0]


# ------------------------------------------------------------ epilogue bias --

def test_bias_with_zero_operands_is_the_bias_in_every_row():
    a = np.zeros((5, 64))
    b = np.zeros((8, 64))
    bias = np.arange(8, dtype=np.float32) * np.float32(0.375) - np.float32(1.0)
    c, e = G.gemm(a, b)
    cb, eb, extra = G.gemm_bias(c, e, bias)
    assert np.array_equal(cb, np.tile(bias.astype(np.float64), (5, 1)))
    assert np.array_equal(eb, e)
    assert np.all(extra == np.abs(cb) * 2.0 ** -23)


def test_bias_along_the_wrong_axis_fails_the_check():
    rng = np.random.default_rng(25)
    a = torch_decode(finite_codes(rng, (16, 32), "e4m3"), "e4m3") * 0.25
    b = torch_decode(finite_codes(rng, (16, 32), "e4m3"), "e4m3") * 0.25
    bias = rng.standard_normal(16).astype(np.float32) * 4.0
    c, e = G.gemm(a, b)
    cb, eb, extra = G.gemm_bias(c, e, bias)
    wrong = c + bias.astype(np.float64)[:, None]
    assert not G.check(wrong, cb, eb, "f32", extra=extra)[0]
    # the fp32 rounding of the biased result is within the allowance
    assert G.check((c.astype(np.float32) + bias).astype(np.float64), cb, eb, "f32", extra=extra)[0]
