"""Scaled-FP8 GEMM over dequantized operands, in float64.

Test infrastructure only (see ``oracle/__init__``).

Whatever the granularity, the scaled-FP8 product is the plain matrix product
of the dequantized operands:

    C[m, n] = sum_k decode(qa[m, k]) * sa(m, k) * decode(qb[n, k]) * sb(n, k)

where sa(m, k) / sb(n, k) is the scale that covers element (m, k) / (n, k):

* per tensor: one scalar each; the Flax guide (section 2.2) contracts the
  codes with fp32 accumulation and multiplies by ``a_scale * b_scale``
  afterwards, which is the same sum.
* per K group (Transformers fine-grained FP8, 一): sa[m, k // 128] times
  sb[n // 128, k // 128].
* two-level (MOSS blog, section 4): S_a * r_a[m, k // 32] times
  S_b * r_b[n, k // 32].

Both operands are stored [rows, K] with K contiguous ("A row-major, B
column-major", the TN layout of the nanochat module, "核心原语").  ``b`` is
therefore [N, K], the layout of ``nn.Linear.weight``.

Alongside C the oracle returns the error budget of each element,
``E[m, n] = sum_k |a_deq[m, k]| * |b_deq[n, k]|``; an FP32-accumulated result
is accepted when ``|gpu - C| <= 1e-3 * E`` (plus one output ulp of |C| for a
bf16 output).

Mixture-of-experts grouping (Transformers fine-grained FP8, 六 6.4:
FP8Experts): token rows [offsets[e], offsets[e+1]) use expert e's weights,
so the product is the plain one per expert, ``C[rows_e] = A[rows_e] B_e^T``
(``gemm_experts``).

Pins (``tests/test_oracle_gemm.py``): exact rational brute force on tiny
shapes (products of two 8-bit floats and their short sums are exact), the
scale = 1 case against an integer matmul on the code grid, and a transposed
operand / dropped scale / sign flip each failing the check.  Expert
grouping: exact rational brute force on two tiny experts, one expert equal
to the plain product, invariance under reordering the experts with their
rows, empty experts, and swapped expert weights failing the check.  Bias:
zero operands give the bias in every row, and a bias applied along the rows
instead of the columns fails the check.
"""
from __future__ import annotations

import numpy as np

from .formats import decode


def dequant_operand(q, fmt, scale_full) -> np.ndarray:
    """decode(q) * scale, float64; ``scale_full`` broadcasts against q."""
    return decode(q, fmt) * np.asarray(scale_full, dtype=np.float64)


def gemm(a_deq, b_deq):
    """C = A @ B^T and E = |A| @ |B|^T, float64; A [M,K], B [N,K]."""
    a = np.asarray(a_deq, dtype=np.float64)
    b = np.asarray(b_deq, dtype=np.float64)
    return a @ b.T, np.abs(a) @ np.abs(b).T


def gemm_experts(a_deq, b_deq_list, offsets):
    """C and E for expert-grouped rows: rows [offsets[e], offsets[e+1]) of
    A [M, K] times expert e's B_e [N, K] (``b_deq_list[e]``), float64."""
    a = np.asarray(a_deq, dtype=np.float64)
    n = np.asarray(b_deq_list[0]).shape[0]
    c = np.zeros((a.shape[0], n))
    e_ = np.zeros((a.shape[0], n))
    for e, b in enumerate(b_deq_list):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            c[r0:r1], e_[r0:r1] = gemm(a[r0:r1], b)
    return c, e_


def gemm_bias(c, e, bias):
    """Epilogue bias (the nanochat module, "实现": Float8Linear adds the
    linear's bias to the FP8 matmul's output, y = x W^T + b): C + bias[n],
    float64, and the extra absolute allowance of one fp32 rounding of the
    biased value (2^-23 |C + b|), because the kernels add the fp32 bias to
    the fp32 result before the output cast."""
    cb = np.asarray(c, dtype=np.float64) + np.asarray(bias, dtype=np.float64)[None, :]
    return cb, np.asarray(e, dtype=np.float64), np.abs(cb) * 2.0 ** -23


def gemm_sampled(a_deq, b_deq, rows, cols):
    """C and E at the (rows[i], cols[i]) output positions only."""
    a = np.asarray(a_deq, dtype=np.float64)[np.asarray(rows)]
    b = np.asarray(b_deq, dtype=np.float64)[np.asarray(cols)]
    return np.sum(a * b, axis=1), np.sum(np.abs(a) * np.abs(b), axis=1)


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 values (8 significant bits) at |v|."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(a)
    ulp = np.ldexp(1.0, ex - 8)
    return np.where(a > 0, ulp, np.ldexp(1.0, -133))


def tolerance(c_ref, e_ref, out_dtype: str, rel: float = 1e-3, extra=0.0) -> np.ndarray:
    tol = rel * np.asarray(e_ref, dtype=np.float64) + extra
    if out_dtype == "bf16":
        tol = tol + bf16_ulp(c_ref)
    return tol


def check(c_gpu, c_ref, e_ref, out_dtype: str, rel: float = 1e-3, extra=0.0):
    """Returns (ok, worst ratio |err| / tol); ``extra`` is an additional
    absolute allowance per element (``gemm_bias``)."""
    err = np.abs(np.asarray(c_gpu, dtype=np.float64) - np.asarray(c_ref, dtype=np.float64))
    tol = tolerance(c_ref, e_ref, out_dtype, rel, extra)
    ratio = err / tol
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return bool(np.all(err <= tol)), worst
