"""The four quantization granularities of scaled-FP8 GEMM.

Test infrastructure only (see ``oracle/__init__``).

Every quantizer follows the Flax guide, section 2.2 (``quantize``):
``q = cast(clip(x / scale, -MAX, MAX))`` with the division, the clip and the
scale in fp32 (``compute_dtype = f32``), and ``scale = amax / MAX`` (section 1,
"scale = amax(x) / MAX").  Dequantization is ``decode(q) * scale`` (section 2.2
``dequantize``).  Inputs are fp32 arrays (bf16 values widen to fp32 exactly).

Granularities:

* per tensor (Flax guide 2.2, current scaling): one fp32 scale.
* per token group (Transformers fine-grained FP8, section 一): one scale per
  1 x 128 run of K in each row.
* per weight block (same section): one scale per 128 x 128 block, shape
  (ceil(N/128), ceil(K/128)).
* two-level (MOSS blog, section 4, steps 1-4): s_i = amax_i / MAX per 1 x 32
  block; global S = max_i s_i (fp32); local r_i = 2**ceil(log2(s_i / S)) in
  (0, 1] (E8M0); effective scale S * r_i.

Scale formats for the group/block granularities (Transformers section 四
``scale_fmt`` and section 七): ``"f32"`` keeps ``amax / MAX``; ``"ue8m0"``
rounds it UP to a power of two and quantizes WITH the rounded scale (section
七: rounding up without re-quantizing silently corrupts the output).

Readings where the pages are silent (each listed in the design notes):

* amax == 0 (an all-zero tensor / group / block): the scale is 1.0 (byte 127
  for UE8M0, r = 1 for two-level); the codes are zero whatever the scale.
* UE8M0 exponent: ceil(log2(s)) evaluated exactly on the fp32 value of
  ``amax / MAX``, clamped to [-127, 127].
* Ragged tails (K or N not a multiple of the group) use the valid elements
  only.

Pins (``tests/test_oracle_quantize.py``, ``tests/test_oracle_division.py``):
the quotient is a true division (inputs whose exact quotient is an FP8
rounding midpoint, where a reciprocal multiply lands on the other code,
decided by exact rational arithmetic); the amax element maps to exactly
+-MAX; hand inputs; round-trip error within half a code step times the scale;
UE8M0 bounds 2**(e-1) < s <= 2**e; the two-level invariants (S is the max of
the s_i and equals fl32(amax/MAX); every r_i is a power of two in (0, 1];
S*r_i >= s_i; no NaN codes); for the per-row global factor the same per row,
equality with the per-tensor scheme when every row holds the tensor amax,
and invariance under power-of-two row scaling.
"""
from __future__ import annotations

import numpy as np

from .formats import ceil_log2_f32, decode, e8m0_encode, encode, fmt_of

F32 = np.float32


def amax(x) -> np.float32:
    """max |x| over the whole array (exact: max is order independent)."""
    x = np.asarray(x, dtype=F32)
    if x.size == 0:
        return F32(0.0)
    return F32(np.max(np.abs(x)))


def scale_from_amax(a, fmt) -> np.ndarray:
    """Per-tensor / per-group fp32 dequant scale ``amax / MAX`` (1.0 when amax == 0)."""
    f = fmt_of(fmt)
    a = np.asarray(a, dtype=F32)
    s = (a / F32(f.max)).astype(F32)
    return np.where(a > 0, s, F32(1.0)).astype(F32)


def quantize_with_scale(x, scale, fmt) -> np.ndarray:
    """``cast(clip(x / scale, +-MAX))`` in fp32; ``scale`` broadcasts against x."""
    f = fmt_of(fmt)
    x = np.asarray(x, dtype=F32)
    s = np.asarray(scale, dtype=F32)
    with np.errstate(over="ignore"):  # x / s beyond fp32 range is inf, then clipped
        y = (x / s).astype(F32)
    y = np.clip(y, F32(-f.max), F32(f.max)).astype(F32)
    return encode(y.astype(np.float64), f)


def dequantize(q, fmt, scale) -> np.ndarray:
    return decode(q, fmt) * np.asarray(scale, dtype=np.float64)


# ---------------------------------------------------------- per tensor ----

def quantize_tensor(x, fmt):
    """Current scaling (Flax guide 2.2): returns (codes, fp32 scale)."""
    s = scale_from_amax(amax(x), fmt)
    return quantize_with_scale(x, s, fmt), F32(s)


# ----------------------------------------------------- group and block ----

def _pad_to(x, rows, cols):
    out = np.zeros((rows, cols), dtype=F32)
    out[: x.shape[0], : x.shape[1]] = x
    return out


def _scales_for(amaxes, fmt, sfmt):
    """Group amaxes -> (scale used to divide, stored scale)."""
    s = scale_from_amax(amaxes, fmt)
    if sfmt == "f32":
        return s, s
    if sfmt == "ue8m0":
        e = np.clip(ceil_log2_f32(s), -127, 127)
        e = np.where(np.asarray(amaxes) > 0, e, 0)
        return np.ldexp(F32(1.0), e).astype(F32), e8m0_encode(e)
    raise ValueError(sfmt)


def quantize_token_group(x, fmt, sfmt="f32", group=128):
    """Per-token 1 x ``group`` scaling (Transformers fine-grained FP8, 一).

    x: [M, K] fp32.  Returns codes [M, K] and scales [M, ceil(K/group)]
    (float32, or uint8 UE8M0 bytes).
    """
    x = np.asarray(x, dtype=F32)
    m, k = x.shape
    g = -(-k // group)
    xp = _pad_to(x, m, g * group).reshape(m, g, group)
    am = np.max(np.abs(xp), axis=2).astype(F32)
    div, stored = _scales_for(am, fmt, sfmt)
    full = np.repeat(div, group, axis=1)[:, :k]
    return quantize_with_scale(x, full, fmt), stored


def quantize_block(w, fmt, sfmt="f32", block=128):
    """128 x 128 weight-block scaling (Transformers fine-grained FP8, 一).

    w: [N, K] fp32.  Returns codes [N, K] and scales
    [ceil(N/block), ceil(K/block)].
    """
    w = np.asarray(w, dtype=F32)
    n, k = w.shape
    bn, bk = -(-n // block), -(-k // block)
    wp = _pad_to(w, bn * block, bk * block).reshape(bn, block, bk, block)
    am = np.max(np.abs(wp), axis=(1, 3)).astype(F32)
    div, stored = _scales_for(am, fmt, sfmt)
    full = np.repeat(np.repeat(div, block, axis=0), block, axis=1)[:n, :k]
    return quantize_with_scale(w, full, fmt), stored


def group_scale_values(stored, sfmt) -> np.ndarray:
    """Stored group/block scales -> float64 multipliers."""
    if sfmt == "f32":
        return np.asarray(stored, dtype=np.float64)
    b = np.asarray(stored, dtype=np.int64)
    return np.ldexp(1.0, b - 127)


# ---------------------------------------------------------- two level ----

def quantize_two_level(x, fmt, block=32, global_per_row=False):
    """MOSS two-level microscaling (MOSS blog, section 4, steps 1-4).

    x: [R, K] fp32 with K % block == 0.  Returns (codes [R,K], local E8M0 bytes
    [R, K/block], global fp32 S).  ``global_per_row``: the global factor of
    step 2 is taken over each row's blocks instead of the whole tensor (the
    garbled extent of the page's "整个 _ 范围" read per row); S is then an
    fp32 array [R] and each row's local factors are relative to its own S.
    """
    f = fmt_of(fmt)
    x = np.asarray(x, dtype=F32)
    r, k = x.shape
    if k % block:
        raise ValueError("two-level: K must be a multiple of the block")
    xb = x.reshape(r, k // block, block)
    am = np.max(np.abs(xb), axis=2).astype(F32) if x.size else np.zeros((r, 0), F32)
    s_i = (am / F32(f.max)).astype(F32)                     # step 1
    if global_per_row:                                      # step 2, per row
        big_s = (np.max(s_i, axis=1) if s_i.size else np.zeros(r)).astype(F32)
        big_s = np.where(big_s > 0, big_s, F32(1.0)).astype(F32)
        ratio = (s_i / big_s[:, None]).astype(F32)          # step 3
        e = np.where(s_i > 0, -127, 0).astype(np.int64)
        pos = ratio > 0
        if np.any(pos):
            e[pos] = np.maximum(ceil_log2_f32(ratio[pos]), -127)
        r_i = np.ldexp(F32(1.0), e).astype(F32)
        eff = (big_s[:, None] * r_i).astype(F32)            # step 4
        q = quantize_with_scale(x, np.repeat(eff, block, axis=1), f)
        return q, e8m0_encode(e), big_s
    big_s = F32(np.max(s_i)) if s_i.size else F32(0.0)      # step 2
    if not big_s > 0:
        big_s = F32(1.0)
    ratio = (s_i / big_s).astype(F32)                       # step 3
    # all-zero block: r = 1; a positive block whose ratio underflows: 2^-127
    e = np.where(s_i > 0, -127, 0).astype(np.int64)
    pos = ratio > 0
    if np.any(pos):
        e[pos] = np.maximum(ceil_log2_f32(ratio[pos]), -127)
    r_i = np.ldexp(F32(1.0), e).astype(F32)
    eff = (big_s * r_i).astype(F32)                         # step 4
    full = np.repeat(eff, block, axis=1)
    q = quantize_with_scale(x, full, f)
    return q, e8m0_encode(e), big_s


def quantize_mxfp8(x, fmt, block=32):
    """One-level microscaling (MOSS blog, section 1): every 32 consecutive
    values along K share one power-of-two scale, the smallest power of two not
    below amax_block / MAX, and the block is divided by it.

    x: [R, K] fp32, K % block == 0.  Returns (codes [R,K], E8M0 bytes
    [R, K/block]).  An all-zero block takes scale 1 (byte 127); exponents are
    clamped to [-127, 127].
    """
    f = fmt_of(fmt)
    x = np.asarray(x, dtype=F32)
    r, k = x.shape
    if k % block:
        raise ValueError("mxfp8: K must be a multiple of the block")
    xb = x.reshape(r, k // block, block)
    am = np.max(np.abs(xb), axis=2).astype(F32) if x.size else np.zeros((r, 0), F32)
    s_i = (am / F32(f.max)).astype(F32)
    e = np.zeros(s_i.shape, dtype=np.int64)
    pos = s_i > 0
    if np.any(pos):
        e[pos] = np.clip(ceil_log2_f32(s_i[pos]), -127, 127)
    scale = np.ldexp(F32(1.0), e).astype(F32)
    q = quantize_with_scale(x, np.repeat(scale, block, axis=1), f)
    return q, e8m0_encode(e)


def dequantize_block(q, fmt, scales, sfmt, block=128):
    """Fold 128x128 block scales into the values (Transformers fine-grained
    FP8, 五: dequantize=True turns the FP8 weights back into bf16): the
    definition decode(q) * scale of the element's block, float64."""
    q = np.asarray(q)
    n, k = q.shape
    return decode(q, fmt) * expand(group_scale_values(scales, sfmt), n, k, block, block)


def two_level_scale_values(local_bytes, global_s) -> np.ndarray:
    """Effective per-block multipliers S * r_i (float64); ``global_s`` is a
    scalar or, for the per-row variant, one factor per row."""
    b = np.asarray(local_bytes, dtype=np.int64)
    g = np.asarray(global_s, dtype=np.float64)
    if g.ndim == 1:
        g = g[:, None]
    return g * np.ldexp(1.0, b - 127)


def expand(scales, rows, cols, row_block, col_block) -> np.ndarray:
    """Broadcast a block-scale grid to the full [rows, cols] element grid."""
    s = np.asarray(scales, dtype=np.float64)
    s = np.repeat(np.repeat(s, row_block, axis=0), col_block, axis=1)
    return s[:rows, :cols]
