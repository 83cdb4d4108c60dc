"""Pins for the oracle's quantizers (oracle/quantize.py).

Evidence independent of the oracle's own code: hand encodings, torch's float8
cast (a library routine) applied to values scaled by an exact power of two,
the defining property that the amax element lands on +-MAX, and the MOSS
two-level invariants.
"""
import numpy as np
import pytest
import torch

import workloads
from golden.fixtures import load
from oracle import formats as F
from oracle import quantize as Q

CONST = load("format_constants.txt")
F32 = np.float32


def torch_cast(vals_f32, name):
    dt = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}[name]
    return torch.tensor(np.asarray(vals_f32, dtype=F32)).to(dt).view(torch.uint8).numpy()


def test_hand_per_tensor():
    # amax 448 -> scale exactly 1.0 -> 1.0, -448, 0.5 encode as by hand
    q, s = Q.quantize_tensor(np.array([1.0, -448.0, 0.5], F32), "e4m3")
    assert s == 1.0 and list(q) == [0x38, 0xFE, 0x30]
    # amax 7 -> scale 7/448 = 1/64 -> 3.5 * 64 = 224 = 0.1110.110
    q, s = Q.quantize_tensor(np.array([3.5, -7.0, 0.0], F32), "e4m3")
    assert s == 1.0 / 64 and list(q) == [0x76, 0xFE, 0x00]
    # E5M2 gradient: amax 57344 * 2 -> scale 2 -> 1.0 encodes as 0.01111.00
    q, s = Q.quantize_tensor(np.array([2.0, -114688.0], F32), "e5m2")
    assert s == 2.0 and list(q) == [0x3C, 0xFB]


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_amax_element_hits_max(name):
    x = workloads.normal((64, 96), 3.0, seed=11).numpy()
    q, s = Q.quantize_tensor(x, name)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(F.decode(q[i], name)) == F.fmt_of(name).max
    assert np.all(np.isfinite(F.decode(q, name)))


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_roundtrip_within_half_step(name):
    f = F.fmt_of(name)
    x = workloads.normal((128, 64), 1.0, seed=5).numpy()
    q, s = Q.quantize_tensor(x, name)
    y = np.abs(x.astype(np.float64) / float(s))
    e = np.maximum(np.floor(np.log2(np.maximum(y, 1e-300))), f.min_normal_exp)
    half_step = np.ldexp(0.5, (e - f.mbits).astype(int)) * float(s)
    err = np.abs(Q.dequantize(q, name, s) - x)
    assert np.all(err <= half_step * (1 + 1e-6) + 1e-30)


def test_zero_and_signed_zero():
    q, s = Q.quantize_tensor(np.zeros((4, 4), F32), "e4m3")
    assert s == 1.0 and not q.any()
    q, s = Q.quantize_tensor(np.array([-0.0, 1.0], F32), "e4m3")
    assert q[0] == 0x80


def test_empty_tensor_reading():
    """Reading R4 extended to zero elements: the amax of nothing is 0 (the
    identity of max over magnitudes), so the scale is 1.0 and there are no
    codes; a planted mistake (amax of nothing taken as 1) would give a scale
    of 1/448 and fails here."""
    x = np.zeros((0,), F32)
    assert Q.amax(x) == 0.0
    q, s = Q.quantize_tensor(x, "e5m2")
    assert s == F32(1.0) and q.size == 0
    assert Q.scale_from_amax(F32(1.0), "e4m3") != F32(1.0)  # the planted mistake differs


def test_pow2_scale_matches_library_cast():
    # with a power-of-two scale the division is exact, so quantization is
    # torch's cast of x * 2^-e (clipped): independent of the oracle's division
    x = workloads.normal((33, 130), 10.0, seed=9).numpy()
    for e in (-3, 0, 4):
        q = Q.quantize_with_scale(x, F32(2.0 ** e), "e4m3")
        ref = torch_cast(np.clip(x * F32(2.0 ** -e), -448, 448), "e4m3")
        assert np.array_equal(q, ref)


def _group_views(x, q, rows, cols):
    for r0 in range(0, x.shape[0], rows):
        for c0 in range(0, x.shape[1], cols):
            yield (r0 // rows, c0 // cols), x[r0:r0 + rows, c0:c0 + cols], q[r0:r0 + rows, c0:c0 + cols]


@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_token_group_properties(sfmt):
    x = workloads.normal((5, 300), 1.0, seed=21).numpy()   # ragged last group (44 wide)
    x[2, 130] = 80.0                                     # outlier in one group only
    x[3, 128:256] = 0.0                                  # an all-zero group
    q, sc = Q.quantize_token_group(x, "e4m3", sfmt)
    assert sc.shape == (5, 3)
    vals = Q.group_scale_values(sc, sfmt)
    for (i, j), xg, qg in _group_views(x, q, 1, 128):
        am = float(np.max(np.abs(xg)))
        mag = np.max(np.abs(F.decode(qg, "e4m3")))
        if am == 0:
            assert vals[i, j] == 1.0 and not qg.any()
            continue
        if sfmt == "f32":
            assert vals[i, j] == np.float32(np.float32(am) / np.float32(448.0))
            assert mag == 448.0
        else:
            e = int(np.log2(vals[i, j]))
            assert vals[i, j] == 2.0 ** e
            assert 2.0 ** (e - 1) < am / 448.0 <= 2.0 ** e * (1 + 2 ** -23)
            assert 224.0 <= mag <= 448.0
            assert np.array_equal(qg, torch_cast(np.clip(xg * F32(2.0 ** -e), -448, 448), "e4m3"))
    # the outlier only moves its own group's scale
    x2 = x.copy()
    x2[2, 130] = 1.0
    q2, sc2 = Q.quantize_token_group(x2, "e4m3", sfmt)
    diff = np.argwhere(np.asarray(sc) != np.asarray(sc2))
    assert [tuple(d) for d in diff] == [(2, 1)]


@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_block_properties_and_transpose(sfmt):
    w = workloads.normal((200, 260), 0.02, seed=22).numpy()   # ragged in both dims
    q, sc = Q.quantize_block(w, "e4m3", sfmt)
    assert sc.shape == (2, 3)
    vals = Q.group_scale_values(sc, sfmt)
    for (i, j), wb, qb in _group_views(w, q, 128, 128):
        am = np.float32(np.max(np.abs(wb)))
        if sfmt == "f32":
            assert vals[i, j] == np.float32(am / np.float32(448.0))
            assert np.max(np.abs(F.decode(qb, "e4m3"))) == 448.0
        else:
            assert 224.0 <= np.max(np.abs(F.decode(qb, "e4m3"))) <= 448.0
    qt, sct = Q.quantize_block(w.T.copy(), "e4m3", sfmt)
    assert np.array_equal(qt, q.T) and np.array_equal(np.asarray(sct), np.asarray(sc).T)


def test_two_level_invariants():
    a, _ = workloads.two_level(m=64, n=8, k=512)
    x = a.float().numpy()
    q, local, big_s = Q.quantize_two_level(x, "e4m3")
    assert local.shape == (64, 16)
    s_i = (np.max(np.abs(x.reshape(64, 16, 32)), axis=2) / F32(448)).astype(F32)
    # global factor = max of the 1x32 fp32 scales = fl32(tensor amax / MAX)
    assert big_s == np.max(s_i) == np.float32(np.float32(np.max(np.abs(x))) / F32(448))
    r = F.e8m0_decode(local)
    assert np.all((r > 0) & (r <= 1))
    assert np.all(np.log2(r) == np.round(np.log2(r)))
    assert np.all(float(big_s) * r >= s_i.astype(np.float64))
    # r is the smallest such power of two
    assert np.all(float(big_s) * r / 2 < s_i.astype(np.float64))
    d = F.decode(q, "e4m3")
    assert np.all(np.isfinite(d)) and np.max(np.abs(d)) <= 448.0
    y = x.reshape(64, 16, 32) / (float(big_s) * r)[:, :, None]
    assert np.max(np.abs(y)) <= 448.0 * (1 + 2 ** -22)


def test_two_level_reduces_to_per_tensor():
    # equal block amaxes -> every r_i = 1 -> per-tensor quantization
    x = workloads.normal((4, 128), 1.0, seed=31).numpy()
    x.reshape(4, 4, 32)[:, :, 0] = 5.0
    q, local, big_s = Q.quantize_two_level(x, "e4m3")
    assert np.all(local == 127)
    qt, st = Q.quantize_tensor(x, "e4m3")
    assert big_s == st and np.array_equal(q, qt)


def test_two_level_rescues_small_blocks():
    # half the 1x32 blocks are 2^-16 smaller: per-tensor scaling pushes them into
    # E4M3 subnormals, the E8M0 local factors lift them back into the normal range
    from oracle.snr import snr_db
    x = workloads.normal((64, 256), 1.0, seed=41).numpy()
    xb = x.reshape(64, 8, 32)
    xb[:, 1::2, :] *= np.float32(2.0 ** -16)
    q2, l2, s2 = Q.quantize_two_level(x, "e4m3")
    d2 = F.decode(q2, "e4m3") * Q.expand(Q.two_level_scale_values(l2, float(s2)), 64, 256, 1, 32)
    qt, st = Q.quantize_tensor(x, "e4m3")
    dt = Q.dequantize(qt, "e4m3", st)
    small = np.zeros_like(xb, dtype=bool)
    small[:, 1::2, :] = True
    small = small.reshape(64, 256)
    assert snr_db(x[small], d2[small]) > snr_db(x[small], dt[small]) + 20.0
    # on the large blocks both schemes agree exactly
    assert np.array_equal(d2[~small], dt[~small])


def test_mxfp8_one_level_properties():
    # MOSS blog, section 1: a power-of-two scale per 32 values from the block amax
    x = workloads.normal((6, 256), 1.0, seed=51).numpy()
    x[1, 32:64] = 0.0
    x[2, :32] *= 1e4
    q, b = Q.quantize_mxfp8(x, "e4m3")
    assert b.shape == (6, 8)
    for i in range(6):
        for j in range(8):
            xb = x[i, 32 * j:32 * j + 32]
            e = int(b[i, j]) - 127
            am = float(np.max(np.abs(xb)))
            if am == 0:
                assert e == 0 and not q[i, 32 * j:32 * j + 32].any()
                continue
            s_i = float(np.float32(np.float32(am) / np.float32(448.0)))
            assert 2.0 ** (e - 1) < s_i <= 2.0 ** e
            mag = np.max(np.abs(F.decode(q[i, 32 * j:32 * j + 32], "e4m3")))
            assert 224.0 <= mag <= 448.0
            ref = torch_cast(np.clip(xb * np.float32(2.0 ** -e), -448, 448), "e4m3")
            assert np.array_equal(q[i, 32 * j:32 * j + 32], ref)


def test_mxfp8_equals_two_level_with_unit_global():
    # with every block amax a power of two times 448 the two schemes coincide
    x = workloads.normal((4, 128), 1.0, seed=52).numpy()
    xb = x.reshape(4, 4, 32)
    xb[:] = np.clip(xb, -1, 1)
    xb[:, :, 0] = 448.0 * 2.0 ** -np.arange(4)[None, :]
    q1, b1 = Q.quantize_mxfp8(x, "e4m3")
    q2, b2, s2 = Q.quantize_two_level(x, "e4m3")
    assert s2 == 1.0
    assert np.array_equal(q1, q2) and np.array_equal(b1, b2)


@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_dequantize_block_roundtrip(sfmt):
    w = workloads.normal((200, 260), 0.02, seed=53).numpy()
    q, sc = Q.quantize_block(w, "e4m3", sfmt)
    d = Q.dequantize_block(q, "e4m3", sc, sfmt)
    vals = Q.group_scale_values(sc, sfmt)
    lib = torch.tensor(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(d, lib * Q.expand(vals, 200, 260, 128, 128))
    # within half an E4M3 step (1/16 relative) of the original, blockwise
    assert np.all(np.abs(d - w) <= np.abs(w) / 16 + Q.expand(vals, 200, 260, 128, 128) * 2.0 ** -10)


def test_two_level_per_row_global_invariants():
    """Per-row global factors: S_r is the max of row r's 1x32 scales (which
    is fl32(row amax / MAX)); every r_i is a power of two in (0, 1] and the
    smallest with S_r * r_i >= s_i."""
    a, _ = workloads.two_level(m=48, n=8, k=512)
    x = a.float().numpy()
    x[5] *= np.float32(2.0 ** -20)          # one row far smaller than the rest
    q, local, big_s = Q.quantize_two_level(x, "e4m3", global_per_row=True)
    assert big_s.shape == (48,)
    s_i = (np.max(np.abs(x.reshape(48, 16, 32)), axis=2) / F32(448)).astype(F32)
    assert np.array_equal(big_s, np.max(s_i, axis=1))
    row_amax = np.max(np.abs(x), axis=1).astype(F32)
    assert np.array_equal(big_s, (row_amax / F32(448)).astype(F32))
    r = F.e8m0_decode(local)
    assert np.all((r > 0) & (r <= 1)) and np.all(np.log2(r) == np.round(np.log2(r)))
    s = big_s.astype(np.float64)[:, None]
    assert np.all(s * r >= s_i) and np.all(s * r / 2 < s_i)
    # each row's block holding the row amax has r = 1 and codes reaching MAX
    assert np.all(np.max(local, axis=1) == 127)
    assert np.all(np.max(np.abs(F.decode(q, "e4m3")), axis=1) == 448.0)


def test_two_level_per_row_equals_per_tensor_when_rows_share_the_max():
    x = workloads.normal((6, 256), 1.0, seed=33).numpy()
    x[:, 17] = 9.0                          # every row holds the tensor amax
    q1, l1, s1 = Q.quantize_two_level(x, "e4m3")
    q2, l2, s2 = Q.quantize_two_level(x, "e4m3", global_per_row=True)
    assert np.all(s2 == s1) and np.array_equal(l1, l2) and np.array_equal(q1, q2)


def test_two_level_per_row_is_row_scale_invariant():
    """Rows that are power-of-two multiples of one row get the same codes and
    local factors, and global factors in the same ratio."""
    base = workloads.normal((1, 256), 1.0, seed=35).numpy()
    x = np.concatenate([base * np.float32(2.0 ** e) for e in (-12, -3, 0, 7)])
    q, local, big_s = Q.quantize_two_level(x, "e4m3", global_per_row=True)
    for i in range(1, 4):
        assert np.array_equal(q[i], q[0]) and np.array_equal(local[i], local[0])
    assert np.array_equal(big_s / big_s[2], np.float32([2.0 ** -12, 2.0 ** -3, 1.0, 2.0 ** 7]))


def test_block_32x32_ue8m0_brute_force():
    """(32, 32) weight blocks (Transformers fine-grained FP8, 八: a non-default
    weight_block_size) with UE8M0 scales, against a loop over the blocks: each
    block's byte is 127 + ceil(log2(fl32(block amax / 448))) (127 for an
    all-zero block) and its codes are the block divided by that power of
    two, with ragged edge blocks."""
    w = workloads.normal((70, 96), 0.02, seed=37).numpy()
    w[32:64, 32:64] = 0.0
    w[5, 70] = 3.0
    q, sc = Q.quantize_block(w, "e4m3", "ue8m0", block=32)
    assert np.asarray(sc).shape == (3, 3)
    for bi in range(3):
        for bj in range(3):
            blk = w[32 * bi:32 * bi + 32, 32 * bj:32 * bj + 32]
            am = np.float32(np.max(np.abs(blk)))
            if am == 0:
                e = 0
            else:
                s = np.float32(am / np.float32(448.0))
                e = int(np.ceil(np.log2(np.float64(s))))
                assert 2.0 ** (e - 1) < s <= 2.0 ** e
            assert int(np.asarray(sc)[bi, bj]) == 127 + e
            ref = Q.quantize_with_scale(blk, np.float32(2.0 ** e), "e4m3")
            assert np.array_equal(q[32 * bi:32 * bi + 32, 32 * bj:32 * bj + 32], ref)


def test_block_32x32_f32_brute_force():
    """(32, 32) weight blocks with FP32 scales (Transformers fine-grained FP8,
    八: weight_block_size (32, 32); 四: scale_fmt float, the default), against
    a loop over the blocks: each scale is fl32(block amax / 448) (1.0 for an
    all-zero block), each block's largest element lands exactly on +-448, and
    its codes are the block divided by its own scale; ragged edge blocks."""
    w = workloads.normal((70, 96), 0.02, seed=41).numpy()
    w[32:64, 32:64] = 0.0
    w[5, 70] = -3.0
    q, sc = Q.quantize_block(w, "e4m3", "f32", block=32)
    sc = np.asarray(sc)
    assert sc.shape == (3, 3) and sc.dtype == np.float32
    for bi in range(3):
        for bj in range(3):
            blk = w[32 * bi:32 * bi + 32, 32 * bj:32 * bj + 32]
            qb = q[32 * bi:32 * bi + 32, 32 * bj:32 * bj + 32]
            am = np.float32(np.max(np.abs(blk)))
            if am == 0:
                assert sc[bi, bj] == 1.0 and not qb.any()
                continue
            assert sc[bi, bj] == np.float32(am / np.float32(448.0))
            assert np.array_equal(qb, Q.quantize_with_scale(blk, sc[bi, bj], "e4m3"))
            assert np.max(np.abs(F.decode(qb, "e4m3"))) == 448.0
    # a block's outlier moves only that block's scale
    w2 = w.copy()
    w2[5, 70] = 0.01
    _, sc2 = Q.quantize_block(w2, "e4m3", "f32", block=32)
    assert [tuple(d) for d in np.argwhere(np.asarray(sc2) != sc)] == [(0, 2)]


def test_token_group_1x32_f32_brute_force():
    """1 x 32 activation groups with FP32 scales, the activation side of
    (32, 32) weight blocks (Transformers fine-grained FP8, 八: the activation
    group follows the block's K size): per row and 32-wide group, scale
    fl32(amax / 448) (1.0 for a zero group), codes of the group divided by it."""
    x = workloads.normal((6, 96), 1.0, seed=42).numpy()
    x[1, 32:64] = 0.0
    x[4, 3] = 200.0
    q, sc = Q.quantize_token_group(x, "e4m3", "f32", group=32)
    sc = np.asarray(sc)
    assert sc.shape == (6, 3)
    for r in range(6):
        for g in range(3):
            xg = x[r, 32 * g:32 * g + 32]
            am = np.float32(np.max(np.abs(xg)))
            want_s = np.float32(am / np.float32(448.0)) if am > 0 else np.float32(1.0)
            assert sc[r, g] == want_s
            assert np.array_equal(q[r, 32 * g:32 * g + 32],
                                  Q.quantize_with_scale(xg, want_s, "e4m3"))
