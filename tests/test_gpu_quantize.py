"""GPU parity of the quantization kernels against the CPU oracle.

Quantized bytes and scales must match bit for bit (the kernel and the oracle
both take the fp32 x / s decision, then round to nearest even)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import FMT, f32_bits, lib, mx_pack, mx_unpack, to_np_u8
from oracle import delayed as OD
from oracle import quantize as OQ

pytestmark = pytest.mark.gpu


def special_input(shape, std, seed, dtype, fmt):
    """Normal draws plus hand-placed edge values: zeros, -0.0, tiny values that
    land in the FP8 subnormal range, and the element that sets the amax."""
    x = workloads.normal(shape, std, seed)
    flat = x.view(-1)
    n = flat.numel()
    if n >= 8:
        flat[0] = 0.0
        flat[1] = -0.0
        flat[2] = std * 1e-3
        flat[3] = -std * 3e-4
        flat[n // 2] = std * 7.0
        flat[n - 1] = -std * 6.5
    return x.to(dtype)


SHAPES = [(1, 8), (7, 24), (128, 128), (300, 520), (513, 1032)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("transpose", [False, True])
def test_current_scaling(shape, fmt, dt, transpose):
    F = lib()
    std = 1.0 if fmt == "e4m3" else 1e-3
    x = special_input(shape, std, 10 + shape[0], dt, fmt)
    xf = x.float().numpy()
    xd = x.cuda()
    amax = torch.empty(1, device="cuda")
    F.fp8_amax(xd, amax)
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    qt = torch.empty((shape[1], shape[0]), dtype=torch.uint8, device="cuda") if transpose else None
    s_out = torch.empty(1, device="cuda")
    F.fp8_quantize_tensor(xd, FMT[fmt], q, amax_in=amax, scale_out=s_out, q_t=qt)
    ref_q, ref_s = OQ.quantize_tensor(xf, fmt)
    assert f32_bits(amax.item()) == f32_bits(OQ.amax(xf))
    assert f32_bits(s_out.item()) == f32_bits(ref_s)
    assert np.array_equal(to_np_u8(q), ref_q)
    if transpose:
        assert np.array_equal(to_np_u8(qt), ref_q.T)


@pytest.mark.parametrize("shape", [(64, 96), (257, 136)])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_given_scale_with_clip_and_fused_amax(shape, fmt):
    F = lib()
    x = special_input(shape, 1.0, 77, torch.bfloat16, fmt)
    xf = x.float().numpy()
    # a scale small enough that the largest values clip at +-MAX
    from oracle.formats import fmt_of
    scale = np.float32(np.float32(OQ.amax(xf)) / np.float32(fmt_of(fmt).max) / np.float32(3.0))
    sd = torch.tensor([float(scale)], dtype=torch.float32, device="cuda")
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    qt = torch.empty((shape[1], shape[0]), dtype=torch.uint8, device="cuda")
    amax_out = torch.full((1,), 123.0, device="cuda")
    F.fp8_quantize_tensor(x.cuda(), FMT[fmt], q, scale=sd, q_t=qt, amax_out=amax_out)
    ref = OQ.quantize_with_scale(xf, scale, fmt)
    assert np.array_equal(to_np_u8(q), ref)
    assert np.array_equal(to_np_u8(qt), ref.T)
    assert f32_bits(amax_out.item()) == f32_bits(OQ.amax(xf))


def test_amax_sizes_and_zero():
    F = lib()
    for n in (1, 7, 8, 1000, 1 << 20):
        x = workloads.normal((n,), 2.0, n)
        out = torch.empty(1, device="cuda")
        F.fp8_amax(x.cuda(), out)
        assert out.item() == float(np.max(np.abs(x.numpy())))
    z = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    out = torch.full((1,), 5.0, device="cuda")
    F.fp8_amax(z, out)
    assert out.item() == 0.0
    q = torch.empty((64, 64), dtype=torch.uint8, device="cuda")
    s = torch.empty(1, device="cuda")
    F.fp8_quantize_tensor(z.view(64, 64), 0, q, amax_in=out, scale_out=s)
    assert s.item() == 1.0 and not q.any()


@pytest.mark.parametrize("shape", [(1, 128), (5, 304), (130, 1024), (64, 7168)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_token_group(shape, sfmt, dt):
    F = lib()
    m, k = shape
    act, _ = workloads.fine_grained(m, k=k, n=128)
    x = act.to(dt)
    if m > 2:
        x[2, : min(128, k)] = 0.0  # an all-zero group
    xf = x.float().numpy()
    g = (k + 127) // 128
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    sc = torch.empty((g, m), dtype=torch.float32 if sfmt == "f32" else torch.uint8, device="cuda")
    F.fp8_quantize_token_group(x.cuda(), 0, 0 if sfmt == "f32" else 1, q, sc)
    ref_q, ref_s = OQ.quantize_token_group(xf, "e4m3", sfmt)
    assert np.array_equal(to_np_u8(q), ref_q)
    got = sc.cpu().numpy().T
    if sfmt == "f32":
        assert np.array_equal(got.view(np.uint32), np.asarray(ref_s, np.float32).view(np.uint32))
    else:
        assert np.array_equal(got, ref_s)


@pytest.mark.parametrize("shape", [(200, 272), (256, 512), (2048, 7168)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_block(shape, sfmt):
    F = lib()
    n, k = shape
    _, w = workloads.fine_grained(1, k=k, n=n)
    wf = w.float().numpy()
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    bn, bk = (n + 127) // 128, (k + 127) // 128
    sc = torch.empty((bn, bk), dtype=torch.float32 if sfmt == "f32" else torch.uint8, device="cuda")
    F.fp8_quantize_block(w.cuda(), 0, 0 if sfmt == "f32" else 1, q, sc)
    ref_q, ref_s = OQ.quantize_block(wf, "e4m3", sfmt)
    assert np.array_equal(to_np_u8(q), ref_q)
    got = sc.cpu().numpy()
    if sfmt == "f32":
        assert np.array_equal(got.view(np.uint32), np.asarray(ref_s, np.float32).view(np.uint32))
    else:
        assert np.array_equal(got, ref_s)


@pytest.mark.parametrize("shape", [(1, 128), (130, 512), (256, 1024), (333, 2048)])
def test_two_level(shape):
    F = lib()
    r, k = shape
    a, _ = workloads.two_level(m=r, n=8, k=k)
    x = a.clone()
    x[0, 32:64] = 0.0  # an all-zero 1x32 block
    xf = x.float().numpy()
    xd = x.cuda()
    amax = torch.empty(1, device="cuda")
    F.fp8_amax(xd, amax)
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    words = F.mx_local_words(r, k)
    words.fill_(0)
    glob = torch.empty(1, device="cuda")
    F.fp8_quantize_mx(xd, 0, amax, glob, q, words)
    ref_q, ref_l, ref_s = OQ.quantize_two_level(xf, "e4m3")
    assert f32_bits(glob.item()) == f32_bits(ref_s)
    assert np.array_equal(to_np_u8(q), ref_q)
    w = words.cpu().numpy()
    assert np.array_equal(mx_unpack(w, r, k), ref_l)
    rpad = (r + 127) // 128 * 128
    if rpad > r:  # padding rows hold factor 1
        rows = np.arange(r, rpad)
        pos = (rows & ~127) + 4 * (rows % 32) + (rows % 128) // 32
        assert np.all(w.view(np.uint32)[:, pos] == 0x7F7F7F7F)


@pytest.mark.parametrize("length", [4, 1024])
def test_delayed_scaling_sequence(length):
    """GPU quantize + fp8_delayed_state_update over 20 steps against the
    guide's in_q order (scale from the previous history, then push)."""
    F = lib()
    hist = torch.zeros(length, device="cuda")
    scale = torch.ones(1, device="cuda")
    amax_cur = torch.empty(1, device="cuda")
    st = OD.DelayedState.initial(length)
    for t in range(20):
        x = workloads.normal((64, 128), 2.0 ** ((t * 3) % 11 - 5), 500 + t).to(torch.bfloat16)
        if t == 4:
            x.zero_()
        xf = x.float().numpy()
        q = torch.empty((64, 128), dtype=torch.uint8, device="cuda")
        used = scale.item()
        F.fp8_quantize_tensor(x.cuda(), 0, q, scale=scale, amax_out=amax_cur)
        F.fp8_delayed_state_update(hist, scale, amax_cur, 0)
        ref_q, ref_scale, st = OD.in_q(xf, "e4m3", st)
        assert f32_bits(used) == f32_bits(ref_scale), t
        assert np.array_equal(to_np_u8(q), ref_q), t
        assert np.array_equal(hist.cpu().numpy().view(np.uint32), st.history.view(np.uint32)), t


def test_delayed_state_update_multi_matches_the_oracle():
    """Nine histories (different lengths, both formats, one amax shared by
    two items, a zero and a NaN amax) in one launch over 12 steps: every
    history and scale bit-exact against the oracle's in_q order."""
    F = lib()
    lengths = [1024, 1024, 16, 1, 1024, 300, 1024, 7, 1024]
    fmts = ["e4m3", "e4m3", "e5m2", "e4m3", "e5m2", "e5m2", "e4m3", "e5m2", "e4m3"]
    code = {"e4m3": F.E4M3, "e5m2": F.E5M2}
    hist = [torch.zeros(n, device="cuda") for n in lengths]
    scale = torch.ones(len(lengths), device="cuda")
    amax = torch.zeros(len(lengths), device="cuda")
    src = [i if i != 1 else 0 for i in range(len(lengths))]  # item 1 reads item 0's amax
    states = [OD.DelayedState.initial(n) for n in lengths]
    items = [F.delayed_item(hist[i], scale[i:i + 1], amax[src[i]:src[i] + 1], code[fmts[i]])
             for i in range(len(lengths))]
    rng = np.random.default_rng(9)
    for t in range(12):
        cur = (rng.random(len(lengths)) * 10.0 ** rng.integers(-3, 4, len(lengths))).astype(np.float32)
        cur[2] = 0.0 if t == 3 else cur[2]
        cur[5] = np.nan if t == 5 else cur[5]
        amax.copy_(torch.from_numpy(cur))
        F.fp8_delayed_state_update_multi(items)
        torch.cuda.synchronize()
        for i, st in enumerate(states):
            # the push, then the scale the next step uses (the order in which
            # the oracle's in_q meets them)
            h = OD.compute_amax_history(np.float32(cur[src[i]]), st.history)
            states[i] = OD.DelayedState(h, OD.compute_scale(np.max(h), st.scale, fmts[i]))
            assert np.array_equal(hist[i].cpu().numpy().view(np.uint32),
                                  states[i].history.view(np.uint32)), (t, i)
            assert f32_bits(scale[i].item()) == f32_bits(states[i].scale), (t, i)


def test_delayed_update_keeps_scale_on_nonfinite():
    F = lib()
    hist = torch.zeros(8, device="cuda")
    hist[3] = float("inf")
    scale = torch.tensor([0.5], device="cuda")
    F.fp8_delayed_state_update(hist, scale, torch.tensor([2.0], device="cuda"), 0)
    assert scale.item() == 0.5
    hist[:] = 0.0
    hist[5] = float("nan")
    F.fp8_delayed_state_update(hist, scale, torch.tensor([2.0], device="cuda"), 0)
    assert scale.item() == 0.5
    hist[:] = 0.0
    F.fp8_delayed_state_update(hist, scale, torch.tensor([0.0], device="cuda"), 1)
    assert scale.item() == 0.5
    F.fp8_delayed_state_update(hist, scale, torch.tensor([57344.0 * 4], device="cuda"), 1)
    assert scale.item() == 4.0


@pytest.mark.parametrize("shape", [(1, 128), (130, 512), (333, 2048)])
def test_mxfp8_one_level(shape):
    F = lib()
    r, k = shape
    a, _ = workloads.two_level(m=r, n=8, k=k)
    x = a.clone()
    x[0, 32:64] = 0.0
    xf = x.float().numpy()
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    words = F.mx_local_words(r, k)
    glob = torch.zeros(1, device="cuda")
    F.fp8_quantize_mx1(x.cuda(), 0, glob, q, words)
    ref_q, ref_l = OQ.quantize_mxfp8(xf, "e4m3")
    assert glob.item() == 1.0
    assert np.array_equal(to_np_u8(q), ref_q)
    assert np.array_equal(mx_unpack(words.cpu().numpy(), r, k), ref_l)


@pytest.mark.parametrize("shape", [(32, 128), (200, 384), (2048, 7168)])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
def test_quantize_block32(shape, fmt, in_dtype):
    """(32, 32) UE8M0 weight blocks: codes and block bytes bit-exact against
    the oracle; the MX words hold each row's block bytes (127 for padding
    rows).  An all-zero block and a tiny block exercise byte 127 and a
    negative exponent."""
    F = lib()
    n, k = shape
    _, w = workloads.fine_grained(1, k=k, n=n)
    w = w.to(in_dtype)
    w[:32, 32:64] = 0.0
    w[(n - 1) // 32 * 32:, -32:] *= 1e-28  # the last block: exponent near -100
    wf = w.float().numpy()
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    sc = torch.empty(((n + 31) // 32, k // 32), dtype=torch.uint8, device="cuda")
    words = F.mx_local_words(n, k)
    F.fp8_quantize_block32(w.cuda(), FMT[fmt], q, sc, words)
    ref_q, ref_s = OQ.quantize_block(wf, fmt, "ue8m0", block=32)
    assert np.array_equal(to_np_u8(q), ref_q)
    assert np.array_equal(to_np_u8(sc), ref_s)
    per_row = np.repeat(ref_s, 32, axis=0)[:n]
    assert np.array_equal(words.cpu().numpy().view(np.uint32), mx_pack(per_row).view(np.uint32))


def test_quantize_block32_without_block_bytes():
    F = lib()
    _, w = workloads.fine_grained(1, k=256, n=96)
    q = torch.empty((96, 256), dtype=torch.uint8, device="cuda")
    words = F.mx_local_words(96, 256)
    F.fp8_quantize_block32(w.cuda(), 0, q, None, words)
    ref_q, ref_s = OQ.quantize_block(w.float().numpy(), "e4m3", "ue8m0", block=32)
    assert np.array_equal(to_np_u8(q), ref_q)
    assert np.array_equal(mx_unpack(words.cpu().numpy(), 96, 256),
                          np.repeat(ref_s, 32, axis=0)[:96])


@pytest.mark.parametrize("shape", [(200, 272), (2048, 7168)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_dequantize_block(shape, sfmt, fmt):
    """Bit-exact against the oracle's definition, rounded the way the kernel
    forms it: the fp32 product of the code's value and the block scale, then
    bf16 round-to-nearest-even."""
    F = lib()
    n, k = shape
    _, w = workloads.fine_grained(1, k=k, n=n)
    q, sc = OQ.quantize_block(w.float().numpy(), fmt, sfmt)
    out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    F.fp8_dequantize_block(torch.from_numpy(q).cuda(), FMT[fmt],
                           torch.from_numpy(np.ascontiguousarray(sc)).cuda(),
                           0 if sfmt == "f32" else 1, out)
    ref = OQ.dequantize_block(q, fmt, sc, sfmt).astype(np.float32)  # fp32 product
    ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16)
    assert torch.equal(out.cpu(), ref_bf16)


def all_finite_bf16():
    """Every bf16 bit pattern except the NaNs (set to +0), as a 256 x 256
    tensor: all normals, subnormals, both zeros and both infinities."""
    bits = np.arange(65536, dtype=np.uint32)
    nan = ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)
    bits[nan] = 0
    x = (bits << 16).view(np.float32).reshape(256, 256)
    return torch.from_numpy(x.copy()).to(torch.bfloat16)


def scales_under_test(seed):
    """Given scales spanning fp32: both ends of the range where the kernels
    divide through the reciprocal (2^-80 .. 2^80) and their neighbours just
    outside it, the usual 1 / MAX, and seeded draws with random mantissas and
    exponents from -100 to 100."""
    rng = np.random.default_rng(seed)
    f = np.float32
    fixed = [f(2.0 ** -80), f(2.0 ** 80), np.nextafter(f(2.0 ** -80), f(0)),
             np.nextafter(f(2.0 ** 80), f(np.inf)), f(1.0) / f(448.0), f(1.0) / f(57344.0),
             f(1.0), f(3.0), f(1e-30), f(1e30)]
    mant = rng.integers(0, 1 << 23, 40, dtype=np.uint32)
    expo = rng.integers(-100, 101, 40).astype(np.int64)
    drawn = ((expo + 127).astype(np.uint32) << 23 | mant).view(np.float32)
    return [f(v) for v in fixed] + [f(v) for v in drawn]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("transpose", [False, True])
def test_given_scale_every_bf16_input(fmt, transpose):
    """fl32(x / s) then the saturating cast, for every finite bf16 x and 50
    scales: the kernels' reciprocal-based quotient must give the codes of the
    IEEE quotient (numpy's fp32 division) bit for bit."""
    F = lib()
    x = all_finite_bf16()
    xf = x.float().numpy()
    xd = x.cuda()
    q = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
    qt = torch.empty((256, 256), dtype=torch.uint8, device="cuda") if transpose else None
    for s in scales_under_test(5):
        F.fp8_quantize_tensor(xd, FMT[fmt], q, scale=torch.tensor([s], device="cuda"), q_t=qt)
        ref = OQ.quantize_with_scale(xf, s, fmt)
        assert np.array_equal(to_np_u8(q), ref), float(s)
        if transpose:
            assert np.array_equal(to_np_u8(qt), ref.T), float(s)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_nan_inputs_give_nan_codes(fmt):
    """NaN inputs of either sign give a NaN code (the oracle defines codes for
    finite and infinite inputs only; a NaN is not cast to a number), on the
    reciprocal path and on the IEEE one, while the finite neighbours in the
    same vectors keep the oracle's codes."""
    from oracle import formats as OF
    F = lib()
    bits = np.full(64 * 32, 0x3F80, dtype=np.uint32)                  # 1.0
    bits[::5] = 0x7FC0                                                # +NaN
    bits[2::7] = 0xFFC1                                               # -NaN
    bits[3::11] = 0xC2F6                                              # -123.0
    x = torch.from_numpy((bits << 16).view(np.float32).reshape(64, 32)).to(torch.bfloat16)
    xf = x.float().numpy()
    nan = np.isnan(xf)
    q = torch.empty((64, 32), dtype=torch.uint8, device="cuda")
    for s in (np.float32(0.37), np.float32(2.0 ** 90)):
        F.fp8_quantize_tensor(x.cuda(), FMT[fmt], q, scale=torch.tensor([s], device="cuda"))
        codes = to_np_u8(q)
        assert np.isnan(OF.decode(codes[nan], OF.fmt_of(fmt))).all(), float(s)
        ref = OQ.quantize_with_scale(np.where(nan, 0, xf), s, fmt)
        assert np.array_equal(codes[~nan], ref[~nan]), float(s)


def midpoint_neighbours(fmt, scales):
    """fp32 inputs x whose quotient x / s lies on or within a few fp32 ulps of
    a rounding midpoint between two FP8 codes (the cases a quotient that is
    not correctly rounded would get wrong after the cast)."""
    from oracle import formats as OF
    f = OF.fmt_of(fmt)
    vals = np.sort(np.unique(np.abs(OF.decode(np.arange(256, dtype=np.uint8), f))))
    vals = vals[np.isfinite(vals)]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    rows = []
    for s in scales:
        base = (mids * np.float32(s)).astype(np.float32)
        for d in range(-3, 4):
            v = base.view(np.int32) + np.int32(d)
            rows.append(v.view(np.float32))
    x = np.concatenate(rows)
    x = np.concatenate([x, -x])
    pad = (-len(x)) % 256
    x = np.concatenate([x, np.zeros(pad, dtype=np.float32)]).reshape(-1, 256)
    return x[np.isfinite(x).all(axis=1)]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_given_scale_fp32_near_fp8_midpoints(fmt):
    F = lib()
    scales = scales_under_test(6)[:30]
    x = midpoint_neighbours(fmt, scales)
    xd = torch.from_numpy(x).cuda()
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    for s in scales:
        F.fp8_quantize_tensor(xd, FMT[fmt], q, scale=torch.tensor([s], device="cuda"))
        assert np.array_equal(to_np_u8(q), OQ.quantize_with_scale(x, s, fmt)), float(s)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_nan_input_gives_nan_code(fmt):
    """The oracle takes finite inputs only; a NaN input must come out as a
    NaN code (satfinite keeps NaN) whichever way the quotient is formed."""
    F = lib()
    x = torch.zeros((2, 128), device="cuda")
    x[0, 5] = float("nan")
    x[1, 7] = -float("nan")
    q = torch.empty((2, 128), dtype=torch.uint8, device="cuda")
    for s in (1.0 / 448.0, 2.0 ** 90):
        F.fp8_quantize_tensor(x, FMT[fmt], q, scale=torch.tensor([s], device="cuda"))
        c = to_np_u8(q)
        nan_codes = {0x7F, 0xFF} if fmt == "e4m3" else {0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF}
        assert int(c[0, 5]) in nan_codes and int(c[1, 7]) in nan_codes
        assert int(c[0, 0]) == 0


# ------------------------------------------ several tensors in one launch --

def run_quantize_tensors(xs, fmts):
    F = lib()
    dev = [x.cuda() for x in xs]
    qs = [torch.empty(x.numel(), dtype=torch.uint8, device="cuda") for x in xs]
    amax = torch.zeros(len(xs), device="cuda")
    scale = torch.zeros(len(xs), device="cuda")
    sync = torch.zeros(F.QUANT_SYNC_WORDS, dtype=torch.int32, device="cuda")
    items = [F.quant_item(d, FMT[f], q, scale[i:i + 1], amax[i:i + 1])
             for i, (d, f, q) in enumerate(zip(dev, fmts, qs))]
    F.fp8_quantize_tensors(items, sync)
    torch.cuda.synchronize()
    return [to_np_u8(q) for q in qs], amax.cpu().numpy(), scale.cpu().numpy()


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_quantize_tensors_matches_oracle(dt):
    """Four tensors: ragged sizes (n % 8 == 1 included), both formats, and an
    all-zero tensor (amax 0 -> scale 1); amax, scale and codes bit-exact."""
    xs = [special_input((300, 520), 1.0, 21, dt, "e4m3"),
          special_input((8, 16), 1e-3, 22, dt, "e5m2"),
          workloads.normal((1001,), 1.0, 23).to(dt),
          torch.zeros((64, 64), dtype=dt)]
    fmts = ["e4m3", "e5m2", "e4m3", "e5m2"]
    codes, amax, scale = run_quantize_tensors(xs, fmts)
    for i, (x, f) in enumerate(zip(xs, fmts)):
        xf = x.float().numpy().reshape(-1)
        ref_q, ref_s = OQ.quantize_tensor(xf, f)
        assert f32_bits(amax[i]) == f32_bits(OQ.amax(xf)), i
        assert f32_bits(scale[i]) == f32_bits(ref_s), i
        assert np.array_equal(codes[i], ref_q), i


def test_quantize_tensors_empty_item():
    """An empty tensor among the items (null pointers, n == 0): amax 0 and
    scale 1 for it, the other items as the oracle gives them."""
    dt = torch.bfloat16
    xs = [workloads.normal((2, 4104), 1.0, 31).to(dt), torch.empty(0, dtype=dt),
          workloads.normal((777,), 3.0, 32).to(dt)]
    fmts = ["e4m3", "e5m2", "e5m2"]
    codes, amax, scale = run_quantize_tensors(xs, fmts)
    assert amax[1] == 0.0 and scale[1] == 1.0 and codes[1].size == 0
    for i in (0, 2):
        xf = xs[i].float().numpy().reshape(-1)
        ref_q, ref_s = OQ.quantize_tensor(xf, fmts[i])
        assert f32_bits(amax[i]) == f32_bits(OQ.amax(xf)), i
        assert f32_bits(scale[i]) == f32_bits(ref_s), i
        assert np.array_equal(codes[i], ref_q), i


def test_amax_empty():
    """n == 0: the call clears the output to 0 (the amax of nothing, as the
    oracle's amax of an empty array) and reads no input."""
    F = lib()
    out = torch.full((1,), 7.0, device="cuda")
    F.fp8_amax(torch.empty(0, device="cuda"), out)
    assert out.item() == 0.0 == float(OQ.amax(np.zeros(0, np.float32)))


def test_quantize_tensors_float8_linear_full_size():
    """The Float8 linear step's x, g and W (8192 x 2048, 8192 x 2048,
    2048 x 2048) in the order the step quantizes them."""
    x, w, g = workloads.float8_linear()
    xs, fmts = [x, g, w], ["e4m3", "e5m2", "e4m3"]
    codes, amax, scale = run_quantize_tensors(xs, fmts)
    for i, (t, f) in enumerate(zip(xs, fmts)):
        tf = t.float().numpy().reshape(-1)
        ref_q, ref_s = OQ.quantize_tensor(tf, f)
        assert f32_bits(scale[i]) == f32_bits(ref_s), i
        assert np.array_equal(codes[i], ref_q), i


def test_quantize_tensors_in_a_cuda_graph():
    """Captured once, replayed on new data: the scratch is cleared by the
    captured memset, so every replay starts from zero."""
    F = lib()
    shapes = [(512, 1024), (256, 256)]
    xs = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in shapes]
    qs = [torch.empty(s, dtype=torch.uint8, device="cuda") for s in shapes]
    scale = torch.zeros(2, device="cuda")
    sync = torch.zeros(F.QUANT_SYNC_WORDS, dtype=torch.int32, device="cuda")
    items = [F.quant_item(xs[i], F.E4M3, qs[i], scale[i:i + 1]) for i in range(2)]
    for i, s in enumerate(shapes):
        xs[i].copy_(workloads.normal(s, 1.0, 30 + i))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        F.fp8_quantize_tensors(items, sync)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        F.fp8_quantize_tensors(items, sync)
    for rep in range(3):
        host = [workloads.normal(s, 0.5 + rep, 40 + 2 * rep + i).to(torch.bfloat16)
                for i, s in enumerate(shapes)]
        for i in range(2):
            xs[i].copy_(host[i])
        graph.replay()
        torch.cuda.synchronize()
        for i in range(2):
            ref_q, ref_s = OQ.quantize_tensor(host[i].float().numpy(), "e4m3")
            assert f32_bits(scale[i].item()) == f32_bits(ref_s), (rep, i)
            assert np.array_equal(to_np_u8(qs[i]), ref_q), (rep, i)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantize_tensors_every_bf16_below_amax(fmt):
    """The scale of current scaling comes from the tensor itself, so every
    quotient is bounded; the kernel then divides without the range guard and
    puts each input's sign into its code.  Checked on tensors that hold every
    finite bf16 value up to 2^k (both zeros, all subnormals, both signs), for
    k from -100 to 100: amax, scale and every code bit-exact."""
    bits = np.arange(65536, dtype=np.uint32)
    allv = (bits << 16).view(np.float32)
    allv = allv[np.isfinite(allv)]
    xs = []
    for k in (-100, -20, -3, 0, 5, 17, 60, 100):
        v = allv[np.abs(allv) <= np.float32(2.0 ** k)]
        xs.append(torch.from_numpy(v.copy()).to(torch.bfloat16))
    for i in range(0, len(xs), 4):
        chunk = xs[i:i + 4]
        codes, amax, scale = run_quantize_tensors(chunk, [fmt] * len(chunk))
        for j, x in enumerate(chunk):
            xf = x.float().numpy()
            ref_q, ref_s = OQ.quantize_tensor(xf, fmt)
            assert f32_bits(scale[j]) == f32_bits(ref_s), (i + j)
            assert np.array_equal(codes[j], ref_q), (i + j)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_amax_rows(dt):
    F = lib()
    x = special_input((300, 520), 1.0, 17, dt, "e4m3")
    x[7] = 0.0
    out = torch.empty(300, device="cuda")
    F.fp8_amax_rows(x.cuda(), out)
    ref = np.max(np.abs(x.float().numpy()), axis=1).astype(np.float32)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("shape", [(1, 128), (130, 512), (333, 2048)])
def test_two_level_per_row_global(shape):
    F = lib()
    r, k = shape
    a, _ = workloads.two_level(m=r, n=8, k=k)
    x = a.clone()
    x[0, 32:64] = 0.0
    if r > 3:
        x[3] *= 2.0 ** -20     # a row far smaller than the others
    xf = x.float().numpy()
    xd = x.cuda()
    am = torch.empty(r, device="cuda")
    F.fp8_amax_rows(xd, am)
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    words = F.mx_local_words(r, k)
    glob = torch.empty(r, device="cuda")
    F.fp8_quantize_mx_rows(xd, 0, am, glob, q, words)
    ref_q, ref_l, ref_s = OQ.quantize_two_level(xf, "e4m3", global_per_row=True)
    assert np.array_equal(glob.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(to_np_u8(q), ref_q)
    assert np.array_equal(mx_unpack(words.cpu().numpy(), r, k), ref_l)
