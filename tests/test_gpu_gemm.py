"""GPU parity of the scaled-FP8 GEMMs against the float64 oracle.

Operands are quantized by the ORACLE on the CPU and uploaded, so each GEMM is
checked on its own.  Acceptance per output element:
|gpu - oracle| <= 1e-3 * sum_k |a_deq| |b_deq| (+ one bf16 ulp of |oracle| for a
bf16 output)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import FMT, lib, mx_pack, sample_positions
from oracle import gemm as OG
from oracle import quantize as OQ

pytestmark = pytest.mark.gpu


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_f32(v):
    return torch.tensor(np.atleast_1d(np.asarray(v, dtype=np.float32)), device="cuda")


def per_tensor_operands(m, n, k, fa, fb, seed):
    sa_std = 1.0 if fa == "e4m3" else 1e-3
    x = workloads.normal((m, k), sa_std, seed).to(torch.bfloat16).float().numpy()
    w = workloads.normal((n, k), 0.02, seed + 1).to(torch.bfloat16).float().numpy()
    qa, sa = OQ.quantize_tensor(x, fa)
    qb, sb = OQ.quantize_tensor(w, fb)
    return qa, sa, qb, sb


def run_tensor(qa, fa, sa, qb, fb, sb, out_dtype, accumulate_into=None):
    F = lib()
    m, n = qa.shape[0], qb.shape[0]
    if accumulate_into is not None:
        out = accumulate_into
    else:
        out = torch.empty((m, n), dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32,
                          device="cuda")
    F.fp8_gemm_tensor(dev_u8(qa), FMT[fa], dev_u8(qb), FMT[fb], dev_f32(sa), dev_f32(sb), out,
                      accumulate=accumulate_into is not None)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


SHAPES = [(128, 256, 128), (1, 64, 32), (16, 64, 32), (129, 300, 272), (300, 520, 1024),
          (256, 512, 4096), (1000, 130, 16)]


@pytest.mark.parametrize("mnk", SHAPES)
@pytest.mark.parametrize("fmts", [("e4m3", "e4m3"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_gemm_tensor(mnk, fmts, out_dtype):
    m, n, k = mnk
    fa, fb = fmts
    qa, sa, qb, sb = per_tensor_operands(m, n, k, fa, fb, seed=m + n + k)
    got = run_tensor(qa, fa, sa, qb, fb, sb, out_dtype)
    c, e = OG.gemm(OG.dequant_operand(qa, fa, sa), OG.dequant_operand(qb, fb, sb))
    ok, worst = OG.check(got, c, e, out_dtype)
    assert ok, worst


def test_gemm_tensor_accumulate():
    m, n, k = 200, 384, 256
    qa, sa, qb, sb = per_tensor_operands(m, n, k, "e5m2", "e4m3", seed=3)
    qa2, sa2, qb2, sb2 = per_tensor_operands(m, n, k, "e5m2", "e4m3", seed=9)
    out = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    run_tensor(qa, "e5m2", sa, qb, "e4m3", sb, "f32", accumulate_into=out)
    got = run_tensor(qa2, "e5m2", sa2, qb2, "e4m3", sb2, "f32", accumulate_into=out)
    c1, e1 = OG.gemm(OG.dequant_operand(qa, "e5m2", sa), OG.dequant_operand(qb, "e4m3", sb))
    c2, e2 = OG.gemm(OG.dequant_operand(qa2, "e5m2", sa2), OG.dequant_operand(qb2, "e4m3", sb2))
    ok, worst = OG.check(got, c1 + c2, e1 + e2, "f32")
    assert ok, worst


def test_tiny_per_tensor_example():
    """The Flax guide's 16x32 . 32x64 example (section 2.2), current scaling,
    fp32 output; b is passed as b^T [64, 32]."""
    F = lib()
    a, b = workloads.tiny_per_tensor()
    ad, btd = a.cuda(), b.t().contiguous().cuda()
    qa = torch.empty((16, 32), dtype=torch.uint8, device="cuda")
    qb = torch.empty((64, 32), dtype=torch.uint8, device="cuda")
    am, bm = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    sa, sb = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    F.fp8_amax(ad, am)
    F.fp8_amax(btd, bm)
    F.fp8_quantize_tensor(ad, 0, qa, amax_in=am, scale_out=sa)
    F.fp8_quantize_tensor(btd, 0, qb, amax_in=bm, scale_out=sb)
    out = torch.empty((16, 64), dtype=torch.float32, device="cuda")
    F.fp8_gemm_tensor(qa, 0, qb, 0, sa, sb, out)
    ra, rsa = OQ.quantize_tensor(a.numpy(), "e4m3")
    rb, rsb = OQ.quantize_tensor(b.t().contiguous().numpy(), "e4m3")
    assert np.array_equal(qa.cpu().numpy(), ra) and np.array_equal(qb.cpu().numpy(), rb)
    assert sa.item() == float(rsa) and sb.item() == float(rsb)
    c, e = OG.gemm(OG.dequant_operand(ra, "e4m3", rsa), OG.dequant_operand(rb, "e4m3", rsb))
    ok, worst = OG.check(out.cpu().numpy(), c, e, "f32")
    assert ok, worst


# ------------------------------------------------------------ per K group --

def group_operands(m, n, k, sfmt, seed):
    act, w = workloads.fine_grained(m, seed=seed, k=k, n=n)
    qa, sa = OQ.quantize_token_group(act.float().numpy(), "e4m3", sfmt)
    qb, sb = OQ.quantize_block(w.float().numpy(), "e4m3", sfmt)
    return qa, sa, qb, sb


def group_reference(qa, sa, qb, sb, sfmt, rows=None, cols=None):
    m, k = qa.shape
    n = qb.shape[0]
    a = OG.dequant_operand(qa, "e4m3", OQ.expand(OQ.group_scale_values(sa, sfmt), m, k, 1, 128))
    b = OG.dequant_operand(qb, "e4m3", OQ.expand(OQ.group_scale_values(sb, sfmt), n, k, 128, 128))
    if rows is None:
        return OG.gemm(a, b)
    return OG.gemm_sampled(a, b, rows, cols)


def run_group(qa, sa, qb, sb, sfmt):
    F = lib()
    m, n = qa.shape[0], qb.shape[0]
    sa_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sa).T)).cuda()   # [G, M]
    sb_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sb))).cuda()     # [N/128, G]
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    F.fp8_gemm_group(dev_u8(qa), sa_dev, dev_u8(qb), sb_dev, 0 if sfmt == "f32" else 1, out)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("mnk", [(1, 256, 512), (128, 128, 128), (200, 384, 1024),
                                 (130, 2048, 7168), (513, 200, 384)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_gemm_group(mnk, sfmt):
    m, n, k = mnk
    qa, sa, qb, sb = group_operands(m, n, k, sfmt, seed=2)
    got = run_group(qa, sa, qb, sb, sfmt)
    c, e = group_reference(qa, sa, qb, sb, sfmt)
    ok, worst = OG.check(got, c, e, "bf16")
    assert ok, worst


@pytest.mark.parametrize("m,k", [(1, 7168), (3, 7168), (1, 20480)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_gemm_group_few_rows(m, k, sfmt):
    """With the switch on a single row runs on the CUDA cores (a stream over
    the weights); more rows, and one row by default, on the few-row
    tensor-core kernel.  Ragged N (301: the last block of the one-row kernel
    holds one valid column), a K with several load steps per lane and a
    partial last one (20480), a bias, both scale formats."""
    F = lib()
    n = 301
    qa, sa, qb, sb = group_operands(m, n, k, sfmt, seed=m + 40)
    bias = _bias(n, m)
    c, e = group_reference(qa, sa, qb, sb, sfmt)
    cb, eb, extra = OG.gemm_bias(c, e, bias)
    sa_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sa).T)).cuda()
    sb_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sb))).cuda()
    code = F.SCALE_F32 if sfmt == "f32" else F.SCALE_UE8M0
    try:
        for few in (1, 0):
            F.fp8_set_option(F.OPT_GEMM_FEW_ROWS, few)
            out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
            F.fp8_gemm_group(dev_u8(qa), sa_dev, dev_u8(qb), sb_dev, code, out,
                             bias=torch.from_numpy(bias).cuda())
            torch.cuda.synchronize()
            ok, worst = OG.check(out.float().cpu().numpy(), cb, eb, "bf16", extra=extra)
            assert ok, (few, worst)
    finally:
        F.fp8_set_option(F.OPT_GEMM_FEW_ROWS, 0)  # the default


@pytest.mark.parametrize("multicast", [0, 1])
@pytest.mark.parametrize("mnk", [(300, 384, 1024), (1000, 2048, 512)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_gemm_group_multicast_switch(mnk, sfmt, multicast):
    """The B-multicast clusters (two CTAs on vertically adjacent row tiles,
    including a last pair whose second tile lies past M) and the plain
    launch give results within the bound, for both scale formats (UE8M0
    beyond M = 128 runs through the E8M0-word block-scaled kernel)."""
    F = lib()
    m, n, k = mnk
    qa, sa, qb, sb = group_operands(m, n, k, sfmt, seed=4)
    F.fp8_set_option(F.OPT_GEMM_MULTICAST, multicast)
    try:
        got = run_group(qa, sa, qb, sb, sfmt)
    finally:
        F.fp8_set_option(F.OPT_GEMM_MULTICAST, 1)
    c, e = group_reference(qa, sa, qb, sb, sfmt)
    ok, worst = OG.check(got, c, e, "bf16")
    assert ok, worst


@pytest.mark.parametrize("mnk", [(1800, 2000, 512), (1024, 9728, 256), (2048, 1800, 384)])
def test_gemm_group_f32_cta_pairs(mnk):
    """FP32 group scales on CTA pairs (256 x 256 tiles, the promotion in both
    CTAs): ragged M and N (1800 rows = 7 * 256 + 8: the last pair's second CTA
    lies wholly past M; 2000 = 7 * 256 + 208 columns; 1800 columns: the last
    tile's second 128-column half lies wholly past N, with no weight scale
    block of its own) and a bias, against the oracle with pairs on and off;
    the switch off runs the one-CTA kernel."""
    F = lib()
    m, n, k = mnk
    qa, sa, qb, sb = group_operands(m, n, k, "f32", seed=9)
    bias = np.asarray(workloads.normal((n,), 0.5, 91).numpy(), np.float32)
    c, e = group_reference(qa, sa, qb, sb, "f32")
    cb, eb, extra = OG.gemm_bias(c, e, bias)
    sa_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sa).T)).cuda()
    sb_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sb))).cuda()
    try:
        for pairs in (1, 0):
            F.fp8_set_option(F.OPT_GEMM_CTA_PAIRS, pairs)
            out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
            F.fp8_gemm_group(dev_u8(qa), sa_dev, dev_u8(qb), sb_dev, 0, out,
                             bias=torch.from_numpy(bias).cuda())
            torch.cuda.synchronize()
            ok, worst = OG.check(out.float().cpu().numpy(), cb, eb, "bf16", extra=extra)
            assert ok, (pairs, worst)
    finally:
        F.fp8_set_option(F.OPT_GEMM_CTA_PAIRS, 1)
    rc, where = F.fp8_get_last_device_error()
    assert rc == 0, (rc, where)


def test_gemm_group_f32_cta_pairs_one_slice_pitched():
    """The CTA-pair FP32 kernel with a single 128-deep K slice (fewer slices
    than the scale prefetch distance) writing a pitched output (ldc = N + 24):
    the padding columns stay untouched and the result agrees with the oracle."""
    F = lib()
    m, n, k, pad = 2048, 1280, 128, 24
    qa, sa, qb, sb = group_operands(m, n, k, "f32", seed=12)
    c, e = group_reference(qa, sa, qb, sb, "f32")
    sa_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sa).T)).cuda()
    sb_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sb))).cuda()
    full = torch.full((m, n + pad), 7.0, dtype=torch.bfloat16, device="cuda")
    F.fp8_gemm_group(dev_u8(qa), sa_dev, dev_u8(qb), sb_dev, 0, full)
    torch.cuda.synchronize()
    got = full.float().cpu().numpy()
    assert np.all(got[:, n:] == 7.0)
    ok, worst = OG.check(got[:, :n], c, e, "bf16")
    assert ok, worst
    assert F.fp8_get_last_device_error()[0] == 0


# -------------------------------------------------------------- two level --

def mx_operands(m, n, k, seed):
    a, b = workloads.two_level(seed=seed, m=m, n=n, k=k)
    qa, la, ga = OQ.quantize_two_level(a.float().numpy(), "e4m3")
    qb, lb, gb = OQ.quantize_two_level(b.float().numpy(), "e4m3")
    return qa, la, ga, qb, lb, gb


def mx_reference(qa, la, ga, qb, lb, gb, rows=None, cols=None):
    m, k = qa.shape
    n = qb.shape[0]
    a = OG.dequant_operand(qa, "e4m3", OQ.expand(OQ.two_level_scale_values(la, ga), m, k, 1, 32))
    b = OG.dequant_operand(qb, "e4m3", OQ.expand(OQ.two_level_scale_values(lb, gb), n, k, 1, 32))
    if rows is None:
        return OG.gemm(a, b)
    return OG.gemm_sampled(a, b, rows, cols)


def run_mx(qa, la, ga, qb, lb, gb, out_dtype="bf16"):
    F = lib()
    m, n = qa.shape[0], qb.shape[0]
    out = torch.empty((m, n), dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32,
                      device="cuda")
    F.fp8_gemm_mx(dev_u8(qa), torch.from_numpy(mx_pack(la)).cuda(), dev_f32(ga), dev_u8(qb),
                  torch.from_numpy(mx_pack(lb)).cuda(), dev_f32(gb), out)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("mnk", [(128, 256, 128), (200, 384, 512), (1, 128, 256), (300, 1000, 1024)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_gemm_mx(mnk, out_dtype):
    m, n, k = mnk
    qa, la, ga, qb, lb, gb = mx_operands(m, n, k, seed=3)
    got = run_mx(qa, la, ga, qb, lb, gb, out_dtype)
    c, e = mx_reference(qa, la, ga, qb, lb, gb)
    ok, worst = OG.check(got, c, e, out_dtype)
    assert ok, worst


@pytest.mark.parametrize("mnk", [(128, 256, 256), (200, 300, 512), (1, 128, 128), (4096, 2048, 7168)])
def test_gemm_mxfp8_by_block32_weights(mnk):
    """One-level MXFP8 activations (1x32 power-of-two scales) times (32, 32)
    UE8M0 weight blocks, both quantized on the GPU and contracted by the
    block-scaled GEMM with unit global factors; the oracle dequantizes with
    its own quantizers' scales.  The large case is checked on sampled
    outputs."""
    F = lib()
    m, n, k = mnk
    a, w = workloads.fine_grained(m, k=k, n=n)
    af, wf = a.float().numpy(), w.float().numpy()
    qa = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    la = F.mx_local_words(m, k)
    ga = torch.zeros(1, device="cuda")
    F.fp8_quantize_mx1(a.cuda(), 0, ga, qa, la)
    qb = torch.empty((n, k), dtype=torch.uint8, device="cuda")
    lb = F.mx_local_words(n, k)
    F.fp8_quantize_block32(w.cuda(), 0, qb, None, lb)
    gb = torch.ones(1, device="cuda")
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    F.fp8_gemm_mx(qa, la, ga, qb, lb, gb, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    rq_a, rl_a = OQ.quantize_mxfp8(af, "e4m3")
    rq_b, rs_b = OQ.quantize_block(wf, "e4m3", "ue8m0", block=32)
    a_deq = OG.dequant_operand(rq_a, "e4m3", OQ.expand(OQ.group_scale_values(rl_a, "ue8m0"), m, k, 1, 32))
    b_deq = OG.dequant_operand(rq_b, "e4m3", OQ.expand(OQ.group_scale_values(rs_b, "ue8m0"), n, k, 32, 32))
    if m * n * k > 1 << 30:
        rows, cols = sample_positions(m, n, 256, seed=9)
        c, e = OG.gemm_sampled(a_deq, b_deq, rows, cols)
        ok, worst = OG.check(got[rows, cols], c, e, "bf16")
    else:
        c, e = OG.gemm(a_deq, b_deq)
        ok, worst = OG.check(got, c, e, "bf16")
    assert ok, worst


def test_gemm_mx_distinct_local_factors():
    """Every 1x32 block of both operands gets its own power-of-two factor, so a
    factor applied to the wrong block or row shows up."""
    m, n, k = 256, 256, 512
    rng = np.random.default_rng(11)
    qa, la, ga, qb, lb, gb = mx_operands(m, n, k, seed=5)
    la = (127 - rng.integers(0, 6, la.shape)).astype(np.uint8)
    lb = (127 - rng.integers(0, 6, lb.shape)).astype(np.uint8)
    got = run_mx(qa, la, ga, qb, lb, gb, "f32")
    c, e = mx_reference(qa, la, ga, qb, lb, gb)
    ok, worst = OG.check(got, c, e, "f32")
    assert ok, worst


@pytest.mark.parametrize("mnk", [(4096, 2048, 7168), (2048, 4096, 1024)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_gemm_group_large(mnk, sfmt):
    """The configured M = 4096 shape and a wider one (FP32 promotion on
    multicast 128-wide tiles; UE8M0 on E8M0 words and 128 x 256 tiles),
    checked on sampled outputs including every edge tile's corners."""
    m, n, k = mnk
    qa, sa, qb, sb = group_operands(m, n, k, sfmt, seed=6)
    got = run_group(qa, sa, qb, sb, sfmt)
    rows, cols = sample_positions(m, n, 512, seed=m + k)
    c, e = group_reference(qa, sa, qb, sb, sfmt, rows, cols)
    ok, worst = OG.check(got[rows, cols], c, e, "bf16")
    assert ok, worst


# ------------------------------------------------------- split K (small M) --

@pytest.mark.parametrize("m", [1, 7, 64, 128])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_gemm_group_small_m_split_k(m, sfmt):
    """Config-3 shapes at decode-like M: the tiles cannot fill the GPU, so K is
    split across CTAs and the last CTA of each tile reduces the fp32 partials.
    Two calls in a row: the arrival counters must be back at zero."""
    n, k = 2048, 7168
    qa, sa, qb, sb = group_operands(m, n, k, sfmt, seed=2)
    c, e = group_reference(qa, sa, qb, sb, sfmt)
    for _ in range(2):
        got = run_group(qa, sa, qb, sb, sfmt)
        ok, worst = OG.check(got, c, e, "bf16")
        assert ok, worst


@pytest.mark.parametrize("mnk", [(2, 300, 1024), (16, 2048, 7168), (17, 1000, 2048),
                                 (33, 384, 7168), (64, 2048, 7168), (65, 200, 512),
                                 (128, 2048, 7168), (100, 7168, 2048), (1, 2048, 256)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_gemm_group_few_rows_kernel(mnk, sfmt):
    """The few-row per-group kernel (weights on the MMA's M side, the M
    activation rows padded to 16, 32, 64 or 128 on its N side, K split over
    a cluster) against the oracle, with the switch on and off: every padded
    width and its edges, ragged N (the last weight tile partly past N), K
    shorter than the cluster (one k block per split), a bias and an output
    pitch wider than N.  Past 64 rows (65, 100, 128) the switch on runs two
    64-row halves of CTAs (the second one ragged at 65 and 100)."""
    F = lib()
    m, n, k = mnk
    qa, sa, qb, sb = group_operands(m, n, k, sfmt, seed=m + n)
    c, e = group_reference(qa, sa, qb, sb, sfmt)
    bias = _bias(n, m + 5)
    cb, eb, extra = OG.gemm_bias(c, e, bias)
    sa_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sa).T)).cuda()
    sb_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sb))).cuda()
    code = F.SCALE_F32 if sfmt == "f32" else F.SCALE_UE8M0
    ldc = n + 24
    try:
        F.fp8_set_option(F.OPT_GEMM_FEW_ROWS, 0)
        for skinny in (1, 0):
            F.fp8_set_option(F.OPT_GEMM_SKINNY, skinny)
            for with_bias in (False, True):
                # (N comes from the weights; the output's row pitch is ldc)
                buf = torch.full((m, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
                F.fp8_gemm_group(dev_u8(qa), sa_dev, dev_u8(qb), sb_dev, code, buf,
                                 bias=torch.from_numpy(bias).cuda() if with_bias else None)
                torch.cuda.synchronize()
                got = buf[:, :n].float().cpu().numpy()
                if with_bias:
                    ok, worst = OG.check(got, cb, eb, "bf16", extra=extra)
                else:
                    ok, worst = OG.check(got, c, e, "bf16")
                assert ok, (skinny, with_bias, worst)
                assert torch.isnan(buf[:, n:].float()).all()  # nothing past N
        assert F.fp8_get_last_device_error()[0] == 0
    finally:
        F.fp8_set_option(F.OPT_GEMM_SKINNY, 1)
        F.fp8_set_option(F.OPT_GEMM_FEW_ROWS, 0)


@pytest.mark.parametrize("mnk", [(1, 2048, 4096), (100, 256, 8192), (33, 1000, 2048)])
def test_gemm_tensor_small_m_split_k(mnk):
    m, n, k = mnk
    qa, sa, qb, sb = per_tensor_operands(m, n, k, "e5m2", "e4m3", seed=m)
    c, e = OG.gemm(OG.dequant_operand(qa, "e5m2", sa), OG.dequant_operand(qb, "e4m3", sb))
    for out_dtype in ("f32", "bf16"):
        got = run_tensor(qa, "e5m2", sa, qb, "e4m3", sb, out_dtype)
        ok, worst = OG.check(got, c, e, out_dtype)
        assert ok, (out_dtype, worst)


def test_gemm_mx_small_m_split_k():
    qa, la, ga, qb, lb, gb = mx_operands(1, 1024, 4096, seed=7)
    c, e = mx_reference(qa, la, ga, qb, lb, gb)
    got = run_mx(qa, la, ga, qb, lb, gb, "bf16")
    ok, worst = OG.check(got, c, e, "bf16")
    assert ok, worst


def test_split_k_on_two_streams():
    """Split-K calls on two streams at once (each tile's splits reduce inside
    their own thread-block cluster, so concurrent calls share nothing) give
    the results of calls on one stream."""
    F = lib()
    m, n, k = 16, 2048, 7168
    qa, sa, qb, sb = group_operands(m, n, k, "f32", seed=4)
    c, e = group_reference(qa, sa, qb, sb, "f32")
    a_d, b_d = dev_u8(qa), dev_u8(qb)
    sa_d = torch.from_numpy(np.ascontiguousarray(np.asarray(sa).T)).cuda()
    sb_d = torch.from_numpy(np.ascontiguousarray(np.asarray(sb))).cuda()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [torch.empty((m, n), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        F.fp8_gemm_group(a_d, sa_d, b_d, sb_d, 0, o, stream=s1 if i % 2 == 0 else s2)
    torch.cuda.synchronize()
    for o in outs:
        ok, worst = OG.check(o.float().cpu().numpy(), c, e, "bf16")
        assert ok, worst


# --------------------------------------------------- CTA pairs (2-SM MMA) --

@pytest.mark.parametrize("mnk", [(2048, 2048, 1024), (1999, 1000, 512), (4096, 768, 2048)])
@pytest.mark.parametrize("fmts", [("e4m3", "e4m3"), ("e5m2", "e4m3")])
def test_gemm_tensor_cta_pairs(mnk, fmts):
    """Shapes large enough for the 256 x 256 CTA-pair path (ragged M and N
    included); the single-CTA path must agree within the same bound."""
    F = lib()
    m, n, k = mnk
    fa, fb = fmts
    qa, sa, qb, sb = per_tensor_operands(m, n, k, fa, fb, seed=k + 1)
    c, e = OG.gemm(OG.dequant_operand(qa, fa, sa), OG.dequant_operand(qb, fb, sb))
    try:
        for pairs in (1, 0):
            F.fp8_set_option(F.OPT_GEMM_CTA_PAIRS, pairs)
            for out_dtype in ("bf16", "f32"):
                got = run_tensor(qa, fa, sa, qb, fb, sb, out_dtype)
                ok, worst = OG.check(got, c, e, out_dtype)
                assert ok, (pairs, out_dtype, worst)
    finally:
        F.fp8_set_option(F.OPT_GEMM_CTA_PAIRS, 1)
    rc, where = F.fp8_get_last_device_error()
    assert rc == 0, (rc, where)


@pytest.mark.parametrize("pad", [24, 3])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_gemm_tensor_tma_store_epilogue(out_dtype, pad):
    """With the switch on, the CTA-pair epilogue writes C with TMA stores
    when c and its pitch allow 16-byte vectors (pad 24: a pitched output,
    ldc = N + 24) and with per-thread stores otherwise (pad 3); both, with a
    bias, ragged M and N, and the switch off (the default) leave the
    padding columns untouched and agree with the oracle."""
    F = lib()
    m, n, k = 1999, 1000, 512
    qa, sa, qb, sb = per_tensor_operands(m, n, k, "e4m3", "e4m3", seed=31)
    bias = _bias(n, 5)
    c, e = OG.gemm(OG.dequant_operand(qa, "e4m3", sa), OG.dequant_operand(qb, "e4m3", sb))
    cb, eb, extra = OG.gemm_bias(c, e, bias)
    dt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    a, b = dev_u8(qa), dev_u8(qb)
    try:
        for tma in (1, 0):
            F.fp8_set_option(F.OPT_GEMM_TMA_STORE, tma)
            full = torch.full((m, n + pad), 7.0, dtype=dt, device="cuda")
            F.fp8_gemm_tensor_grouped([F.gemm_problem(a, F.E4M3, b, F.E4M3, dev_f32(sa),
                                                      dev_f32(sb), full,
                                                      bias=torch.from_numpy(bias).cuda())])
            torch.cuda.synchronize()
            got = full.float().cpu().numpy()
            assert np.all(got[:, n:] == 7.0), tma
            ok, worst = OG.check(got[:, :n], cb, eb, out_dtype, extra=extra)
            assert ok, (tma, worst)
    finally:
        F.fp8_set_option(F.OPT_GEMM_TMA_STORE, 0)  # the default
    assert F.fp8_get_last_device_error()[0] == 0


# ------------------------------------------------------ grouped per tensor --

def _linear_problems(t, d_in, d_out, seed):
    """y = x W^T, dx = g W, dW = g^T x as three per-tensor problems."""
    x = workloads.normal((t, d_in), 1.0, seed).to(torch.bfloat16).float().numpy()
    w = workloads.normal((d_out, d_in), 0.02, seed + 1).to(torch.bfloat16).float().numpy()
    g = workloads.normal((t, d_out), 1e-3, seed + 2).to(torch.bfloat16).float().numpy()
    qx, sx = OQ.quantize_tensor(x, "e4m3")
    qw, sw = OQ.quantize_tensor(w, "e4m3")
    qg, sg = OQ.quantize_tensor(g, "e5m2")
    return [  # (A codes, fa, sa, B codes, fb, sb)
        (qx, "e4m3", sx, qw, "e4m3", sw),
        (qg, "e5m2", sg, np.ascontiguousarray(qw.T), "e4m3", sw),
        (np.ascontiguousarray(qg.T), "e5m2", sg, np.ascontiguousarray(qx.T), "e4m3", sx),
    ]


@pytest.mark.parametrize("shape", [(2048, 1024, 1024), (2000, 784, 1296), (256, 128, 256)])
def test_gemm_tensor_grouped_linear(shape):
    """The forward and both backward GEMMs of a linear layer in one call.
    Every size is some GEMM's K, so all are multiples of 16; (2000, 784, 1296)
    is ragged against the 256-wide tiles; (256, 128, 256) is too small for the
    grouped CTA-pair launch and exercises the one-after-another fallback."""
    F = lib()
    probs = _linear_problems(*shape, seed=shape[0])
    outs, descs, keep = [], [], []
    for i, (qa, fa, sa, qb, fb, sb) in enumerate(probs):
        m, n = qa.shape[0], qb.shape[0]
        dt = torch.float32 if i == 2 else torch.bfloat16
        out = torch.empty((m, n), dtype=dt, device="cuda")
        t = (dev_u8(qa), dev_u8(qb), dev_f32(sa), dev_f32(sb))
        keep.append(t)
        descs.append(F.gemm_problem(t[0], FMT[fa], t[1], FMT[fb], t[2], t[3], out))
        outs.append(out)
    F.fp8_gemm_tensor_grouped(descs)
    torch.cuda.synchronize()
    for i, (qa, fa, sa, qb, fb, sb) in enumerate(probs):
        c, e = OG.gemm(OG.dequant_operand(qa, fa, sa), OG.dequant_operand(qb, fb, sb))
        ok, worst = OG.check(outs[i].float().cpu().numpy(), c, e, "f32" if i == 2 else "bf16")
        assert ok, (i, worst)
    assert F.fp8_get_last_device_error()[0] == 0


def test_gemm_tensor_grouped_accumulate_and_ragged():
    F = lib()
    shapes = [(1024, 520, 4096), (777, 1000, 512), (2048, 512, 128)]
    probs, descs, outs, keep, prev = [], [], [], [], []
    for i, (m, n, k) in enumerate(shapes):
        qa, sa, qb, sb = per_tensor_operands(m, n, k, "e4m3", "e4m3", seed=40 + i)
        probs.append((qa, sa, qb, sb))
        init = workloads.normal((m, n), 1.0, 90 + i)
        out = init.clone().cuda()
        prev.append(init.numpy().astype(np.float64))
        t = (dev_u8(qa), dev_u8(qb), dev_f32(sa), dev_f32(sb))
        keep.append(t)
        descs.append(F.gemm_problem(t[0], F.E4M3, t[1], F.E4M3, t[2], t[3], out, accumulate=True))
        outs.append(out)
    F.fp8_gemm_tensor_grouped(descs)
    torch.cuda.synchronize()
    for i, (qa, sa, qb, sb) in enumerate(probs):
        c, e = OG.gemm(OG.dequant_operand(qa, "e4m3", sa), OG.dequant_operand(qb, "e4m3", sb))
        ok, worst = OG.check(outs[i].cpu().numpy(), c + prev[i], e + np.abs(prev[i]) * 1e-3, "f32")
        assert ok, (i, worst)


# ------------------------------------------------- MN-major operand layouts --

def run_tensor_layout(qa, fa, sa, qb, fb, sb, a_mn, b_mn, out_dtype="bf16"):
    """One per-tensor GEMM through fp8_gemm_tensor_grouped with the operands
    uploaded in the requested layout: MN-major means the codes of the
    transposed operand, row-major ([K, M] for A, [K, N] for B)."""
    F = lib()
    m, n = qa.shape[0], qb.shape[0]
    a = dev_u8(qa.T if a_mn else qa)
    b = dev_u8(qb.T if b_mn else qb)
    out = torch.empty((m, n), dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32,
                      device="cuda")
    lay = lambda mn: F.MN_MAJOR if mn else F.K_MAJOR
    F.fp8_gemm_tensor_grouped([F.gemm_problem(a, FMT[fa], b, FMT[fb], dev_f32(sa), dev_f32(sb),
                                              out, a_layout=lay(a_mn), b_layout=lay(b_mn))])
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


# (M, N, K): CTA-pair path, single-CTA path, ragged M / N, split-K (small M),
# and K that is not a multiple of 16 (allowed when both operands are MN-major)
MN_SHAPES = [(2048, 2048, 1024), (1296, 784, 2000), (256, 512, 384), (208, 400, 256),
             (32, 2048, 4096)]


@pytest.mark.parametrize("mnk", MN_SHAPES)
@pytest.mark.parametrize("layout", [(False, True), (True, False), (True, True)])
def test_gemm_tensor_mn_major(mnk, layout):
    F = lib()
    m, n, k = mnk
    a_mn, b_mn = layout
    qa, sa, qb, sb = per_tensor_operands(m, n, k, "e5m2", "e4m3", seed=m + 7 * k)
    c, e = OG.gemm(OG.dequant_operand(qa, "e5m2", sa), OG.dequant_operand(qb, "e4m3", sb))
    try:
        for pairs in (1, 0):
            F.fp8_set_option(F.OPT_GEMM_CTA_PAIRS, pairs)
            got = run_tensor_layout(qa, "e5m2", sa, qb, "e4m3", sb, a_mn, b_mn)
            ok, worst = OG.check(got, c, e, "bf16")
            assert ok, (pairs, worst)
    finally:
        F.fp8_set_option(F.OPT_GEMM_CTA_PAIRS, 1)
    assert F.fp8_get_last_device_error()[0] == 0


@pytest.mark.parametrize("k", [1, 8, 200, 1000])
def test_gemm_tensor_mn_major_ragged_k(k):
    """Both operands MN-major: K is the outer dimension of both tensor maps,
    so any K works (the last K slice is zero-filled by TMA)."""
    m, n = 256, 512
    qa, sa, qb, sb = per_tensor_operands(m, n, k, "e4m3", "e4m3", seed=k)
    c, e = OG.gemm(OG.dequant_operand(qa, "e4m3", sa), OG.dequant_operand(qb, "e4m3", sb))
    got = run_tensor_layout(qa, "e4m3", sa, qb, "e4m3", sb, True, True, "f32")
    ok, worst = OG.check(got, c, e, "f32")
    assert ok, worst


@pytest.mark.parametrize("shape", [(2048, 1024, 1024), (2000, 784, 1296), (8192, 2048, 2048)])
def test_gemm_tensor_grouped_linear_without_transposed_copies(shape):
    """The linear layer's three GEMMs on the row-major codes of x, W and g
    only: y = x W^T (K-major, K-major), dx = g W (K-major, W MN-major),
    dW = g^T x (g MN-major, x MN-major); the last shape is the full-size
    Float8 linear, checked on sampled outputs."""
    F = lib()
    t, d_in, d_out = shape
    seed = t + 1
    x = workloads.normal((t, d_in), 1.0, seed).to(torch.bfloat16).float().numpy()
    w = workloads.normal((d_out, d_in), 0.02, seed + 1).to(torch.bfloat16).float().numpy()
    g = workloads.normal((t, d_out), 1e-3, seed + 2).to(torch.bfloat16).float().numpy()
    qx, sx = OQ.quantize_tensor(x, "e4m3")
    qw, sw = OQ.quantize_tensor(w, "e4m3")
    qg, sg = OQ.quantize_tensor(g, "e5m2")
    dx_, dw_, dg_ = dev_u8(qx), dev_u8(qw), dev_u8(qg)
    s = [dev_f32(sx), dev_f32(sw), dev_f32(sg)]
    y = torch.empty((t, d_out), dtype=torch.bfloat16, device="cuda")
    dxo = torch.empty((t, d_in), dtype=torch.bfloat16, device="cuda")
    dwo = torch.empty((d_out, d_in), dtype=torch.float32, device="cuda")
    K, MN = F.K_MAJOR, F.MN_MAJOR
    F.fp8_gemm_tensor_grouped([
        F.gemm_problem(dx_, F.E4M3, dw_, F.E4M3, s[0], s[1], y),
        F.gemm_problem(dg_, F.E5M2, dw_, F.E4M3, s[2], s[1], dxo, b_layout=MN),
        F.gemm_problem(dg_, F.E5M2, dx_, F.E4M3, s[2], s[0], dwo, a_layout=MN, b_layout=MN),
    ])
    torch.cuda.synchronize()
    xd = OG.dequant_operand(qx, "e4m3", sx)
    wd = OG.dequant_operand(qw, "e4m3", sw)
    gd = OG.dequant_operand(qg, "e5m2", sg)
    cases = [(y, xd, wd, "bf16"), (dxo, gd, np.ascontiguousarray(wd.T), "bf16"),
             (dwo, np.ascontiguousarray(gd.T), np.ascontiguousarray(xd.T), "f32")]
    full = t * d_in * d_out <= 2048 ** 3
    for i, (out, a, b, odt) in enumerate(cases):
        got = out.float().cpu().numpy()
        if full:
            c, e = OG.gemm(a, b)
            ok, worst = OG.check(got, c, e, odt)
        else:
            rows, cols = sample_positions(a.shape[0], b.shape[0], 300, seed=i)
            c, e = OG.gemm_sampled(a, b, rows, cols)
            ok, worst = OG.check(got[rows, cols], c, e, odt)
        assert ok, (i, worst)
    assert F.fp8_get_last_device_error()[0] == 0


# ------------------------------------------------- MoE expert-grouped GEMM --

def expert_operands(experts, tokens, n, k, sfmt, seed, counts=None):
    act, w, drawn = workloads.moe_experts(experts, tokens, n, k, seed=seed)
    counts = drawn if counts is None else torch.tensor(counts, dtype=torch.int64)
    offsets = np.concatenate([[0], np.cumsum(counts.numpy())]).astype(np.int32)
    m = int(offsets[-1])
    act = act[:m]
    qa, sa = OQ.quantize_token_group(act.float().numpy(), "e4m3", sfmt)
    a_deq = OG.dequant_operand(qa, "e4m3", OQ.expand(OQ.group_scale_values(sa, sfmt), m, k, 1, 128))
    qbs, sbs, b_deq = [], [], []
    for e in range(experts):
        qb, sb = OQ.quantize_block(w[e].float().numpy(), "e4m3", sfmt)
        qbs.append(qb)
        sbs.append(np.asarray(sb))
        b_deq.append(OG.dequant_operand(qb, "e4m3",
                                        OQ.expand(OQ.group_scale_values(sb, sfmt), n, k, 128, 128)))
    c, e_ = OG.gemm_experts(a_deq, b_deq, offsets)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return (dev(qa), dev(np.asarray(sa).T), dev(np.stack(qbs)), dev(np.stack(sbs)),
            dev(offsets), c, e_, m)


@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
@pytest.mark.parametrize("case", [
    # experts, tokens, N, K, fixed counts (None: drawn)
    (8, 1000, 256, 1024, None),
    (5, 0, 384, 512, [0, 300, 1, 0, 129]),       # empty experts, a 1-row expert
    (3, 0, 200, 256, [130, 0, 257]),             # N not a multiple of 128
    (16, 4096, 512, 2048, None),
    (8, 4096, 2048, 1024, None),                 # 128 x 256 tiles
    (8, 4096, 2048, 7168, None),                 # the MoE workload bench.py times
])
def test_gemm_group_experts(sfmt, case):
    """Beyond M = 256 with N % 128 == 0 the UE8M0 case runs as the
    block-scaled kernel on per-expert-row-tile E8M0 words."""
    F = lib()
    experts, tokens, n, k, counts = case
    if counts is not None:
        tokens = sum(counts)
    qa, sa, qb, sb, offs, c, e, m = expert_operands(experts, tokens, n, k, sfmt, seed=experts + n,
                                                    counts=counts)
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    code = F.SCALE_F32 if sfmt == "f32" else F.SCALE_UE8M0
    F.fp8_gemm_group_experts(qa, sa, qb, sb, code, offs, out)
    torch.cuda.synchronize()
    ok, worst = OG.check(out.float().cpu().numpy(), c, e, "bf16")
    assert ok, worst
    assert F.fp8_get_last_device_error()[0] == 0


def test_gemm_group_experts_f32_cta_pairs():
    """FP32 expert-grouped rows on the CTA-pair kernel (256-row expert tiles):
    an empty expert, a 1-row expert, experts of 255 and 257 rows (a tile
    boundary just short of and just past the expert's end), ragged N (1000 =
    3 * 256 + 232), against the oracle, with pairs on and off (off: the
    one-CTA kernel)."""
    F = lib()
    counts = [700, 0, 1, 1100, 255, 257]
    n, k = 1000, 384
    qa, sa, qb, sb, offs, c, e, m = expert_operands(len(counts), sum(counts), n, k, "f32",
                                                    seed=77, counts=counts)
    try:
        for pairs in (1, 0):
            F.fp8_set_option(F.OPT_GEMM_CTA_PAIRS, pairs)
            out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
            F.fp8_gemm_group_experts(qa, sa, qb, sb, F.SCALE_F32, offs, out)
            torch.cuda.synchronize()
            ok, worst = OG.check(out.float().cpu().numpy(), c, e, "bf16")
            assert ok, (pairs, worst)
    finally:
        F.fp8_set_option(F.OPT_GEMM_CTA_PAIRS, 1)
    assert F.fp8_get_last_device_error()[0] == 0


# ------------------------------------------------------------ epilogue bias --

def _bias(n, seed):
    return (workloads.normal((n,), 0.5, seed)).numpy().astype(np.float32)


@pytest.mark.parametrize("mnk", [(2048, 2048, 1024), (200, 384, 1024), (16, 2048, 8192)])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_gemm_tensor_bias(mnk, out_dtype):
    """CTA-pair path, single-CTA path and the split-K cluster path, each with
    a bias added in the epilogue."""
    F = lib()
    m, n, k = mnk
    qa, sa, qb, sb = per_tensor_operands(m, n, k, "e4m3", "e4m3", seed=k + 11)
    bias = _bias(n, m + 1)
    out = torch.empty((m, n), dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32,
                      device="cuda")
    a, b = dev_u8(qa), dev_u8(qb)
    F.fp8_gemm_tensor_grouped([F.gemm_problem(a, F.E4M3, b, F.E4M3, dev_f32(sa), dev_f32(sb), out,
                                              bias=torch.from_numpy(bias).cuda())])
    torch.cuda.synchronize()
    c, e = OG.gemm(OG.dequant_operand(qa, "e4m3", sa), OG.dequant_operand(qb, "e4m3", sb))
    cb, eb, extra = OG.gemm_bias(c, e, bias)
    ok, worst = OG.check(out.float().cpu().numpy(), cb, eb, out_dtype, extra=extra)
    assert ok, worst


@pytest.mark.parametrize("m", [1, 200, 2048])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
def test_gemm_group_bias(m, sfmt):
    F = lib()
    n, k = 2048, 7168 if m == 1 else 2048
    qa, sa, qb, sb = group_operands(m, n, k, sfmt, seed=m + 3)
    c, e = group_reference(qa, sa, qb, sb, sfmt)
    bias = _bias(n, m + 7)
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    code = F.SCALE_F32 if sfmt == "f32" else F.SCALE_UE8M0
    F.fp8_gemm_group(dev_u8(qa), torch.from_numpy(np.ascontiguousarray(np.asarray(sa).T)).cuda(),
                     dev_u8(qb), torch.from_numpy(np.ascontiguousarray(sb)).cuda(), code, out,
                     bias=torch.from_numpy(bias).cuda())
    torch.cuda.synchronize()
    cb, eb, extra = OG.gemm_bias(c, e, bias)
    ok, worst = OG.check(out.float().cpu().numpy(), cb, eb, "bf16", extra=extra)
    assert ok, worst


@pytest.mark.parametrize("mnk", [(256, 384, 512), (200, 1000, 1024), (16, 2048, 8192)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_gemm_mx_per_row_global(mnk, out_dtype):
    """Two-level operands with a global factor per row of A and per row of B
    (per output column): the epilogue multiplies by S_a[m] * S_b[n].  The last
    shape runs the split-K cluster path."""
    F = lib()
    m, n, k = mnk
    a, b = workloads.two_level(seed=7, m=m, n=n, k=k)
    af, bf = a.float().numpy(), b.float().numpy()
    af[1] *= np.float32(2.0 ** -12)
    qa, la, ga = OQ.quantize_two_level(af, "e4m3", global_per_row=True)
    qb, lb, gb = OQ.quantize_two_level(bf, "e4m3", global_per_row=True)
    out = torch.empty((m, n), dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32,
                      device="cuda")
    F.fp8_gemm_mx_rows(dev_u8(qa), torch.from_numpy(mx_pack(la)).cuda(), dev_f32(ga), dev_u8(qb),
                       torch.from_numpy(mx_pack(lb)).cuda(), dev_f32(gb), out)
    torch.cuda.synchronize()
    c, e = mx_reference(qa, la, ga, qb, lb, gb)
    ok, worst = OG.check(out.float().cpu().numpy(), c, e, out_dtype)
    assert ok, worst
