"""(32, 32) weight blocks with FP32 scales (Transformers fine-grained FP8, 八:
weight_block_size (32, 32); 四: float scale_fmt, the default) and their 1 x
32 activation groups, against the oracle.

Quantizers: codes and scales bit-exact (ragged sizes, an all-zero group and
block, bf16 and fp32 inputs).  GEMM: operands quantized by the oracle and
uploaded, so the GEMM is checked on its own -- every output element within
|gpu - oracle| <= 1e-3 * sum |a||b| + one bf16 ulp; small, ragged, split-K
(small M) and a full fine-grained shape (M 4096, N 2048, K 7168) on sampled
outputs.  Then the whole path (GPU quantizers + GEMM) on the fine-grained
workload's activations and weights."""
import functools

import numpy as np
import pytest
import torch

import workloads
from gpu_util import lib, sample_positions, to_np_u8
from oracle import gemm as OG
from oracle import quantize as OQ

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(1, 32), (5, 304), (130, 1024), (64, 7168)])
@pytest.mark.parametrize("sfmt", ["f32", "ue8m0"])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_token_group32(shape, sfmt, dt):
    F = lib()
    m, k = shape
    act, _ = workloads.fine_grained(m, k=k, n=128)
    x = act.to(dt)
    if m > 2:
        x[2, :32] = 0.0  # an all-zero group
    xf = x.float().numpy()
    g = (k + 31) // 32
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    sc = torch.empty((g, m), dtype=torch.float32 if sfmt == "f32" else torch.uint8, device="cuda")
    F.fp8_quantize_token_group32(x.cuda(), F.E4M3, 0 if sfmt == "f32" else 1, q, sc)
    torch.cuda.synchronize()
    ref_q, ref_s = OQ.quantize_token_group(xf, "e4m3", sfmt, group=32)
    assert np.array_equal(to_np_u8(q), ref_q)
    got = sc.cpu().numpy().T
    if sfmt == "f32":
        assert np.array_equal(got.view(np.uint32), np.asarray(ref_s, np.float32).view(np.uint32))
    else:
        assert np.array_equal(got, ref_s)


@pytest.mark.parametrize("shape", [(32, 32), (70, 96), (300, 1024), (512, 2048)])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_block32_f32(shape, dt, fmt):
    F = lib()
    n, k = shape
    w = workloads.normal((n, k), 0.02, seed=n + k).to(dt)
    if n >= 64 and k >= 64:
        w[32:64, 32:64] = 0.0  # an all-zero block
    wf = w.float().numpy()
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    sc = torch.empty(((n + 31) // 32, k // 32), dtype=torch.float32, device="cuda")
    F.fp8_quantize_block32_f32(w.cuda(), F.E4M3 if fmt == "e4m3" else F.E5M2, q, sc)
    torch.cuda.synchronize()
    ref_q, ref_s = OQ.quantize_block(wf, fmt, "f32", block=32)
    assert np.array_equal(to_np_u8(q), ref_q)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32),
                          np.asarray(ref_s, np.float32).view(np.uint32))


@functools.lru_cache(maxsize=4)
def weights32(n, k, seed):
    """The oracle's (32, 32) quantization of the workload's weights (shared
    by the tests that use the same shape)."""
    _, w = workloads.fine_grained(1, k=k, n=n, seed=seed)
    return OQ.quantize_block(w.float().numpy(), "e4m3", "f32", block=32)


def operands32(m, n, k, seed):
    act, _ = workloads.fine_grained(m, k=k, n=8, seed=seed)
    qa, sa = OQ.quantize_token_group(act.float().numpy(), "e4m3", "f32", group=32)
    qb, sb = weights32(n, k, seed)
    return qa, sa, qb, sb


def deq32(qa, sa, qb, sb, m, n, k):
    a = OG.dequant_operand(qa, "e4m3", OQ.expand(np.asarray(sa, np.float64), m, k, 1, 32))
    b = OG.dequant_operand(qb, "e4m3", OQ.expand(np.asarray(sb, np.float64), n, k, 32, 32))
    return a, b


def run32(qa, sa, qb, sb):
    F = lib()
    m, n = qa.shape[0], qb.shape[0]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    F.fp8_gemm_group32(dev(qa), dev(np.asarray(sa, np.float32).T), dev(qb),
                       dev(np.asarray(sb, np.float32)), out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("mnk", [(128, 128, 128), (1, 64, 256), (130, 300, 1024),
                                 (16, 2048, 7168), (200, 520, 2048)])
def test_gemm_group32(mnk):
    m, n, k = mnk
    qa, sa, qb, sb = operands32(m, n, k, seed=2)
    got = run32(qa, sa, qb, sb).float().cpu().numpy()
    c, e = OG.gemm(*deq32(qa, sa, qb, sb, m, n, k))
    ok, worst = OG.check(got, c, e, "bf16")
    assert ok, worst
    rc, where = lib().fp8_get_last_device_error()
    assert rc == 0, (rc, where)


def test_gemm_group32_fine_grained_size_sampled():
    m, n, k = 4096, 2048, 7168
    qa, sa, qb, sb = operands32(m, n, k, seed=2)
    out = run32(qa, sa, qb, sb)
    rows, cols = sample_positions(m, n, 2048, 5)
    a, b = deq32(qa[rows], np.asarray(sa)[rows], qb, sb, len(rows), n, k)
    cref, eref = OG.gemm_sampled(a, b[cols], np.arange(len(rows)), np.arange(len(cols)))
    ri, ci = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    ok, worst = OG.check(out[ri, ci].double().cpu().numpy(), cref, eref, "bf16")
    assert ok, worst


def test_block32_path_end_to_end():
    """GPU quantizers then the GEMM, on the fine-grained workload's
    distributions (M 256, N 512, K 7168):
    codes and scales as the oracle's, the product within the bound."""
    F = lib()
    m, n, k = 256, 512, 7168
    act, w = workloads.fine_grained(m, k=k, n=n)
    qa = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    sa = torch.empty((k // 32, m), dtype=torch.float32, device="cuda")
    qb = torch.empty((n, k), dtype=torch.uint8, device="cuda")
    sb = torch.empty((n // 32, k // 32), dtype=torch.float32, device="cuda")
    F.fp8_quantize_token_group32(act.cuda(), F.E4M3, F.SCALE_F32, qa, sa)
    F.fp8_quantize_block32_f32(w.cuda(), F.E4M3, qb, sb)
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    F.fp8_gemm_group32(qa, sa, qb, sb, out)
    torch.cuda.synchronize()
    ra, rsa = OQ.quantize_token_group(act.float().numpy(), "e4m3", "f32", group=32)
    rb, rsb = OQ.quantize_block(w.float().numpy(), "e4m3", "f32", block=32)
    assert np.array_equal(to_np_u8(qa), ra) and np.array_equal(to_np_u8(qb), rb)
    assert np.array_equal(sa.cpu().numpy().T, np.asarray(rsa, np.float32))
    assert np.array_equal(sb.cpu().numpy(), np.asarray(rsb, np.float32))
    c, e = OG.gemm(*deq32(ra, rsa, rb, rsb, m, n, k))
    ok, worst = OG.check(out.float().cpu().numpy(), c, e, "bf16")
    assert ok, worst
