"""Failure detection without a GPU fault: every device-side wait in the GEMM
kernels is bounded.  With the bound set to zero the first wait that is not
already satisfied runs out; the kernel records FP8_ERR_TIMEOUT (and which role
gave up) in the device error word, drains its in-flight copies, frees its
TMEM and exits.  The host reads the status, and the same CUDA context then
computes correctly again."""
import numpy as np
import pytest
import torch

from gpu_util import lib
from oracle import gemm as OG
from test_gpu_gemm import (group_operands, group_reference, per_tensor_operands, run_group,
                           run_tensor)

pytestmark = pytest.mark.gpu


def forced_timeout(fn):
    F = lib()
    assert F.fp8_get_last_device_error()[0] == 0
    F.fp8_set_option(F.OPT_WAIT_LIMIT_US, 0)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        F.fp8_set_option(F.OPT_WAIT_LIMIT_US, 2_000_000)
    return F.fp8_get_last_device_error()


@pytest.mark.parametrize("mnk", [(2048, 2048, 16384), (128, 256, 65536)])
def test_timeout_reported_then_context_usable(mnk):
    """(2048, 2048) runs on CTA pairs, (128, 256) on one CTA per tile with K
    split over a cluster.  A wait only runs out once it outlasts the
    barrier's own suspend window (mbarrier.try_wait blocks for a while before
    it reports "not yet"), so K is long enough that the epilogue waits for
    many k blocks."""
    F = lib()
    m, n, k = mnk
    qa, sa, qb, sb = per_tensor_operands(m, n, k, "e4m3", "e4m3", seed=5)
    rc, where = forced_timeout(lambda: run_tensor(qa, "e4m3", sa, qb, "e4m3", sb, "bf16"))
    assert rc == F.FP8_ERR_TIMEOUT and where in (1, 2, 3), (rc, where)
    assert F.fp8_get_last_device_error() == (0, 0)  # read clears the word
    c, e = OG.gemm(OG.dequant_operand(qa, "e4m3", sa), OG.dequant_operand(qb, "e4m3", sb))
    ok, worst = OG.check(run_tensor(qa, "e4m3", sa, qb, "e4m3", sb, "bf16"), c, e, "bf16")
    assert ok, worst
    assert F.fp8_get_last_device_error()[0] == 0


def run_group_noalloc(qa, sa, qb, sb, sfmt="f32"):
    F = lib()
    m, n = qa.shape[0], qb.shape[0]
    sa_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sa).T)).cuda()   # [G, M]
    sb_dev = torch.from_numpy(np.ascontiguousarray(np.asarray(sb))).cuda()     # [N/128, G]
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    F.fp8_gemm_group_noalloc(torch.from_numpy(qa).cuda(), sa_dev, torch.from_numpy(qb).cuda(),
                             sb_dev, 0 if sfmt == "f32" else 1, out)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def test_timeout_in_group_gemm_resets_split_k_counters():
    """The no-allocation entry point splits K over CTAs that meet through
    arrival counters in its fixed scratch; a timed-out call can leave counters
    behind, every call clears the counters it uses before its kernel runs, and
    the next calls (that entry point and the regular one) are correct.  UE8M0 scales keep one
    accumulator per tile, so the epilogue's first wait spans the CTA's whole
    share of K (M = 128 limits the split to eight 64-block shares), long
    enough to outlast the barrier's suspend window; the FP32 mode's waits
    are one 128-deep slice each and may all end within it."""
    F = lib()
    qa, sa, qb, sb = group_operands(128, 256, 65536, "ue8m0", seed=2)
    rc, where = forced_timeout(lambda: run_group_noalloc(qa, sa, qb, sb, "ue8m0"))
    assert rc == F.FP8_ERR_TIMEOUT, (rc, where)
    c, e = group_reference(qa, sa, qb, sb, "ue8m0")
    for _ in range(2):
        ok, worst = OG.check(run_group_noalloc(qa, sa, qb, sb, "ue8m0"), c, e, "bf16")
        assert ok, worst
    ok, worst = OG.check(run_group(qa, sa, qb, sb, "ue8m0"), c, e, "bf16")
    assert ok, worst


def test_timeout_in_few_row_kernel():
    """The few-row per-group kernel bounds its waits the same way.  Its K
    splits meet in a cluster exchange that every CTA still reaches after one
    of its waits gave up, so the call ends, the timeout is reported, and the
    next call is correct.  K 65536 over two weight tiles gives each CTA 64 k
    blocks, so the producer refills its ring many times."""
    F = lib()
    qa, sa, qb, sb = group_operands(16, 256, 65536, "f32", seed=3)
    rc, where = forced_timeout(lambda: run_group(qa, sa, qb, sb, "f32"))
    assert rc == F.FP8_ERR_TIMEOUT and where in (1, 2, 3), (rc, where)
    c, e = group_reference(qa, sa, qb, sb, "f32")
    ok, worst = OG.check(run_group(qa, sa, qb, sb, "f32"), c, e, "bf16")
    assert ok, worst
    assert F.fp8_get_last_device_error()[0] == 0


def test_timeout_in_multi_tensor_quantize():
    """The cooperative quantize waits on its copies and on the other CTAs'
    amax shares; with the bound at zero one of them runs out, the kernel
    reports it and exits, and the next call is exact."""
    F = lib()
    import workloads
    from gpu_util import FMT, f32_bits, to_np_u8
    from oracle import quantize as OQ
    x = workloads.normal((2048, 2048), 1.0, 7).to(torch.bfloat16).cuda()
    q = torch.empty((2048, 2048), dtype=torch.uint8, device="cuda")
    scale = torch.zeros(1, device="cuda")
    sync = torch.zeros(F.QUANT_SYNC_WORDS, dtype=torch.int32, device="cuda")
    items = [F.quant_item(x, FMT["e4m3"], q, scale)]
    rc, where = forced_timeout(lambda: F.fp8_quantize_tensors(items, sync))
    assert rc == F.FP8_ERR_TIMEOUT and 11 <= where <= 15, (rc, where)
    F.fp8_quantize_tensors(items, sync)
    torch.cuda.synchronize()
    ref_q, ref_s = OQ.quantize_tensor(x.float().cpu().numpy(), "e4m3")
    assert f32_bits(scale.item()) == f32_bits(ref_s)
    assert np.array_equal(to_np_u8(q), ref_q)
    assert F.fp8_get_last_device_error()[0] == 0
