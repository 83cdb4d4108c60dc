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


@pytest.mark.parametrize("mnk", [(2048, 2048, 16384), (128, 256, 16384)])
def test_timeout_reported_then_context_usable(mnk):
    """(2048, 2048) runs on CTA pairs, (128, 256) on one CTA per tile with
    split K."""
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


def test_timeout_in_group_gemm_resets_split_k_counters():
    """A timed-out split-K call can leave arrival counters behind; reading the
    error resets them, so the next call on the same stream is correct."""
    F = lib()
    qa, sa, qb, sb = group_operands(16, 2048, 7168, "f32", seed=2)
    rc, where = forced_timeout(lambda: run_group(qa, sa, qb, sb, "f32"))
    assert rc == F.FP8_ERR_TIMEOUT, (rc, where)
    c, e = group_reference(qa, sa, qb, sb, "f32")
    for _ in range(2):
        ok, worst = OG.check(run_group(qa, sa, qb, sb, "f32"), c, e, "bf16")
        assert ok, worst
