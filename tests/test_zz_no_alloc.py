"""fp8_gemm_group_noalloc: the per-K-group GEMM for callers that cannot let
the library allocate device memory (runtimes that reserve all device memory
up front in their own pool, code that must never stall on the allocator).
Where it splits K, its scratch is a fixed array inside the library instead of
memory allocated on first use.

Checked through the C ABI on the same inputs, two calls in a row (the array
keeps the previous call's contents, so the second call shows that what must
start at zero is cleared): against the oracle's float64 product within the
GEMM bound, and against the regular fp8_gemm_group within the same bound.
Kept in a file of its own that pytest collects last; it passes alone in a
fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import lib
from oracle import gemm as OG
from oracle import quantize as OQ

pytestmark = pytest.mark.gpu


def operands(m, n, k, sfmt):
    act, w = workloads.fine_grained(m, k=k, n=n)
    qa, sa = OQ.quantize_token_group(act.float().numpy(), "e4m3", sfmt)
    qb, sb = OQ.quantize_block(w.float().numpy(), "e4m3", sfmt)
    a = OG.dequant_operand(qa, "e4m3", OQ.expand(OQ.group_scale_values(sa, sfmt), m, k, 1, 128))
    b = OG.dequant_operand(qb, "e4m3", OQ.expand(OQ.group_scale_values(sb, sfmt), n, k, 128, 128))
    c, e = OG.gemm(a, b)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return dev(qa), dev(np.asarray(sa).T), dev(qb), dev(np.asarray(sb)), c, e


@pytest.mark.parametrize("m,n,k,sfmt", [(16, 2048, 7168, "f32"), (1, 2048, 7168, "ue8m0"),
                                        (128, 2048, 7168, "f32"), (200, 384, 1024, "ue8m0")])
def test_noalloc_matches_regular_entry_point(m, n, k, sfmt):
    F = lib()
    qa, sa, qb, sb, c, e = operands(m, n, k, sfmt)
    code = F.SCALE_F32 if sfmt == "f32" else F.SCALE_UE8M0
    ref = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    F.fp8_gemm_group(qa, sa, qb, sb, code, ref)
    torch.cuda.synchronize()
    want = ref.float().cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        F.fp8_gemm_group_noalloc(qa, sa, qb, sb, code, out)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        ok, worst = OG.check(got, c, e, "bf16")
        assert ok, ("oracle", call, worst)
        ok, worst = OG.check(got, want, e, "bf16")
        assert ok, ("fp8_gemm_group", call, worst)
    rc, where = F.fp8_get_last_device_error()
    assert rc == 0, (rc, where)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """M 128, N 6144, K 7168 with UE8M0 scales (128-wide tiles at this M)
    splits K three ways: 9.4 MB of partials, more than the 8 MiB the fixed
    scratch holds."""
    F = lib()
    m, n, k = 128, 6144, 7168
    qa = torch.zeros((m, k), dtype=torch.uint8, device="cuda")
    qb = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
    sa = torch.full((k // 128, m), 127, dtype=torch.uint8, device="cuda")
    sb = torch.full((n // 128, k // 128), 127, dtype=torch.uint8, device="cuda")
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(F.Fp8Error) as exc:
        F.fp8_gemm_group_noalloc(qa, sa, qb, sb, F.SCALE_UE8M0, out)
    assert exc.value.status == F.FP8_ERR_SCRATCH_LIMIT
    assert "scratch" in str(exc.value)
