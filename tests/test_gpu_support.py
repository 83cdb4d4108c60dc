"""The training step's support kernels against the oracle.

* SwiGLU fused with delayed-scaling quantization (Flax guide 2.3: quantize
  with the stored scale, record the current amax): the plain kernels' bf16
  values are within one bf16 ulp of the oracle's SwiGLU, and the fused codes
  and amaxes equal, bit for bit, the oracle quantizing those bf16 values with
  the given scale (both sides decide each code from the same bf16 value).
  Scales that clip, scales outside the reciprocal-quotient range, ragged and
  empty sizes.
* Multi-tensor AdamW with the step counter on the device: every tensor
  against the oracle's AdamW at the advanced step, over several steps, with
  an empty item; with the next step's weight codes: the codes and amax of
  the updated bf16 weights bit-exact against the oracle quantizing them with
  the given scale.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import lib, to_np_u8
from oracle import gemm as OG
from oracle import quantize as OQ
from oracle import training as OT

pytestmark = pytest.mark.gpu


def f32(t):
    return t.detach().float().cpu().numpy()


def bf16_ulps(gpu, ref):
    ref = np.asarray(ref, np.float64)
    gpu = np.asarray(gpu, np.float64)
    tol = np.maximum(OG.bf16_ulp(ref), OG.bf16_ulp(gpu))
    return float(np.max(np.abs(gpu - ref) / tol)) if ref.size else 0.0


def inputs(n, seed):
    h = (workloads.normal((n,), 3.0, seed)).to(torch.bfloat16).cuda()
    u = (workloads.normal((n,), 1.0, seed + 1)).to(torch.bfloat16).cuda()
    da = (workloads.normal((n,), 1e-3, seed + 2)).to(torch.bfloat16).cuda()
    return h, u, da


SIZES = [0, 8, 4104, (1 << 20) + 24]
# (forward scale, backward scales): moderate; clipping (small scales); a
# scale below the reciprocal-quotient range (IEEE division path)
SCALES = [(0.02, (2e-5, 3e-5)), (0.001, (1e-8, 5e-9)), (2.0 ** -100, (2.0 ** -100, 1e-6))]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("scales", SCALES)
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_swiglu_forward_quantize(n, scales, fmt):
    F = lib()
    code = F.E4M3 if fmt == "e4m3" else F.E5M2
    h, u, _ = inputs(max(n, 8), seed=n + 3)
    h, u = h[:n].contiguous(), u[:n].contiguous()
    s = torch.tensor([scales[0]], dtype=torch.float32, device="cuda")
    a = torch.empty_like(h)
    q = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
    amax = torch.full((1,), -1.0, device="cuda")
    F.fp8_swiglu_forward(h, u, a)
    F.fp8_swiglu_forward_quantize(h, u, code, s, q, amax)
    torch.cuda.synchronize()
    a_bf = f32(a)
    assert bf16_ulps(a_bf, OT.swiglu_forward(f32(h), f32(u))) <= 1.0
    want = OQ.quantize_with_scale(a_bf, np.float32(scales[0]), fmt)
    assert np.array_equal(to_np_u8(q), want)
    assert np.float32(amax.item()) == OQ.amax(a_bf)


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("scales", SCALES)
def test_swiglu_backward_quantize(n, scales):
    F = lib()
    h, u, da = inputs(max(n, 8), seed=n + 7)
    h, u, da = h[:n].contiguous(), u[:n].contiguous(), da[:n].contiguous()
    sh = torch.tensor([scales[1][0]], dtype=torch.float32, device="cuda")
    su = torch.tensor([scales[1][1]], dtype=torch.float32, device="cuda")
    dh, du = torch.empty_like(h), torch.empty_like(h)
    qh = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
    qu = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
    am = torch.full((2,), -1.0, device="cuda")
    F.fp8_swiglu_backward(da, h, u, dh, du)
    F.fp8_swiglu_backward_quantize(da, h, u, F.E5M2, sh, su, qh, qu, am[0:1], am[1:2])
    torch.cuda.synchronize()
    dh_ref, du_ref = OT.swiglu_backward(f32(da), f32(h), f32(u))
    assert bf16_ulps(f32(dh), dh_ref) <= 1.0
    assert bf16_ulps(f32(du), du_ref) <= 1.0
    for q, bf, s_, k in ((qh, f32(dh), scales[1][0], 0), (qu, f32(du), scales[1][1], 1)):
        assert np.array_equal(to_np_u8(q), OQ.quantize_with_scale(bf, np.float32(s_), "e5m2"))
        assert np.float32(am[k].item()) == OQ.amax(bf)


def test_swiglu_quantize_without_amax_and_argument_checks():
    F = lib()
    h, u, da = inputs(64, seed=11)
    s = torch.tensor([0.05], device="cuda")
    q1 = torch.empty(64, dtype=torch.uint8, device="cuda")
    q2 = torch.empty(64, dtype=torch.uint8, device="cuda")
    F.fp8_swiglu_forward_quantize(h, u, F.E4M3, s, q1)
    a = torch.empty_like(h)
    F.fp8_swiglu_forward(h, u, a)
    torch.cuda.synchronize()
    assert np.array_equal(to_np_u8(q1), OQ.quantize_with_scale(f32(a), np.float32(0.05), "e4m3"))
    am = torch.zeros(1, device="cuda")
    with pytest.raises(F.Fp8Error):  # one amax without the other
        F.fp8_swiglu_backward_quantize(da, h, u, F.E5M2, s, s, q1, q2, am, None)
    with pytest.raises(F.Fp8Error):  # amax aliasing the scale
        F.fp8_swiglu_forward_quantize(h, u, F.E4M3, s, q1, s)


def test_adamw_multi_device_step():
    F = lib()
    sizes = [4096, 0, 1000, 65536 + 4]
    rng = np.random.default_rng(5)
    host = []
    dev = []
    for n in sizes:
        p = (rng.standard_normal(n) * 0.02).astype(np.float32)
        host.append([p.astype(np.float64), np.zeros(n), np.zeros(n)])
        t = [torch.from_numpy(p).cuda(), torch.empty(n, device="cuda"),
             torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda"),
             torch.empty(n, dtype=torch.bfloat16, device="cuda")]
        dev.append(t)
    step = torch.zeros(1, dtype=torch.int64, device="cuda")
    items = [F.adamw_item(p, g, m, v, pb) for p, g, m, v, pb in dev]
    for t in range(1, 6):
        grads = [(rng.standard_normal(n) * 10.0 ** rng.integers(-6, 0)).astype(np.float32)
                 for n in sizes]
        for (p, g, m, v, pb), gr in zip(dev, grads):
            g.copy_(torch.from_numpy(gr))
        if t % 2:
            F.fp8_adamw_multi(items, step)
        else:  # the advance alone, then the update at that t
            F.fp8_adamw_multi([], step)
            F.fp8_adamw_multi(items[:2], step, advance=False)
            F.fp8_adamw_multi(items[2:], step, advance=False)
        torch.cuda.synchronize()
        assert int(step.item()) == t
        for k, n in enumerate(sizes):
            p_ref, m_ref, v_ref = OT.adamw_step(*host[k][:1], grads[k].astype(np.float64),
                                                host[k][1], host[k][2], step=t)
            host[k] = [p_ref, m_ref, v_ref]
            p, g, m, v, pb = dev[k]
            assert np.allclose(p.double().cpu().numpy(), p_ref, rtol=2e-6, atol=1e-9), (t, k)
            assert np.allclose(m.double().cpu().numpy(), m_ref, rtol=1e-5,
                               atol=1e-6 * (np.max(np.abs(m_ref)) if n else 0))
            assert torch.equal(pb, p.to(torch.bfloat16))
            # the next step continues from the GPU's own state
            host[k] = [p.double().cpu().numpy(), m.double().cpu().numpy(),
                       v.double().cpu().numpy()]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_adamw_multi_writes_the_next_weight_codes(fmt):
    """The fused quantization of fp8_adamw_multi: items with codes (a scale
    in the reciprocal-quotient range, one below it, one that clips), an item
    without, an empty item; codes and amax bit-exact against the oracle's
    quantize_with_scale / amax of the updated bf16 weights."""
    F = lib()
    code = F.E4M3 if fmt == "e4m3" else F.E5M2
    sizes = [4096, 1000, 0, 65536 + 4, 2048]
    scales = [3e-4, 2.0 ** -100, 1.0, 1e-5, 0.0]  # the fourth clips; the last has no codes
    rng = np.random.default_rng(17)
    dev = []
    for n in sizes:
        p = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).cuda()
        g = torch.from_numpy((rng.standard_normal(n) * 1e-3).astype(np.float32)).cuda()
        dev.append([p, g, torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda"),
                    torch.empty(n, dtype=torch.bfloat16, device="cuda"),
                    torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")])
    sc = torch.tensor(scales, dtype=torch.float32, device="cuda")
    am = torch.full((len(sizes),), -1.0, device="cuda")
    items = []
    for k, (p, g, m, v, pb, q) in enumerate(dev):
        kw = dict(q=q, q_scale=sc[k:k + 1], q_amax=am[k:k + 1], q_fmt=code) if k < 4 else {}
        items.append(F.adamw_item(p, g, m, v, pb, **kw))
    step = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in range(2):
        F.fp8_adamw_multi(items, step)
        torch.cuda.synchronize()
        for k, (p, g, m, v, pb, q) in enumerate(dev):
            assert torch.equal(pb, p.to(torch.bfloat16))
            if k >= 4:
                assert np.all(to_np_u8(q) == 0xAB)  # no codes asked: untouched
                continue
            if sizes[k] == 0:
                continue  # an empty item's codes pointer is null: nothing is written
            wb = f32(pb)
            assert np.array_equal(to_np_u8(q), OQ.quantize_with_scale(wb, np.float32(scales[k]),
                                                                      fmt)), (t, k)
            assert np.float32(am[k].item()) == OQ.amax(wb), (t, k)
