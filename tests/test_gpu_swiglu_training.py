"""FP8 SwiGLU training with delayed scaling: GPU step against the oracle,
teacher-forced (each stage is checked on the GPU's own inputs to it).

Per step: every quantized operand bit-exact against the oracle's delayed-
scaling state machine (which also fixes the scale used); the nine GEMMs
within the GEMM bound; SwiGLU forward/backward within one bf16 ulp; AdamW
within fp32 rounding; the nine amax histories exactly.  16 steps at a reduced
size (T 512, d 256, ffn 896).

The trainer quantizes a, dh and du inside the SwiGLU passes (the bf16 tensors
are never written).  Their bf16 values are recomputed here by the plain
SwiGLU kernels from the GPU's own h, u and da, and the oracle quantizes those:
the fused codes must equal the oracle's bit for bit, and the plain kernels'
values must be within one bf16 ulp of the oracle's SwiGLU."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import lib, to_np_u8
from oracle import delayed as OD
from oracle import gemm as OG
from oracle import quantize as OQ
from oracle import training as OT

pytestmark = pytest.mark.gpu

T, D, FFN, STEPS = 512, 256, 896, 16


def f32(t):
    return t.detach().float().cpu().numpy()


def bf16_close(gpu, ref):
    ref = np.asarray(ref, np.float64)
    gpu = np.asarray(gpu, np.float64)
    tol = np.maximum(OG.bf16_ulp(ref), OG.bf16_ulp(gpu))
    return float(np.max(np.abs(gpu - ref) / tol))


def swiglu_bf16(tr):
    """The bf16 a, dh, du the fused passes quantized, recomputed by the plain
    SwiGLU kernels from the trainer's h, u and da."""
    F = lib()
    a = torch.empty_like(tr.h)
    dh, du = torch.empty_like(tr.h), torch.empty_like(tr.h)
    F.fp8_swiglu_forward(tr.h, tr.u, a)
    F.fp8_swiglu_backward(tr.da, tr.h, tr.u, dh, du)
    return a, dh, du


@pytest.mark.parametrize("fuse_forward", [True, False])
def test_swiglu_training_teacher_forced(fuse_forward):
    """The weight gradients are stored (fuse_optimizer=False) so that the
    three dW GEMMs and the standalone AdamW are checked on their own; the
    forward runs as the gated epilogue or as the standalone fused pass."""
    lib()
    from fp8_quantized_gemm_gb300.mlp import (A2, G1, G2, G3, K1, K2, K3, X1, X3,
                                              SwiGLUTrainer)
    x, w1, w3, w2 = workloads.swiglu(d=D, ffn=FFN, tokens=T)
    tr = SwiGLUTrainer(w1.cuda(), w3.cuda(), w2.cuda(), tokens=T, fuse_forward=fuse_forward,
                       fuse_optimizer=False)
    xd = x.cuda()
    xf = f32(x)
    st = [OD.DelayedState.initial(1024) for _ in range(9)]
    fmt = {i: ("e5m2" if i in (G1, G3, G2) else "e4m3") for i in range(9)}
    for t in range(STEPS):
        dy = workloads.swiglu_grad(t, tokens=T, d=D).cuda()
        wb = [f32(w) for w in tr.w_bf]
        wm = [w.double().cpu().numpy() for w in tr.w_master]
        mm = [w.double().cpu().numpy() for w in tr.m]
        vv = [w.double().cpu().numpy() for w in tr.v]
        sc_gpu = tr.scale.cpu().numpy().copy()
        tr.forward_backward(xd, dy)
        a_bf, dh_bf, du_bf = swiglu_bf16(tr)
        torch.cuda.synchronize()

        # quantized operands: oracle in_q on the tensor each slot quantizes
        inputs = {X1: xf, X3: xf, K1: wb[0], K3: wb[1], K2: wb[2], A2: f32(a_bf),
                  G2: f32(dy), G1: f32(dh_bf), G3: f32(du_bf)}
        codes, scales = {}, {}
        for i in range(9):
            q, s_used, st[i] = OD.in_q(inputs[i], fmt[i], st[i])
            assert np.float32(sc_gpu[i]) == s_used, (t, i)
            codes[i], scales[i] = q, s_used
        gpu_q = {X1: tr.xq, K1: tr.w1q, K3: tr.w3q, K2: tr.w2q, A2: tr.aq, G2: tr.dyq,
                 G1: tr.dhq, G3: tr.duq}
        for i, qg in gpu_q.items():
            assert np.array_equal(to_np_u8(qg), codes[i]), (t, i)

        def deq(i, transpose=False):
            c = codes[i].T if transpose else codes[i]
            return OG.dequant_operand(c, fmt[i], scales[i])

        # the nine GEMMs
        checks = [
            ("h", tr.h, deq(X1), deq(K1), "bf16"),
            ("u", tr.u, deq(X1), deq(K3), "bf16"),
            ("y", tr.y, deq(A2), deq(K2), "bf16"),
            ("da", tr.da, deq(G2), deq(K2, True), "bf16"),
            ("dW2", tr.dw[2], deq(G2, True), deq(A2, True), "f32"),
            ("dW1", tr.dw[0], deq(G1, True), deq(X1, True), "f32"),
            ("dW3", tr.dw[1], deq(G3, True), deq(X1, True), "f32"),
        ]
        for name, out, a, b, odt in checks:
            c, e = OG.gemm(a, b)
            ok, worst = OG.check(f32(out), c, e, odt)
            assert ok, (t, name, worst)
        c1, e1 = OG.gemm(deq(G1), deq(K1, True))
        c2, e2 = OG.gemm(deq(G3), deq(K3, True))
        ok, worst = OG.check(f32(tr.dx), c1 + c2, e1 + e2, "f32")
        assert ok, (t, "dx", worst)

        # SwiGLU on the GPU's own h, u, da
        h, u, da = f32(tr.h), f32(tr.u), f32(tr.da)
        assert bf16_close(f32(a_bf), OT.swiglu_forward(h, u)) <= 1.0, t
        dh_ref, du_ref = OT.swiglu_backward(da, h, u)
        assert bf16_close(f32(dh_bf), dh_ref) <= 1.0, t
        assert bf16_close(f32(du_bf), du_ref) <= 1.0, t

        # optimizer and histories
        dws = [w.double().cpu().numpy() for w in tr.dw]
        tr.optimizer_and_state()
        torch.cuda.synchronize()
        for i in range(3):
            p_ref, m_ref, v_ref = OT.adamw_step(wm[i], dws[i], mm[i], vv[i], step=t + 1)
            p_gpu = tr.w_master[i].double().cpu().numpy()
            assert np.allclose(p_gpu, p_ref, rtol=2e-6, atol=1e-9), (t, i)
            # fp32 moments: b*m + (1-b)*g can cancel, so the absolute error is
            # a couple of fp32 ulps of the larger term, not of the result
            assert np.allclose(tr.m[i].double().cpu().numpy(), m_ref, rtol=1e-5,
                               atol=1e-6 * np.max(np.abs(m_ref)))
            assert np.allclose(tr.v[i].double().cpu().numpy(), v_ref, rtol=1e-5,
                               atol=1e-6 * np.max(np.abs(v_ref)))
            assert torch.equal(tr.w_bf[i], tr.w_master[i].to(torch.bfloat16))
        hist = tr.hist.cpu().numpy()
        for i in range(9):
            assert np.array_equal(hist[i].view(np.uint32), st[i].history.view(np.uint32)), (t, i)


def test_swiglu_training_automatic_weight_scaling():
    """MOSS automatic scaling (section 5, eq. 10) in the training step: each
    weight's scale is (amax_0 + lr * t) / MAX from the amax at the last
    max-reduction, t steps ago; the reduction is redone every 3 steps here."""
    lib()
    from fp8_quantized_gemm_gb300.mlp import K1, K2, K3, SwiGLUTrainer
    x, w1, w3, w2 = workloads.swiglu(d=D, ffn=FFN, tokens=T)
    tr = SwiGLUTrainer(w1.cuda(), w3.cuda(), w2.cuda(), tokens=T, weight_scaling="auto",
                       rescale_interval=3)
    xd = x.cuda()
    slots = (K1, K3, K2)
    qs = ((lambda: tr.w1q), (lambda: tr.w3q), (lambda: tr.w2q))
    amax0 = [float(np.max(np.abs(f32(w)))) for w in tr.w_bf]
    t_since = 0
    for step in range(7):
        wb = [f32(w) for w in tr.w_bf]
        tr.forward_backward(xd, workloads.swiglu_grad(step, tokens=T, d=D).cuda())
        torch.cuda.synchronize()
        sc = tr.scale.cpu().numpy()
        for i in range(3):
            want = OT.auto_weight_scale(amax0[i], 1e-4, t_since, 448.0)
            assert np.float32(sc[slots[i]]) == want, (step, i)
            assert np.array_equal(to_np_u8(qs[i]()), OQ.quantize_with_scale(wb[i], want, "e4m3"))
        tr.optimizer_and_state()
        torch.cuda.synchronize()
        t_since += 1
        if t_since == 3:  # max-reduction on the updated bf16 weights
            t_since = 0
            amax0 = [float(np.max(np.abs(f32(w)))) for w in tr.w_bf]
        assert np.allclose(tr.w_amax0.cpu().numpy(), amax0, rtol=0, atol=0)


def _bf16(v):
    """float64 -> nearest fp32 -> nearest bf16, as the GPU rounds its fp32
    results for a bf16 output."""
    t = torch.from_numpy(np.asarray(v, dtype=np.float32))
    return t.to(torch.bfloat16).float().numpy().astype(np.float64)


def _fp32(v):
    return np.asarray(v, dtype=np.float32).astype(np.float64)


def oracle_trajectory(x, w_init, dys, steps):
    """The oracle's own 16-step run of the FP8 SwiGLU training step (delayed
    scaling, E4M3 forward / E5M2 gradients, Flax guide 2.3 and 3.3; AdamW):
    nothing is taken from the GPU.  Returns per-step scales, the final
    float64 master weights, and the last step's y and dx."""
    from fp8_quantized_gemm_gb300.mlp import A2, G1, G2, G3, K1, K2, K3, X1, X3
    st = [OD.DelayedState.initial(1024) for _ in range(9)]
    master = [np.asarray(w, np.float64) for w in w_init]
    m = [np.zeros_like(w) for w in master]
    v = [np.zeros_like(w) for w in master]
    w_bf = [np.asarray(w, np.float64) for w in w_init]
    scales = []
    y = dx = None
    for t in range(steps):
        used = [None] * 9

        def inq(i, tensor, fmt):
            q, s, st[i] = OD.in_q(np.asarray(tensor, np.float32), fmt, st[i])
            used[i] = s
            return OG.dequant_operand(q, fmt, s)

        xd = inq(X1, x, "e4m3")
        inq(X3, x, "e4m3")
        w1d, w3d, w2d = inq(K1, w_bf[0], "e4m3"), inq(K3, w_bf[1], "e4m3"), inq(K2, w_bf[2], "e4m3")
        h = _bf16(xd @ w1d.T)
        u = _bf16(xd @ w3d.T)
        ad = inq(A2, _bf16(OT.swiglu_forward(h, u)), "e4m3")
        y = _bf16(ad @ w2d.T)
        dyd = inq(G2, dys[t], "e5m2")
        da = _bf16(dyd @ w2d)
        dw2 = _fp32(dyd.T @ ad)
        dh, du = OT.swiglu_backward(da, h, u)
        dhd = inq(G1, _bf16(dh), "e5m2")
        dud = inq(G3, _bf16(du), "e5m2")
        dx = _fp32(dhd @ w1d + dud @ w3d)
        dws = [_fp32(dhd.T @ xd), _fp32(dud.T @ xd), dw2]
        for i in range(3):
            master[i], m[i], v[i] = OT.adamw_step(master[i], dws[i], m[i], v[i], step=t + 1)
            w_bf[i] = _bf16(master[i])
        scales.append(np.asarray(used, np.float64))
    return scales, master, y, dx


@pytest.mark.parametrize("fuse_optimizer", [False, True])
def test_swiglu_training_16_steps_free_running(fuse_optimizer):
    """16 steps of the GPU trainer against the oracle's own trajectory from the
    same initial weights and gradients (not teacher-forced: the two runs only
    share their inputs).  Rounding-boundary flips of single codes are expected
    between them, so the check is on what they must agree on: every scale used
    within 1%, the 16-step weight updates within 1% (relative Frobenius
    norm), and the last step's y and dx within 1%."""
    lib()
    from fp8_quantized_gemm_gb300.mlp import SwiGLUTrainer
    x, w1, w3, w2 = workloads.swiglu(d=D, ffn=FFN, tokens=T)
    dys = [workloads.swiglu_grad(t, tokens=T, d=D) for t in range(STEPS)]
    w_init = [f32(w).astype(np.float64) for w in (w1, w3, w2)]
    tr = SwiGLUTrainer(w1.cuda(), w3.cuda(), w2.cuda(), tokens=T, fuse_optimizer=fuse_optimizer)
    xd = x.cuda()
    gpu_scales = []
    for t in range(STEPS):
        gpu_scales.append(tr.scale.double().cpu().numpy().copy())
        tr.step(xd, dys[t].cuda())
    torch.cuda.synchronize()
    rc, where = lib().fp8_get_last_device_error()
    assert rc == 0, (rc, where)
    ref_scales, ref_master, ref_y, ref_dx = oracle_trajectory(
        f32(x), w_init, [f32(g) for g in dys], STEPS)
    for t in range(STEPS):
        assert np.allclose(gpu_scales[t], ref_scales[t], rtol=1e-2, atol=0), t

    def rel(a, b):
        return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / np.linalg.norm(b))

    for i in range(3):
        upd_gpu = tr.w_master[i].double().cpu().numpy() - w_init[i]
        upd_ref = ref_master[i] - w_init[i]
        assert np.linalg.norm(upd_ref) > 0
        assert rel(upd_gpu, upd_ref) <= 1e-2, i
    assert rel(f32(tr.y), ref_y) <= 1e-2
    assert rel(f32(tr.dx), ref_dx) <= 1e-2


def test_fused_epilogues_match_standalone_passes():
    """The gated SwiGLU epilogue and the AdamW epilogues give the same bits as
    the standalone passes (fp8_swiglu_forward_quantize, stored dW +
    fp8_adamw_multi) over several steps: h, u, a's codes, every amax and
    scale, the weights, moments and bf16 copies."""
    lib()
    from fp8_quantized_gemm_gb300.mlp import SwiGLUTrainer
    x, w1, w3, w2 = workloads.swiglu(d=D, ffn=FFN, tokens=T)
    fused = SwiGLUTrainer(w1.cuda(), w3.cuda(), w2.cuda(), tokens=T, fuse_forward=True,
                          fuse_optimizer=True)
    plain = SwiGLUTrainer(w1.cuda(), w3.cuda(), w2.cuda(), tokens=T, fuse_forward=False,
                          fuse_optimizer=False)
    from fp8_quantized_gemm_gb300.mlp import K1, K2, K3
    assert plain.fuse_wq and not fused.fuse_wq
    xd = x.cuda()
    for t in range(4):
        dy = workloads.swiglu_grad(t, tokens=T, d=D).cuda()
        for tr in (fused, plain):
            tr.step(xd, dy)
        torch.cuda.synchronize()
        for name in ("h", "u", "aq", "y", "da", "dhq", "duq", "dx", "scale", "hist"):
            assert torch.equal(getattr(fused, name), getattr(plain, name)), (t, name)
        # the weights' amax slots: the AdamW epilogue path leaves the amax of
        # the weights this step used, the standalone update (which quantizes
        # the next step's weights) the amax of the updated ones
        others = [i for i in range(9) if i not in (K1, K3, K2)]
        assert torch.equal(fused.amax[others], plain.amax[others]), t
        for i, k in enumerate((K1, K3, K2)):
            assert plain.amax[k].item() == plain.w_bf[i].abs().max().float().item(), (t, k)
        for name in ("w_master", "m", "v", "w_bf"):
            for i in range(3):
                assert torch.equal(getattr(fused, name)[i], getattr(plain, name)[i]), (t, name, i)
        assert int(fused.step_dev.item()) == int(plain.step_dev.item()) == t + 1
    rc, where = lib().fp8_get_last_device_error()
    assert rc == 0, (rc, where)
