"""FP8 SwiGLU training with delayed scaling: GPU step against the oracle,
teacher-forced (each stage is checked on the GPU's own inputs to it).

Per step: every quantized operand bit-exact against the oracle's delayed-
scaling state machine (which also fixes the scale used); the nine GEMMs
within the GEMM bound; SwiGLU forward/backward within one bf16 ulp; AdamW
within fp32 rounding; the nine amax histories exactly.  16 steps at a reduced
size (T 512, d 256, ffn 896)."""
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


def test_swiglu_training_teacher_forced():
    lib()
    from fp8_quantized_gemm_gb300.mlp import (A2, G1, G2, G3, K1, K2, K3, X1, X3,
                                              SwiGLUTrainer)
    x, w1, w3, w2 = workloads.swiglu(d=D, ffn=FFN, tokens=T)
    tr = SwiGLUTrainer(w1.cuda(), w3.cuda(), w2.cuda(), tokens=T)
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
        torch.cuda.synchronize()

        # quantized operands: oracle in_q on the tensor each slot quantizes
        inputs = {X1: xf, X3: xf, K1: wb[0], K3: wb[1], K2: wb[2], A2: f32(tr.a),
                  G2: f32(dy), G1: f32(tr.dh), G3: f32(tr.du)}
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
        assert bf16_close(f32(tr.a), OT.swiglu_forward(h, u)) <= 1.0, t
        dh_ref, du_ref = OT.swiglu_backward(da, h, u)
        assert bf16_close(f32(tr.dh), dh_ref) <= 1.0, t
        assert bf16_close(f32(tr.du), du_ref) <= 1.0, t

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
