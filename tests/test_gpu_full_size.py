"""Parity at the configured full sizes, in the launch configuration the
benchmark times.

* FP8 SwiGLU training step with delayed scaling, d 4096, ffn 14336, 16384
  tokens (Flax guide 2.3 delayed scaling, 3.3 E4M3 forward / E5M2
  gradients): two steps of the trainer (weight gradients stored, standalone
  AdamW), the second checked teacher-forced --
  every scale used and every amax-history entry exactly, the codes of every
  quantized tensor bit-exact on sampled rows (the amaxes over the whole
  tensors), the nine GEMMs within the GEMM bound on 4096 sampled outputs each
  plus tile corners, SwiGLU within one bf16 ulp on sampled rows, AdamW on
  sampled weights.  Then the trainer with both epilogue variants (gated
  SwiGLU, AdamW in the weight-gradient GEMMs) against that path, bit for bit.
* MOSS two-level microscaling GEMM, M = N = K = 8192 (MOSS blog, section 4,
  steps 1-4) on the two-level workload's own inputs (8 outlier K columns x100
  in A): amax and global factor bit-exact, codes and local factors bit-exact
  on sampled rows (plus the row holding the tensor max, which fixes the global
  factor), the GEMM within the bound on sampled outputs plus tile corners.

The oracle works on host copies of what it needs; sampling happens on the
GPU's outputs only (positions are seeded)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import lib, mx_unpack, sample_positions, to_np_u8
from oracle import delayed as OD
from oracle import gemm as OG
from oracle import quantize as OQ
from oracle import training as OT

pytestmark = pytest.mark.gpu


def f32(t):
    return t.detach().float().cpu().numpy()


def amax_host(t):
    """Oracle amax of a device tensor, copied to the host in row chunks (the
    max of the chunks' maxes is the max)."""
    out = np.float32(0.0)
    rows = t.shape[0]
    step = max(1, (1 << 26) // max(1, t[0].numel()))
    for r in range(0, rows, step):
        out = max(out, OQ.amax(f32(t[r:r + step])))
    return np.float32(out)


def bf16_ulps(gpu, ref):
    ref = np.asarray(ref, np.float64)
    gpu = np.asarray(gpu, np.float64)
    tol = np.maximum(OG.bf16_ulp(ref), OG.bf16_ulp(gpu))
    return float(np.max(np.abs(gpu - ref) / tol))


def test_swiglu_training_step_full_size():
    F = lib()
    from fp8_quantized_gemm_gb300.mlp import (A2, G1, G2, G3, K1, K2, K3, X1, X3,
                                              SwiGLUTrainer)
    dev = torch.device("cuda")
    x, w1, w3, w2 = workloads.swiglu(device=dev)
    T, d = x.shape
    ffn = w1.shape[0]
    # dW stored, so that the weight-gradient GEMMs are checked on their own
    # (the AdamW epilogue is checked against this path bit for bit below)
    tr = SwiGLUTrainer(w1, w3, w2, tokens=T, fuse_optimizer=False)
    del w1, w3, w2
    fmt = {i: ("e5m2" if i in (G1, G3, G2) else "e4m3") for i in range(9)}
    states = [OD.DelayedState.initial(1024) for _ in range(9)]

    def swiglu_bf16():
        a = torch.empty_like(tr.h)
        dh, du = torch.empty_like(tr.h), torch.empty_like(tr.h)
        F.fp8_swiglu_forward(tr.h, tr.u, a)
        F.fp8_swiglu_backward(tr.da, tr.h, tr.u, dh, du)
        return a, dh, du

    for t in range(2):
        dy = workloads.swiglu_grad(t, device=dev)
        w_bf = [w.clone() for w in tr.w_bf]
        p0 = [w.clone() for w in tr.w_master]
        m0 = [w.clone() for w in tr.m]
        v0 = [w.clone() for w in tr.v]
        scale_used = tr.scale.cpu().numpy().copy()
        tr.forward_backward(x, dy)
        a_bf, dh_bf, du_bf = swiglu_bf16()
        torch.cuda.synchronize()
        tensors = {X1: x, X3: x, K1: w_bf[0], K3: w_bf[1], K2: w_bf[2], A2: a_bf, G2: dy,
                   G1: dh_bf, G3: du_bf}
        # the oracle's delayed-scaling state machine on the GPU's inputs: the
        # scale each slot used, and the amax each slot pushes
        amaxes = {}
        for i in range(9):
            s_expect = OD.compute_scale(np.max(states[i].history), states[i].scale, fmt[i])
            assert np.float32(scale_used[i]) == s_expect, (t, i)
            amaxes[i] = amax_host(tensors[i]) if i != X3 else amaxes[X1]
            states[i] = OD.DelayedState(OD.compute_amax_history(amaxes[i], states[i].history),
                                        s_expect)
        assert np.array_equal(tr.amax.cpu().numpy()[[X1, K1, K3, K2, A2, G2, G1, G3]],
                              np.array([amaxes[i] for i in (X1, K1, K3, K2, A2, G2, G1, G3)],
                                       dtype=np.float32)), t
        if t == 0:
            tr.optimizer_and_state()
            continue

        # ---- codes, bit-exact on sampled rows
        rng = np.random.default_rng(2024)
        codes = {X1: tr.xq, K1: tr.w1q, K3: tr.w3q, K2: tr.w2q, A2: tr.aq, G2: tr.dyq,
                 G1: tr.dhq, G3: tr.duq}
        for i, q in codes.items():
            rows = np.sort(rng.choice(q.shape[0], size=min(256, q.shape[0]), replace=False))
            ri = torch.from_numpy(rows).to(dev)
            src = f32(tensors[i].index_select(0, ri))
            want = OQ.quantize_with_scale(src, np.float32(scale_used[i]), fmt[i])
            assert np.array_equal(to_np_u8(q.index_select(0, ri)), want), (t, i)

        # ---- the nine GEMMs on 4096 sampled outputs each (+ tile corners)
        s = {i: np.float64(np.float32(scale_used[i])) for i in range(9)}

        def rows_of(q, idx, i):       # rows idx of a [R, K] code tensor, dequantized
            ii = torch.from_numpy(np.asarray(idx)).to(dev)
            return OG.dequant_operand(to_np_u8(q.index_select(0, ii)), fmt[i], s[i])

        def cols_of(q, idx, i):       # columns idx of a [K, R] code tensor, as rows
            ii = torch.from_numpy(np.asarray(idx)).to(dev)
            return OG.dequant_operand(to_np_u8(q.index_select(1, ii).t().contiguous()), fmt[i],
                                      s[i])

        def out_at(c, r, k):
            ri, ci = torch.from_numpy(r).to(dev), torch.from_numpy(k).to(dev)
            return c[ri, ci].double().cpu().numpy()

        cases = [
            # name, output, M, N, A rows (sampled rows), B rows (sampled cols), out dtype
            ("h", tr.h, T, ffn, lambda r: rows_of(tr.xq, r, X1), lambda c: rows_of(tr.w1q, c, K1),
             "bf16"),
            ("u", tr.u, T, ffn, lambda r: rows_of(tr.xq, r, X1), lambda c: rows_of(tr.w3q, c, K3),
             "bf16"),
            ("y", tr.y, T, d, lambda r: rows_of(tr.aq, r, A2), lambda c: rows_of(tr.w2q, c, K2),
             "bf16"),
            ("da", tr.da, T, ffn, lambda r: rows_of(tr.dyq, r, G2),
             lambda c: cols_of(tr.w2q, c, K2), "bf16"),
            ("dW2", tr.dw[2], d, ffn, lambda r: cols_of(tr.dyq, r, G2),
             lambda c: cols_of(tr.aq, c, A2), "f32"),
            ("dW1", tr.dw[0], ffn, d, lambda r: cols_of(tr.dhq, r, G1),
             lambda c: cols_of(tr.xq, c, X1), "f32"),
            ("dW3", tr.dw[1], ffn, d, lambda r: cols_of(tr.duq, r, G3),
             lambda c: cols_of(tr.xq, c, X1), "f32"),
        ]
        for seed, (name, out, M, N, arows, brows, odt) in enumerate(cases):
            r, c = sample_positions(M, N, 4096, seed)
            cref, eref = OG.gemm_sampled(arows(r), brows(c), np.arange(len(r)), np.arange(len(c)))
            ok, worst = OG.check(out_at(out, r, c), cref, eref, odt)
            assert ok, (name, worst)
        r, c = sample_positions(T, d, 4096, 99)
        c1, e1 = OG.gemm_sampled(rows_of(tr.dhq, r, G1), cols_of(tr.w1q, c, K1),
                                 np.arange(len(r)), np.arange(len(c)))
        c2, e2 = OG.gemm_sampled(rows_of(tr.duq, r, G3), cols_of(tr.w3q, c, K3),
                                 np.arange(len(r)), np.arange(len(c)))
        ok, worst = OG.check(out_at(tr.dx, r, c), c1 + c2, e1 + e2, "f32")
        assert ok, ("dx", worst)

        # ---- SwiGLU on sampled rows of the GPU's own h, u, da
        rows = torch.from_numpy(np.sort(rng.choice(T, 64, replace=False))).to(dev)
        h, u, da = (f32(z.index_select(0, rows)) for z in (tr.h, tr.u, tr.da))
        assert bf16_ulps(f32(a_bf.index_select(0, rows)), OT.swiglu_forward(h, u)) <= 1.0
        dh_ref, du_ref = OT.swiglu_backward(da, h, u)
        assert bf16_ulps(f32(dh_bf.index_select(0, rows)), dh_ref) <= 1.0
        assert bf16_ulps(f32(du_bf.index_select(0, rows)), du_ref) <= 1.0

        # ---- optimizer on sampled weights, then the histories
        picks = [torch.from_numpy(rng.choice(w.numel(), 65536, replace=False)).to(dev)
                 for w in tr.w_master]
        g = [tr.dw[i].reshape(-1)[picks[i]].double().cpu().numpy() for i in range(3)]
        tr.optimizer_and_state()
        torch.cuda.synchronize()
        for i in range(3):
            sel = picks[i]
            p_ref, m_ref, v_ref = OT.adamw_step(
                p0[i].reshape(-1)[sel].double().cpu().numpy(), g[i],
                m0[i].reshape(-1)[sel].double().cpu().numpy(),
                v0[i].reshape(-1)[sel].double().cpu().numpy(), step=t + 1)
            p_gpu = tr.w_master[i].reshape(-1)[sel].double().cpu().numpy()
            assert np.allclose(p_gpu, p_ref, rtol=2e-6, atol=1e-9), i
        hist = tr.hist.cpu().numpy()
        for i in range(9):
            assert np.array_equal(hist[i].view(np.uint32), states[i].history.view(np.uint32)), i
            new_scale = OD.compute_scale(np.max(states[i].history), states[i].scale, fmt[i])
            assert np.float32(tr.scale[i].item()) == new_scale, i
    rc, where = F.fp8_get_last_device_error()
    assert rc == 0, (rc, where)


def test_fused_training_step_full_size_matches_standalone_passes():
    """At full size, two steps of the trainer with both epilogue variants
    (gated SwiGLU, AdamW in the weight-gradient GEMMs) give the bits of the
    standalone passes (checked against the oracle in the test above)."""
    lib()
    from fp8_quantized_gemm_gb300.mlp import SwiGLUTrainer
    dev = torch.device("cuda")
    x, w1, w3, w2 = workloads.swiglu(device=dev)
    T = x.shape[0]
    fused = SwiGLUTrainer(w1, w3, w2, tokens=T, fuse_forward=True, fuse_optimizer=True)
    plain = SwiGLUTrainer(w1, w3, w2, tokens=T, fuse_forward=False, fuse_optimizer=False)
    del w1, w3, w2
    for t in range(2):
        dy = workloads.swiglu_grad(t, device=dev)
        for tr in (fused, plain):
            tr.step(x, dy)
        torch.cuda.synchronize()
        for name in ("h", "u", "aq", "dhq", "duq", "amax", "scale", "hist"):
            assert torch.equal(getattr(fused, name), getattr(plain, name)), (t, name)
        for name in ("w_master", "m", "v", "w_bf"):
            for i in range(3):
                assert torch.equal(getattr(fused, name)[i], getattr(plain, name)[i]), (t, name, i)
    rc, where = lib().fp8_get_last_device_error()
    assert rc == 0, (rc, where)


def test_two_level_gemm_8192_cubed():
    """Codes and local factors are checked on 512 sampled rows of each operand
    plus the row that holds the tensor's largest |x|: the global factor is the
    max over every block's s_i, which that row carries, so the oracle run on
    these rows gives exactly the full tensor's S, codes and local factors for
    them.  The GEMM is checked on the GPU's codes and factors (teacher-forced)
    at 4096 sampled outputs plus tile corners."""
    F = lib()
    dev = torch.device("cuda")
    M = N = K = 8192
    a, b = workloads.two_level(m=M, n=N, k=K)
    ops = []
    for t, r in ((a, M), (b, N)):
        td = t.to(dev)
        am, gl = torch.empty(1, device=dev), torch.empty(1, device=dev)
        q = torch.empty((r, K), dtype=torch.uint8, device=dev)
        words = F.mx_local_words(r, K, device=dev)
        F.fp8_amax(td, am)
        F.fp8_quantize_mx(td, F.E4M3, am, gl, q, words)
        ops.append((am, gl, q, words))
        del td
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    F.fp8_gemm_mx(ops[0][2], ops[0][3], ops[0][1], ops[1][2], ops[1][3], ops[1][1], y)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    gpu_ops = []
    for (am, gl, q, words), t, r in zip(ops, (a, b), (M, N)):
        tf = t.float().numpy()
        assert np.float32(am.item()) == OQ.amax(tf)
        top = int(np.argmax(np.max(np.abs(tf), axis=1)))
        rows = np.union1d(rng.choice(r, 512, replace=False), [top])
        q_ref, loc_ref, s_ref = OQ.quantize_two_level(tf[rows], "e4m3")
        q_gpu = to_np_u8(q)
        loc_gpu = mx_unpack(words.cpu().numpy(), r, K)
        assert np.float32(gl.item()) == np.float32(s_ref)
        assert np.array_equal(q_gpu[rows], q_ref)
        assert np.array_equal(loc_gpu[rows], loc_ref)
        gpu_ops.append((q_gpu, loc_gpu, np.float32(gl.item())))
        del tf
    # the outlier K columns move some local factors of A below 1 (the point of
    # the configuration)
    assert np.unique(gpu_ops[0][1]).size > 1
    rows, cols = sample_positions(M, N, 4096, 3)

    def operand_rows(q_all, loc_all, s, idx):
        return OG.dequant_operand(
            q_all[idx], "e4m3",
            OQ.expand(OQ.two_level_scale_values(loc_all[idx], s), len(idx), K, 1, 32))

    ar = operand_rows(*gpu_ops[0], rows)
    br = operand_rows(*gpu_ops[1], cols)
    cref, eref = OG.gemm_sampled(ar, br, np.arange(len(rows)), np.arange(len(cols)))
    ri, ci = torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)
    ok, worst = OG.check(y[ri, ci].double().cpu().numpy(), cref, eref, "bf16")
    assert ok, worst
    rc, where = F.fp8_get_last_device_error()
    assert rc == 0, (rc, where)
