"""FP8 SwiGLU MLP training step with delayed scaling, as a sequence of C-ABI
calls (every arithmetic step runs in the library's kernels).

    h = x W1^T,  u = x W3^T,  a = silu(h) * u,  y = a W2^T
    da = dy W2,  dW2 = dy^T a,  dh, du = swiglu_backward(da, h, u)
    dx = dh W1 + du W3,  dW1 = dh^T x,  dW3 = du^T x
    AdamW on fp32 master weights; bf16 copies feed the next step's quantizer.

E4M3 for activations and weights, E5M2 for gradients (Flax guide 3.3).  Each
linear keeps three (amax history, scale) pairs -- input, kernel, output
gradient -- as the Flax guide's per-layer meta does (section 5.1); a tensor is
quantized with the scale left by the previous step and its fused amax is
pushed afterwards (section 2.3).  Both W1 and W3 take x as input: their two
input states receive the same amax every step and so always hold the same
scale; x is quantized once, with the first.

Weight scaling: "delayed" (above) or "auto", the MOSS blog's automatic
scaling (section 5, eq. 10): each weight's scale is predicted as
(amax_0 + lr * t) / MAX from the amax_0 of its last max-reduction, t steps
ago, without reading the weight; the max-reduction (fp8_amax) is redone every
`rescale_interval` steps (500 in the blog).

Every tensor is quantized once, to row-major codes; the GEMMs read them
K-major or MN-major as they need (dx = dh W1 reads W1's codes MN-major,
dW1 = dh^T x reads dh's and x's codes MN-major), so no transposed copies are
written.  GEMMs with independent outputs share one grouped launch (h and u;
da and dW2; dx's first term, dW1 and dW3).

Delayed scaling fixes every scale before its tensor exists, so the SwiGLU
passes quantize what they produce: a, dh and du reach memory only as FP8
codes (the same codes and amaxes as the bf16 tensors quantized afterwards
would give).  The forward's element-wise work also moves into a GEMM
epilogue (fp8_gemm_tensor_grouped's gated variant): h and u come out of one
launch whose epilogue also writes a's codes (``fuse_forward``, default on).
``fuse_optimizer=True`` has the three weight-gradient GEMMs apply AdamW to
their tiles instead of storing dW (the AdamW epilogue: the same bits, no dW
buffers, measured no faster than the standalone update at these shapes, so
off by default: dW is stored in ``self.dw`` and fp8_adamw_multi updates the
weights after the backward; ``overlap_optimizer=True`` instead updates each
weight on a second stream as soon as its gradient exists, beside the
compute-bound GEMMs that remain -- the same bits, measured no faster on this
GPU, whose step runs under its power cap).  The
optimizer keeps its step count on the device, so `step` issues the same
calls every time and can be captured as a CUDA graph (the second stream
forks from and joins the capturing one) and replayed.

With delayed weight scaling and the standalone update (the defaults), the
next step's weight quantization also moves into the optimizer: the amax
histories are pushed first, which fixes the scales the next step quantizes
the weights with, and fp8_adamw_multi then writes the codes of the updated
weights (as bf16) under those scales and their amaxes -- what the next
step's fp8_quantize_tensor calls on the bf16 copies would give -- so from
the second step on the forward quantizes only x, and no call reads a bf16
copy of the weights: the update writes none (`w_bf` then returns the bf16
rounding of the fp32 masters, the values such a copy would hold).

Buffers are allocated once (device memory through torch); `step` issues the
calls on the current stream.
"""
from __future__ import annotations

import torch

import fp8_quantized_gemm_gb300 as F

# state slots: (input, kernel, output grad) for linear 1 (W1), 3 (W3), 2 (W2)
X1, K1, G1, X3, K3, G3, A2, K2, G2 = range(9)
STATE_NAMES = ("x@W1", "W1", "dh", "x@W3", "W3", "du", "a@W2", "W2", "dy")
HISTORY = 1024


class SwiGLUTrainer:
    def __init__(self, w1: torch.Tensor, w3: torch.Tensor, w2: torch.Tensor, tokens: int,
                 lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
                 history: int = HISTORY, weight_scaling: str = "delayed",
                 rescale_interval: int = 500, fuse_forward: bool = True,
                 fuse_optimizer: bool = False, overlap_optimizer: bool = False):
        if weight_scaling not in ("delayed", "auto"):
            raise ValueError(weight_scaling)
        self.weight_scaling = weight_scaling
        self.fuse_forward, self.fuse_optimizer = fuse_forward, fuse_optimizer
        # the standalone AdamW of each weight runs on a second stream as soon
        # as that weight's gradient exists, beside the remaining GEMMs
        self.overlap = overlap_optimizer and not fuse_optimizer
        self.side = torch.cuda.Stream(device=w1.device) if self.overlap else None
        self.rescale_interval = rescale_interval
        # the optimizer writes the next step's weight codes (see the module
        # docstring); until the first update the forward quantizes them
        self.fuse_wq = weight_scaling == "delayed" and not fuse_optimizer and not self.overlap
        self.w_codes_ready = False
        dev = w1.device
        ffn, d = w1.shape
        assert w3.shape == (ffn, d) and w2.shape == (d, ffn)
        self.T, self.d, self.ffn = tokens, d, ffn
        self.hp = dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay)
        self.t = 0
        bf, f32 = dict(dtype=torch.bfloat16, device=dev), dict(dtype=torch.float32, device=dev)
        u8 = dict(dtype=torch.uint8, device=dev)
        T = tokens
        # weights: fp32 masters, moments, bf16 copies
        # (bf16 copies kept up to date only where a later call reads them:
        # when the optimizer writes the next step's codes itself, nothing
        # does, and the copies stay the initial weights; see w_bf)
        self._w_bf = [w1.contiguous().clone(), w3.contiguous().clone(), w2.contiguous().clone()]
        self.keep_bf16 = not self.fuse_wq
        self.w_master = [w.float() for w in self._w_bf]
        self.m = [torch.zeros_like(w) for w in self.w_master]
        self.v = [torch.zeros_like(w) for w in self.w_master]
        # delayed-scaling state
        self.hist = torch.zeros((9, history), **f32)
        self.scale = torch.ones(9, **f32)
        self.amax = torch.zeros(9, **f32)
        # quantized operands (row-major codes)
        self.xq = torch.empty((T, d), **u8)
        self.w1q, self.w3q = torch.empty((ffn, d), **u8), torch.empty((ffn, d), **u8)
        self.w2q = torch.empty((d, ffn), **u8)
        self.aq = torch.empty((T, ffn), **u8)
        self.dyq = torch.empty((T, d), **u8)
        self.dhq, self.duq = torch.empty((T, ffn), **u8), torch.empty((T, ffn), **u8)
        # activations and gradients (a, dh and du exist only as codes)
        self.h, self.u = (torch.empty((T, ffn), **bf) for _ in range(2))
        self.y = torch.empty((T, d), **bf)
        self.da = torch.empty((T, ffn), **bf)
        self.dx = torch.empty((T, d), **f32)
        self.flops_per_step = 9 * 2.0 * T * d * ffn
        # optimizer step count on the device (advanced by fp8_adamw_multi)
        self.step_dev = torch.zeros(1, dtype=torch.int64, device=dev)
        if fuse_optimizer:
            # the weight-gradient GEMMs update the weights in their epilogues
            self.dw = [None, None, None]
            self.adamw_ep = [F.adamw_epilogue(self.w_master[i], self.m[i], self.v[i],
                                              self._w_bf[i], self.step_dev, **self.hp)
                             for i in range(3)]
        else:
            self.dw = [torch.empty((ffn, d), **f32), torch.empty((ffn, d), **f32),
                       torch.empty((d, ffn), **f32)]
            self.adamw_ep = [None, None, None]
            wq, slot = (self.w1q, self.w3q, self.w2q), (K1, K3, K2)
            self.adamw_items = [
                F.adamw_item(self.w_master[i], self.dw[i], self.m[i], self.v[i],
                             self._w_bf[i] if self.keep_bf16 else None,
                             **(dict(q=wq[i], q_scale=self.scale[slot[i]:slot[i] + 1],
                                     q_amax=self.amax[slot[i]:slot[i] + 1], q_fmt=F.E4M3)
                                if self.fuse_wq else {}))
                for i in range(3)]
        # gated forward: h | u in one launch whose epilogue also quantizes a
        self.swiglu_ep = (F.swiglu_epilogue(self.w3q, self.scale[K3:K3 + 1], self.u, self.aq,
                                            F.E4M3, self.scale[A2:A2 + 1],
                                            self.amax[A2:A2 + 1]) if fuse_forward else None)
        # automatic weight scaling: amax at the last max-reduction, steps since
        self.w_amax0 = torch.zeros(3, **f32)
        self.t_since = 0
        if weight_scaling == "auto":
            self.refresh_weight_amax()

    def refresh_weight_amax(self):
        """The max-reduction of automatic scaling (fp8_amax of each weight)."""
        for i in range(3):
            F.fp8_amax(self._w_bf[i], self.w_amax0[i:i + 1])
        self.t_since = 0

    @property
    def w_bf(self):
        """The bf16 weights: the maintained copies, or, once the optimizer
        writes the next step's codes itself (and keeps no bf16 copy), the bf16
        rounding of the fp32 masters -- the same values the copies would hold
        (plumbing for inspection; the step never reads it)."""
        if self.keep_bf16 or not self.w_codes_ready:
            return self._w_bf
        return [w.to(torch.bfloat16) for w in self.w_master]

    def _sc(self, i):
        return self.scale[i:i + 1]

    def _am(self, i):
        return self.amax[i:i + 1]

    def forward_backward(self, x: torch.Tensor, dy: torch.Tensor):
        """The nine GEMMs with their quantize and SwiGLU passes; with the fused
        optimizer also the AdamW updates (in the weight-gradient GEMMs)."""
        E4, E5, MN = F.E4M3, F.E5M2, F.MN_MAJOR
        q, P, run = F.fp8_quantize_tensor, F.gemm_problem, F.fp8_gemm_tensor_grouped
        w1, w3, w2 = self._w_bf
        sc = self._sc
        # forward
        q(x, E4, self.xq, scale=sc(X1), amax_out=self._am(X1))
        if self.weight_scaling == "auto":
            for i, slot in ((0, K1), (1, K3), (2, K2)):
                F.fp8_auto_weight_scale(self.w_amax0[i:i + 1], self.t_since, self.hp["lr"], E4,
                                        sc(slot))
            wam = (None, None, None)
        else:
            wam = (self._am(K1), self._am(K3), self._am(K2))
        if not (self.fuse_wq and self.w_codes_ready):  # else the optimizer wrote them
            q(w1, E4, self.w1q, scale=sc(K1), amax_out=wam[0])
            q(w3, E4, self.w3q, scale=sc(K3), amax_out=wam[1])
            q(w2, E4, self.w2q, scale=sc(K2), amax_out=wam[2])
        if self.fuse_forward:
            run([P(self.xq, E4, self.w1q, E4, sc(X1), sc(K1), self.h,       # h, u = x W1^T, x W3^T
                   swiglu=self.swiglu_ep)])                                 # a = silu(h) u
        else:
            run([P(self.xq, E4, self.w1q, E4, sc(X1), sc(K1), self.h),      # h = x W1^T
                 P(self.xq, E4, self.w3q, E4, sc(X1), sc(K3), self.u)])     # u = x W3^T
            F.fp8_swiglu_forward_quantize(self.h, self.u, E4, sc(A2), self.aq,  # a = silu(h) u
                                          self._am(A2))
        run([P(self.aq, E4, self.w2q, E4, sc(A2), sc(K2), self.y)])         # y = a W2^T
        # backward
        if self.fuse_optimizer or self.overlap:
            F.fp8_adamw_multi([], self.step_dev, **self.hp)  # t of this step's updates
        ep = self.adamw_ep
        q(dy, E5, self.dyq, scale=sc(G2), amax_out=self._am(G2))
        run([P(self.dyq, E5, self.w2q, E4, sc(G2), sc(K2), self.da, b_layout=MN),   # da = dy W2
             P(self.dyq, E5, self.aq, E4, sc(G2), sc(A2), self.dw[2],               # dW2 = dy^T a
               a_layout=MN, b_layout=MN, adamw=ep[2])])
        if self.overlap:
            self._side_adamw([self.adamw_items[2]])                         # W2, beside the rest
        F.fp8_swiglu_backward_quantize(self.da, self.h, self.u, E5, sc(G1), sc(G3),  # dh, du
                                       self.dhq, self.duq, self._am(G1), self._am(G3))
        run([P(self.dhq, E5, self.w1q, E4, sc(G1), sc(K1), self.dx, b_layout=MN),   # dx = dh W1
             P(self.dhq, E5, self.xq, E4, sc(G1), sc(X1), self.dw[0],               # dW1 = dh^T x
               a_layout=MN, b_layout=MN, adamw=ep[0]),
             P(self.duq, E5, self.xq, E4, sc(G3), sc(X1), self.dw[1],               # dW3 = du^T x
               a_layout=MN, b_layout=MN, adamw=ep[1])])
        if self.overlap:
            self._side_adamw(self.adamw_items[:2])                          # W1, W3
        run([P(self.duq, E5, self.w3q, E4, sc(G3), sc(K3), self.dx, b_layout=MN,    # dx += du W3
               accumulate=True)])

    def _side_adamw(self, items):
        """AdamW on `items` on the second stream once the current stream has
        produced their gradients; t is the step's (already advanced) count.
        Nothing later in the step reads those weights' masters, moments or bf16
        copies (the GEMMs read the codes), so the update overlaps the GEMMs."""
        ready = torch.cuda.Event()
        ready.record()
        self.side.wait_event(ready)
        with torch.cuda.stream(self.side):
            F.fp8_adamw_multi(items, self.step_dev, advance=False, **self.hp)

    def optimizer_and_state(self):
        """AdamW on the three weights (unless the weight-gradient GEMMs did it),
        then the nine amax-history pushes; with the fused weight quantization
        the pushes first, then AdamW (which quantizes the updated weights with
        the scales the pushes left)."""
        self.t += 1
        if self.fuse_wq:
            self._push_histories(auto=False)
            F.fp8_adamw_multi(self.adamw_items, self.step_dev, **self.hp)
            self.w_codes_ready = True
            return
        if self.overlap:
            torch.cuda.current_stream().wait_stream(self.side)  # the updates are done
        elif not self.fuse_optimizer:
            F.fp8_adamw_multi(self.adamw_items, self.step_dev, **self.hp)
        auto = self.weight_scaling == "auto"
        if auto:
            self.t_since += 1
            if self.t_since >= self.rescale_interval:
                self.refresh_weight_amax()
        self._push_histories(auto)

    def _push_histories(self, auto: bool):
        """The amax-history pushes of every delayed-scaling state, one launch."""
        items = []
        for i in range(9):
            if auto and i in (K1, K3, K2):
                continue  # weights follow eq. (10), not a history
            cur = X1 if i == X3 else i  # the x@W3 input state takes x's amax
            fmt = F.E5M2 if i in (G1, G3, G2) else F.E4M3
            items.append(F.delayed_item(self.hist[i], self.scale[i:i + 1], self._am(cur), fmt))
        F.fp8_delayed_state_update_multi(items)  # the histories in one launch

    def step(self, x: torch.Tensor, dy: torch.Tensor):
        self.forward_backward(x, dy)
        self.optimizer_and_state()
