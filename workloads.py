"""Seeded synthetic inputs for the scaled-FP8 GEMM workloads.

This module only draws random tensors.  It holds none of the method's
arithmetic (no amax, no scale, no quantization, no contraction), so both the
CUDA path and the CPU oracle may import it without sharing any of the
computation they are compared on.

Every tensor is drawn on the host with a seeded ``torch.Generator`` in fp32 and
then rounded to bf16 (round-to-nearest-even, torch's own cast), so the bytes fed
to the GPU and to the oracle are identical.

Workloads (shapes and distributions follow the five scaled-FP8 configurations):

* ``tiny_per_tensor``   a[16,32], b[32,64] uniform[0,1), fp32, seed 0 (the
  Flax FP8 guide's 16x32 . 32x64 example, section 2.1/2.2).
* ``float8_linear``     x[8192,2048] ~N(0,1), W[2048,2048] ~N(0,0.02),
  g[8192,2048] ~N(0,1e-3), bf16, seed 1 (the nanochat Float8 linear,
  forward and backward).
* ``fine_grained``      act[M,7168] ~N(0,1) with 0.5 % of the K columns x50,
  W[2048,7168] ~N(0,0.02), bf16, seed 2 (Transformers fine-grained FP8).
* ``two_level``         A[8192,8192] ~N(0,1) with 0.1 % of the K columns x100,
  B[8192,8192] ~N(0,0.02), bf16, seed 3 (MOSS two-level microscaling).
* ``swiglu``            SwiGLU MLP: x[T,d] ~N(0,1), W1/W3[ffn,d], W2[d,ffn]
  ~N(0,0.02), bf16, seed 4; step-t output gradient dy ~N(0,1e-3), seed 1000+t.
* ``moe_experts``       mixture-of-experts layer (Transformers fine-grained
  FP8, FP8Experts): token counts per expert from a seeded multinomial over
  expert weights ~ U[0.2, 1) (uneven, some experts may get no tokens),
  activations [T, K] ~N(0,1) with 0.5 % outlier columns x50 ordered by
  expert, expert weights [E, N, K] ~N(0,0.02), bf16, seed 5.

Outlier columns: count = round(frac * K); the indices are the first ``count``
entries of a seeded permutation of range(K); the multiply is done in fp32
before the bf16 rounding.
"""
from __future__ import annotations

import torch


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std: float, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device) * std


def _outlier_columns(x: torch.Tensor, frac: float, factor: float,
                     gen: torch.Generator) -> torch.Tensor:
    k = x.shape[-1]
    count = int(round(frac * k))
    idx = torch.randperm(k, generator=gen)[:count]
    x[..., idx] *= factor
    return x


def tiny_per_tensor(seed: int = 0):
    """a[16,32], b[32,64] ~ U[0,1) in fp32."""
    g = _gen(seed)
    a = torch.rand(16, 32, generator=g, dtype=torch.float32)
    b = torch.rand(32, 64, generator=g, dtype=torch.float32)
    return a, b


def float8_linear(seed: int = 1, tokens: int = 8192, d_in: int = 2048,
                  d_out: int = 2048):
    """x[tokens,d_in], W[d_out,d_in], g[tokens,d_out] in bf16."""
    g = _gen(seed)
    x = _normal((tokens, d_in), 1.0, g).to(torch.bfloat16)
    w = _normal((d_out, d_in), 0.02, g).to(torch.bfloat16)
    go = _normal((tokens, d_out), 1e-3, g).to(torch.bfloat16)
    return x, w, go


def fine_grained(m: int, seed: int = 2, k: int = 7168, n: int = 2048,
                 outlier_frac: float = 0.005, outlier_factor: float = 50.0):
    """act[m,k] with outlier columns, W[n,k], both bf16.

    The weight is drawn first so that it is the same for every m.
    """
    g = _gen(seed)
    w = _normal((n, k), 0.02, g).to(torch.bfloat16)
    ga = _gen(seed * 1_000_003 + m)
    act = _normal((m, k), 1.0, ga)
    act = _outlier_columns(act, outlier_frac, outlier_factor, ga)
    return act.to(torch.bfloat16), w


def two_level(seed: int = 3, m: int = 8192, n: int = 8192, k: int = 8192,
              outlier_frac: float = 0.001, outlier_factor: float = 100.0):
    """A[m,k] with outlier K-channels, B[n,k] (stored [N,K]), both bf16."""
    g = _gen(seed)
    a = _normal((m, k), 1.0, g)
    a = _outlier_columns(a, outlier_frac, outlier_factor, g)
    b = _normal((n, k), 0.02, g)
    return a.to(torch.bfloat16), b.to(torch.bfloat16)


def swiglu(seed: int = 4, d: int = 4096, ffn: int = 14336, tokens: int = 16384,
           device="cpu"):
    """x[tokens,d], W1[ffn,d], W3[ffn,d], W2[d,ffn] in bf16.

    ``device`` selects the generator: the CPU stream (used by the parity
    tests) or a seeded CUDA stream (different values, same distribution; used
    to draw the full-size training workload quickly)."""
    g = _gen(seed, device)
    x = _normal((tokens, d), 1.0, g).to(torch.bfloat16)
    w1 = _normal((ffn, d), 0.02, g).to(torch.bfloat16)
    w3 = _normal((ffn, d), 0.02, g).to(torch.bfloat16)
    w2 = _normal((d, ffn), 0.02, g).to(torch.bfloat16)
    return x, w1, w3, w2


def swiglu_grad(step: int, tokens: int = 16384, d: int = 4096, device="cpu"):
    """Synthetic loss gradient dy[tokens,d] ~N(0,1e-3) for training step ``step``."""
    g = _gen(1000 + step, device)
    return _normal((tokens, d), 1e-3, g).to(torch.bfloat16)


def moe_experts(experts: int, tokens: int, n: int, k: int, seed: int = 5,
                outlier_frac: float = 0.005, outlier_factor: float = 50.0):
    """(act[tokens,k] bf16, w[experts,n,k] bf16, counts[experts] int64): the
    rows of act are already grouped by expert, counts[e] rows for expert e."""
    g = _gen(seed)
    probs = torch.rand(experts, generator=g) * 0.8 + 0.2
    idx = torch.multinomial(probs, tokens, replacement=True, generator=g)
    counts = torch.bincount(idx, minlength=experts).to(torch.int64)
    w = _normal((experts, n, k), 0.02, g).to(torch.bfloat16)
    act = _normal((tokens, k), 1.0, g)
    act = _outlier_columns(act, outlier_frac, outlier_factor, g)
    return act.to(torch.bfloat16), w, counts


def uniform(shape, lo: float, hi: float, seed: int) -> torch.Tensor:
    """fp32 uniform[lo,hi) draw, for edge-case tests."""
    g = _gen(seed)
    return torch.rand(*shape, generator=g, dtype=torch.float32) * (hi - lo) + lo


def normal(shape, std: float, seed: int) -> torch.Tensor:
    """fp32 N(0,std) draw, for edge-case tests."""
    return _normal(shape, std, _gen(seed))
