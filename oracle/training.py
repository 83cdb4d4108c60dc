"""Support arithmetic of the FP8 SwiGLU training workload.

Test infrastructure only (see ``oracle/__init__``).

The pages describe the FP8 linear (Flax guide 3.3: E4M3 activations and
weights forward, E5M2 gradients backward; nanochat module "实现": the three
GEMMs of a linear layer) but not the MLP around it or the optimizer; the MOSS
blog (section 5) trains with Adam/AdamW.  Plain readings adopted:

* SwiGLU MLP: h = x W1^T, u = x W3^T, a = silu(h) * u, y = a W2^T with
  silu(z) = z / (1 + exp(-z)).  Backward: da = dy W2, dW2 = dy^T a,
  dh = da * u * silu'(h), du = da * silu(h), dx = dh W1 + du W3,
  dW1 = dh^T x, dW3 = du^T x, where silu'(z) = s(z) (1 + z (1 - s(z))) and
  s is the logistic function.
* AdamW (decoupled weight decay, bias-corrected moments) with
  beta1 = 0.9, beta2 = 0.999, eps = 1e-8, weight_decay = 0.01, lr = 1e-4:
  p <- p - lr*wd*p;  m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
  p <- p - lr * (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps).

Automatic weight scaling (MOSS blog, section 5, eq. 10): within a re-scaling
interval the weight scale is predicted, without reading the weights, as
``(amax_0 + eta * t) / MAX``: amax_0 from the last max-reduction, t the steps
since then, eta the learning rate (an Adam step moves a weight by about eta at
most).  Evaluated in fp32 as fl32(fl32(amax_0 + fl32(eta * t)) / MAX).

Float64 throughout (fp32 for the scale formula).  Pins
(``tests/test_oracle_snr_training.py``): silu'(z)
against a central finite difference, silu at 0 and large |z|; every element
of dh and du against its own central difference of the forward; AdamW's
first step on a constant gradient (an update of lr * g / (|g| + eps') after
the decay); the automatic scale bounds amax(W_t) on an AdamW trajectory
with the Adam per-step bound (1 - beta1) / sqrt(1 - beta2) times eta, equals
the current-scaling scale at t = 0 bit for bit, and stays within two fp32
ulps of the exact rational (amax_0 + eta t) / MAX for t >= 1.
"""
from __future__ import annotations

import numpy as np

ADAMW = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def silu_grad(z):
    z = np.asarray(z, dtype=np.float64)
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def swiglu_forward(h, u):
    """a = silu(h) * u."""
    return silu(h) * np.asarray(u, dtype=np.float64)


def swiglu_backward(da, h, u):
    """(dh, du) for a = silu(h) * u."""
    da = np.asarray(da, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    return da * u * silu_grad(h), da * silu(h)


def adamw_step(p, g, m, v, step: int, lr=ADAMW["lr"], beta1=ADAMW["beta1"],
               beta2=ADAMW["beta2"], eps=ADAMW["eps"],
               weight_decay=ADAMW["weight_decay"]):
    """One AdamW update; returns new (p, m, v).  ``step`` counts from 1."""
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    p = p * (1.0 - lr * weight_decay)
    mhat = m / (1.0 - beta1 ** step)
    vhat = v / (1.0 - beta2 ** step)
    p = p - lr * mhat / (np.sqrt(vhat) + eps)
    return p, m, v


def auto_weight_scale(amax0, lr, t, fmt_max) -> np.float32:
    """MOSS eq. (10): predicted scale (amax_0 + eta * t) / MAX, in fp32."""
    F32 = np.float32
    grow = F32(np.float64(lr) * np.float64(t))
    return F32(F32(F32(amax0) + grow) / F32(fmt_max))
