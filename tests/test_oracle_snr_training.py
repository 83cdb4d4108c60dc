"""Pins for the SNR metric (oracle/snr.py) and the training support math
(oracle/training.py): closed forms and finite differences."""
import math

import numpy as np

from oracle import snr as S
from oracle import training as T


def test_snr_exact_is_infinite():
    x = np.array([1.0, -2.0, 0.5])
    assert S.snr_db(x, x) == float("inf")


def test_snr_closed_form():
    n, c, delta = 1000, 3.0, 1e-2
    x = np.full(n, c)
    sgn = np.where(np.arange(n) % 2 == 0, 1.0, -1.0)
    assert math.isclose(S.snr_db(x, x + delta * c * sgn), -20 * math.log10(delta), rel_tol=1e-12)
    # 3 dB is (about) half the noise power
    assert math.isclose(S.snr_db(x, x + delta * c * sgn / math.sqrt(2)) - S.snr_db(x, x + delta * c * sgn),
                        10 * math.log10(2), rel_tol=1e-12)


def test_silu_closed_forms():
    assert T.silu(0.0) == 0.0
    assert math.isclose(float(T.silu(50.0)), 50.0, rel_tol=1e-15)
    assert abs(float(T.silu(-50.0))) < 1e-19
    assert math.isclose(float(T.silu(1.0)), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    z = np.linspace(-8, 8, 161)
    h = 1e-6
    fd = (T.silu(z + h) - T.silu(z - h)) / (2 * h)
    assert np.allclose(T.silu_grad(z), fd, atol=1e-8)


def test_swiglu_backward_matches_finite_difference():
    rng = np.random.default_rng(0)
    h, u, da = rng.standard_normal(50), rng.standard_normal(50), rng.standard_normal(50)
    dh, du = T.swiglu_backward(da, h, u)
    eps = 1e-6
    fd_h = (np.sum(da * T.swiglu_forward(h + eps, u)) - np.sum(da * T.swiglu_forward(h - eps, u))) / (2 * eps)
    fd_u = (np.sum(da * T.swiglu_forward(h, u + eps)) - np.sum(da * T.swiglu_forward(h, u - eps))) / (2 * eps)
    # perturbing every element at once: the directional derivative is the sum
    assert math.isclose(np.sum(dh), fd_h, rel_tol=1e-6, abs_tol=1e-8)
    assert math.isclose(np.sum(du), fd_u, rel_tol=1e-6, abs_tol=1e-8)


def test_adamw_first_step_closed_form():
    # on the first step m_hat = g and v_hat = g^2, so the step is lr * g / (|g| + eps)
    p0, g = np.array([1.0, -2.0, 0.5]), np.array([0.3, -1e-3, 0.0])
    p1, m1, v1 = T.adamw_step(p0, g, np.zeros(3), np.zeros(3), step=1)
    lr, wd, eps = 1e-4, 0.01, 1e-8
    exp = p0 * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    assert np.allclose(p1, exp, rtol=0, atol=1e-15)
    assert np.allclose(m1, 0.1 * g) and np.allclose(v1, 0.001 * g * g)


def test_adamw_update_is_bounded_by_lr():
    # MOSS blog, section 5: an Adam step moves each weight by about lr at most
    rng = np.random.default_rng(1)
    p = rng.standard_normal(1000)
    m = np.zeros(1000)
    v = np.zeros(1000)
    for t in range(1, 20):
        g = rng.standard_normal(1000) * 10.0 ** rng.integers(-6, 3)
        p_new, m, v = T.adamw_step(p, g, m, v, step=t, weight_decay=0.0)
        assert np.max(np.abs(p_new - p)) <= 1e-4 * 3.2
        p = p_new


def test_auto_scale_bounds_adamw_trajectory():
    """MOSS blog, section 5: Adam's step is bounded by eta times
    (1 - beta1) / sqrt(1 - beta2) per coordinate, so amax(W_t) never exceeds
    amax_0 + that bound times eta * t; the eq. (10) prediction with eta itself
    is the blog's tighter (typical-case) version of it."""
    rng = np.random.default_rng(3)
    w = rng.standard_normal(4096) * 0.02
    m = np.zeros_like(w)
    v = np.zeros_like(w)
    lr = 1e-4
    c = (1 - 0.9) / math.sqrt(1 - 0.999)
    amax0 = float(np.max(np.abs(w)))
    for t in range(1, 40):
        g = rng.standard_normal(4096) * 10.0 ** rng.integers(-5, 1)
        w, m, v = T.adamw_step(w, g, m, v, step=t)
        assert float(np.max(np.abs(w))) <= amax0 + c * lr * t + 1e-12
        s_pred = float(T.auto_weight_scale(amax0, c * lr, t, 448.0))
        assert np.max(np.abs(w)) / s_pred <= 448.0 * (1 + 1e-6)
    # eq. (10) grows linearly: equal steps add equal increments (fp32)
    s1 = T.auto_weight_scale(0.5, 1e-4, 100, 448.0)
    s2 = T.auto_weight_scale(0.5, 1e-4, 200, 448.0)
    assert abs((float(s2) - float(s1)) - 1e-4 * 100 / 448.0) < 1e-9
