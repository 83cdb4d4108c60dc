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


def test_swiglu_backward_elementwise_central_difference():
    """Each element of dh and du against its own central difference of the
    forward (a swapped pair, a permuted index or a missing factor of da or u
    fails here even where a sum would cancel)."""
    rng = np.random.default_rng(7)
    n = 400
    h = rng.standard_normal(n) * 3.0
    u = rng.standard_normal(n)
    da = rng.standard_normal(n)
    dh, du = T.swiglu_backward(da, h, u)
    eps = 1e-5
    fd_h = da * (T.swiglu_forward(h + eps, u) - T.swiglu_forward(h - eps, u)) / (2 * eps)
    fd_u = da * (T.swiglu_forward(h, u + eps) - T.swiglu_forward(h, u - eps)) / (2 * eps)
    assert np.allclose(dh, fd_h, rtol=1e-7, atol=1e-9)
    assert np.allclose(du, fd_u, rtol=1e-7, atol=1e-9)
    # a is linear in u, so du is exact: da * silu(h)
    assert np.array_equal(du, da * T.silu(h))
    # one element: z = 0 gives silu'(0) = 1/2, so dh = da * u / 2
    dh0, du0 = T.swiglu_backward(np.array([2.0]), np.array([0.0]), np.array([3.0]))
    assert dh0[0] == 3.0 and du0[0] == 0.0


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


def test_auto_scale_start_and_step_count():
    """MOSS blog, section 5, eq. (10) at its start and first steps: t = 0 is
    the current-scaling scale of the weight, bit for bit (the per-tensor
    ``scale_from_amax``, pinned on its own); every later t lies within two
    fp32 ulps of the exact rational (amax_0 + eta * t) / MAX, which moves by
    eta / MAX per step -- far more than two ulps at these magnitudes, so an
    off-by-one in t fails."""
    from fractions import Fraction

    from oracle import quantize as OQ
    rng = np.random.default_rng(11)
    w = (rng.standard_normal(4096) * 0.02).astype(np.float32)
    amax0 = OQ.amax(w)
    lr = 1e-4
    assert T.auto_weight_scale(amax0, lr, 0, 448.0) == OQ.scale_from_amax(amax0, "e4m3")
    for fmt_max, fmt in ((448.0, "e4m3"), (57344.0, "e5m2")):
        assert T.auto_weight_scale(amax0, lr, 0, fmt_max) == OQ.scale_from_amax(amax0, fmt)
    ulp = np.spacing(np.float32(amax0 / 448.0))
    for t in range(1, 6):
        exact = (Fraction(float(amax0)) + Fraction(lr) * t) / 448
        got = T.auto_weight_scale(amax0, lr, t, 448.0)
        assert abs(Fraction(float(got)) - exact) <= 2 * Fraction(float(ulp))
        # neighbouring step counts are distinguishable at this resolution
        assert abs(Fraction(float(got)) - (exact - Fraction(lr) / 448)) > 4 * Fraction(float(ulp))
