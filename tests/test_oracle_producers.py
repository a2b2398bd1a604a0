"""Pins of the oracle's producers (RMSNorm, SwiGLU) against closed forms,
textbook values and invariants that do not come from the oracle itself.

RMSNorm: leone-cuda "CUDA kernel design", RMSNorm paragraphs (s = x (+ r),
y = s / sqrt(mean(s^2) + eps) * g).  SwiGLU: leone-cuda "CUDA kernel design",
SwiGLU paragraph (silu(gate) * up).
"""
import math

import numpy as np
import pytest

import oracle


def test_rmsnorm_hand_example():
    # x = (3, 4, 0, ..., 0) over K = 32: mean square 25/32, so y = x * sqrt(32) / 5
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 3, 4
    y, s = oracle.rmsnorm(x, np.ones(32, np.float32), 0.0)
    assert y[0, 0] == pytest.approx(3 * math.sqrt(32) / 5, rel=1e-15)
    assert y[0, 1] == pytest.approx(4 * math.sqrt(32) / 5, rel=1e-15)
    assert np.all(y[0, 2:] == 0)
    assert np.array_equal(s, x)


def test_rmsnorm_constant_row_closed_form():
    # a constant row c: y = g * c / sqrt(c^2 + eps)
    K, c, eps = 256, np.float32(-0.75), 1e-5
    g = np.linspace(-2, 2, K).astype(np.float32)
    y, _ = oracle.rmsnorm(np.full((1, K), c, np.float32), g, eps)
    want = g.astype(np.float64) * float(c) / math.sqrt(float(c) ** 2 + eps)
    assert np.allclose(y[0], want, rtol=1e-14, atol=0)


def test_rmsnorm_unit_mean_square_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 4096)).astype(np.float32)
    y, _ = oracle.rmsnorm(x, np.ones(4096, np.float32), 0.0)
    assert np.allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-13)
    y8, _ = oracle.rmsnorm(x * np.float32(8), np.ones(4096, np.float32), 0.0)   # power of two: exact in f32
    assert np.allclose(y8, y, rtol=1e-14)
    # the weight enters linearly
    g = rng.standard_normal(4096).astype(np.float32)
    yg, _ = oracle.rmsnorm(x, g, 0.0)
    y2g, _ = oracle.rmsnorm(x, 2 * g, 0.0)
    assert np.allclose(y2g, 2 * yg, rtol=1e-15)


def test_rmsnorm_residual_variant_normalizes_the_binary32_sum():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 512)).astype(np.float32)
    r = rng.standard_normal((2, 512)).astype(np.float32)
    g = rng.standard_normal(512).astype(np.float32)
    y, s = oracle.rmsnorm(x, g, 1e-6, r=r)
    assert np.array_equal(s, x + r)                           # numpy's binary32 add
    y2, _ = oracle.rmsnorm(x + r, g, 1e-6)
    assert np.array_equal(y, y2)


def test_rmsnorm_eps_dominates_a_zero_row():
    y, _ = oracle.rmsnorm(np.zeros((1, 64), np.float32), np.ones(64, np.float32), 1e-5)
    assert np.all(y == 0)


# logistic function values sigma(t) = 1 / (1 + e^-t) from tables (15+ digits), silu(t) = t * sigma(t)
SIGMA = {0.0: 0.5, 1.0: 0.7310585786300049, -1.0: 0.2689414213699951, 2.0: 0.8807970779778823,
         -2.0: 0.11920292202211755, 4.0: 0.9820137900379085}


def test_swiglu_logistic_table():
    gates = np.array(list(SIGMA), np.float32)
    F = 32
    gu = np.zeros((1, 2 * F), np.float32)
    gu[0, :gates.size] = gates
    gu[0, F:F + gates.size] = 1.0
    h = oracle.swiglu(gu, F)
    for i, t in enumerate(SIGMA):
        assert h[0, i] == pytest.approx(t * SIGMA[t], rel=1e-14, abs=1e-300)
    assert np.all(h[0, gates.size:] == 0)                      # silu(0) * 0


def test_swiglu_identity_and_linearity():
    # silu(t) - silu(-t) = t, and h is linear in up
    rng = np.random.default_rng(3)
    F = 96
    g = rng.standard_normal(F).astype(np.float32) * 4
    u = rng.standard_normal(F).astype(np.float32)
    ones = np.ones(F, np.float32)
    hp = oracle.swiglu(np.concatenate([g, ones])[None], F)[0]
    hm = oracle.swiglu(np.concatenate([-g, ones])[None], F)[0]
    assert np.allclose(hp - hm, g.astype(np.float64), rtol=1e-14, atol=1e-14)
    hu = oracle.swiglu(np.concatenate([g, u])[None], F)[0]
    assert np.allclose(hu, hp * u.astype(np.float64), rtol=1e-15, atol=0)


def test_swiglu_reads_the_two_halves_of_a_padded_row():
    F, ld = 64, 160
    rng = np.random.default_rng(4)
    gu = rng.standard_normal((2, ld)).astype(np.float32)
    # a row wider than 2F: the padding after the up half is ignored
    h_wide = oracle.swiglu(gu, F)
    h_tight = oracle.swiglu(np.ascontiguousarray(gu[:, :2 * F]), F)
    assert np.array_equal(h_wide, h_tight)
