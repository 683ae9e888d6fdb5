"""Pins of the oracle's gate prologue against what the pages and the
mathematics fix ("[논문 리뷰] Kimi K3 Technical Report", section 3.5:
g = g_min Sigmoid(e^A z), g_min = -5, alpha = exp(g), g in (-5, 0))."""
import numpy as np

import oracle


def test_gate_values_and_bounds():
    H, d = 2, 8
    A = np.linspace(-2, 1, H * d).reshape(H, d)
    q = np.ones((3, H, d))
    k = np.ones((3, H, d))
    z = np.zeros((3, H, d))
    _, _, g = oracle.gate_prologue(q, k, z, A, 1.0)
    np.testing.assert_array_equal(g, -2.5)                 # sigmoid(0) = 1/2
    z = np.stack([np.full((H, d), 1e4), np.full((H, d), -1e4), np.full((H, d), 0.3)])
    _, _, g = oracle.gate_prologue(q, k, z, A, 1.0)
    np.testing.assert_allclose(g[0], -5.0, rtol=0, atol=1e-12)   # z -> +inf: the lower bound
    np.testing.assert_allclose(g[1], 0.0, rtol=0, atol=1e-12)    # z -> -inf: no decay
    assert np.all(g[2] < 0) and np.all(g[2] > -5)
    # A = 0 reduces to g_min sigmoid(z); larger e^A z decays more
    _, _, g0 = oracle.gate_prologue(q[:1], k[:1], z[2:], np.zeros((H, d)), 1.0)
    np.testing.assert_allclose(g0, -5.0 / (1.0 + np.exp(-0.3)), rtol=1e-15)
    zz = np.linspace(-3, 3, 7)[:, None, None] * np.ones((1, H, d))
    _, _, gz = oracle.gate_prologue(np.ones((7, H, d)), np.ones((7, H, d)), zz, A, 1.0)
    assert np.all(np.diff(gz, axis=0) < 0)


def test_qk_normalisation():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((11, 3, 16)) * 7.0
    k = rng.standard_normal((11, 3, 16)) * 0.01
    z = rng.standard_normal((11, 3, 16))
    A = rng.standard_normal((3, 16))
    qh, kh, g = oracle.gate_prologue(q, k, z, A, 0.125)
    np.testing.assert_allclose(np.linalg.norm(kh, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(qh, axis=-1), 0.125, rtol=1e-14)
    # direction is kept: the result does not change when q, k are rescaled
    qh2, kh2, _ = oracle.gate_prologue(3.0 * q, 0.5 * k, z, A, 0.125)
    np.testing.assert_allclose(qh2, qh, rtol=1e-14)
    np.testing.assert_allclose(kh2, kh, rtol=1e-14)


def test_gate_value_with_nonzero_A():
    # e^A z = 1 at A = ln 2, z = 1/2, so g = -5 sigmoid(1); the slip e^{-A}
    # would give e^{-A} z = 1/4 instead, and a missing exponential A z = ln2/2.
    H, d = 1, 4
    A = np.full((H, d), np.log(2.0))
    z = np.full((1, H, d), 0.5)
    _, _, g = oracle.gate_prologue(np.ones((1, H, d)), np.ones((1, H, d)), z, A, 1.0)
    np.testing.assert_allclose(g, -5.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)
    # A = ln 4, z = -1/8: e^A z = -1/2
    A = np.full((H, d), np.log(4.0))
    z = np.full((1, H, d), -0.125)
    _, _, g = oracle.gate_prologue(np.ones((1, H, d)), np.ones((1, H, d)), z, A, 1.0)
    np.testing.assert_allclose(g, -5.0 / (1.0 + np.exp(0.5)), rtol=1e-15)
