"""Pins of the prologue / epilogue oracle (oracle/prologue.py) against closed
forms and properties the definitions fix, independent of the oracle's own code:
a dropped tap, a reversed or shifted kernel, a missing eps or a wrong sign in
any step fails one of them."""
import math

import numpy as np
import pytest

from oracle import prologue as op


def test_conv_impulse_response_is_the_kernel_reversed_in_time():
    """A unit impulse at token t0 of channel c comes out as w[c, W-1], w[c, W-2], ...
    at tokens t0, t0 + 1, ... (tap W - 1 on the current token), zero elsewhere."""
    B, T, H, d, W, t0 = 2, 12, 3, 4, 4, 5
    rng = np.random.default_rng(1)
    w = rng.standard_normal((H * d, W))
    x = np.zeros((B, T, H, d))
    b, h, c = 1, 2, 3
    x[b, t0, h, c] = 1.0
    y = op.short_conv(x, w)
    expect = np.zeros_like(x)
    for i in range(W):
        expect[b, t0 + i, h, c] = w[h * d + c, W - 1 - i]
    np.testing.assert_array_equal(y, expect)


def test_conv_is_causal_and_starts_from_zeros():
    rng = np.random.default_rng(2)
    B, T, H, d, W = 1, 10, 2, 4, 3
    w = rng.standard_normal((H * d, W))
    x = rng.standard_normal((B, T, H, d))
    y = op.short_conv(x, w)
    x2 = x.copy()
    x2[:, 6:] += rng.standard_normal((B, T - 6, H, d))
    np.testing.assert_array_equal(op.short_conv(x2, w)[:, :6], y[:, :6])
    # token 0 sees only itself (the sequence starts from zeros)
    np.testing.assert_allclose(y[0, 0], x[0, 0] * w.reshape(H, d, W)[:, :, W - 1], rtol=0, atol=0)


def test_conv_is_linear_and_width_one_scales():
    rng = np.random.default_rng(3)
    B, T, H, d = 2, 7, 2, 4
    w = rng.standard_normal((H * d, 4))
    x, z = rng.standard_normal((2, B, T, H, d))
    np.testing.assert_allclose(op.short_conv(2.0 * x - 3.0 * z, w),
                               2.0 * op.short_conv(x, w) - 3.0 * op.short_conv(z, w), rtol=1e-13, atol=1e-13)
    w1 = rng.standard_normal((H * d, 1))
    np.testing.assert_array_equal(op.short_conv(x, w1), x * w1.reshape(H, d)[None, None])


def test_activation_closed_forms():
    assert op.sigmoid(0.0) == 0.5
    assert op.sigmoid(math.log(3.0)) == pytest.approx(0.75, abs=1e-15)
    x = np.linspace(-30, 30, 61)
    np.testing.assert_allclose(op.sigmoid(x) + op.sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    assert op.silu(0.0) == 0.0
    assert op.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), abs=1e-15)
    np.testing.assert_allclose(op.silu(x) - op.silu(-x), x, rtol=0, atol=1e-13)   # x(s(x) + s(-x)) = x
    assert op.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-15)
    assert op.softplus(math.log(math.e - 1.0)) == pytest.approx(1.0, abs=1e-15)
    assert op.softplus(60.0) == pytest.approx(60.0, abs=1e-15)
    assert op.softplus(-60.0) == pytest.approx(math.exp(-60.0), rel=1e-12)


def test_l2_normalize():
    np.testing.assert_allclose(op.l2_normalize(np.array([3.0, 4.0]), 0.0), [0.6, 0.8], rtol=0, atol=1e-16)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 128))
    y = op.l2_normalize(x, 0.0)
    np.testing.assert_allclose(np.sum(y * y, axis=-1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(op.l2_normalize(7.5 * x, 0.0), y, rtol=1e-14, atol=1e-15)
    # eps sits inside the root: |y|^2 = s / (s + eps)
    s = np.sum(x * x, axis=-1)
    ye = op.l2_normalize(x, 0.25)
    np.testing.assert_allclose(np.sum(ye * ye, axis=-1), s / (s + 0.25), rtol=1e-14)
    np.testing.assert_array_equal(op.l2_normalize(np.zeros(8), 1e-6), np.zeros(8))


def test_decay_gate():
    a = np.array([0.5, 2.0, 1.0])
    b = np.array([0.1, -0.3, 0.0])
    z = np.zeros((2, 4, 3)) - b[None, None, :]          # z + b = 0
    np.testing.assert_allclose(op.decay_gate(z, a, b), -a[None, None, :] * math.log(2.0) * np.ones((2, 4, 3)),
                               rtol=1e-15)
    np.testing.assert_array_equal(op.decay_gate(np.ones((1, 2, 3)), np.zeros(3), b), np.zeros((1, 2, 3)))
    # alpha = exp(g) stays in (0, 1] for a > 0
    rng = np.random.default_rng(5)
    zz = 5.0 * rng.standard_normal((2, 6, 3))
    g = op.decay_gate(zz, a, b)
    assert np.all(g <= 0.0) and np.all(np.exp(g) > 0.0)
    # KDA with the same bias in every channel: the Gated DeltaNet gate per channel
    dk = 4
    zk = np.repeat(zz[..., None], dk, axis=-1)
    gk = op.decay_gate(zk, a, np.repeat(b[:, None], dk, axis=1))
    np.testing.assert_allclose(gk, np.repeat(g[..., None], dk, axis=-1), rtol=1e-15)


def test_rmsnorm_gated():
    weight = np.array([1.0, -2.0, 0.5, 3.0])
    g = np.array([[[[0.3, -1.0, 2.0, 0.0]]]])
    c = -1.7
    o = np.full((1, 1, 1, 4), c)
    # a constant row normalises to its sign (eps = 0)
    np.testing.assert_allclose(op.rmsnorm_gated(o, g, weight, 0.0), np.sign(c) * weight * op.silu(g), rtol=1e-15)
    rng = np.random.default_rng(6)
    o2 = rng.standard_normal((2, 3, 2, 4))
    g2 = rng.standard_normal((2, 3, 2, 4))
    np.testing.assert_allclose(op.rmsnorm_gated(9.0 * o2, g2, weight, 0.0), op.rmsnorm_gated(o2, g2, weight, 0.0),
                               rtol=1e-14)
    # the mean of squares of the normalised row is 1 (eps = 0, unit gain, silu gate removed)
    y = op.rmsnorm_gated(o2, np.full_like(g2, 50.0), np.ones(4), 0.0) / op.silu(50.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_array_equal(op.rmsnorm_gated(o2, np.zeros_like(g2), weight, 1e-6), np.zeros_like(o2))


def test_prologue_composition_with_identity_convolution():
    """Width-one unit kernels: q = l2norm(silu(q_in)), k likewise, v = silu(v_in)."""
    rng = np.random.default_rng(7)
    B, T, H, dk, dv = 1, 5, 2, 8, 4
    q, k = rng.standard_normal((2, B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    bl = rng.standard_normal((B, T, H))
    one_k, one_v = np.ones((H * dk, 1)), np.ones((H * dv, 1))
    qo, ko, vo, beta, gate = op.prologue(q, k, v, one_k, one_k, one_v, bl, mode=op.MODE_DELTANET, eps=0.0)
    sq = q / (1.0 + np.exp(-q))   # x sigmoid(x), written independently of the oracle's form
    np.testing.assert_allclose(np.linalg.norm(qo, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(qo * np.linalg.norm(sq, axis=-1, keepdims=True), sq, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(vo, v / (1.0 + np.exp(-v)), rtol=1e-14)
    np.testing.assert_allclose(beta, 1.0 / (1.0 + np.exp(-bl)), rtol=1e-14)
    assert gate is None
