"""Pins of the oracle's per-token steps around the recurrence (oracle.layer_ops)
against closed forms and library routines, on the CPU."""
from __future__ import annotations

import numpy as np

from oracle import layer_ops as L


def _rng(seed):
    return np.random.default_rng(seed)


def test_short_conv_impulse_response_is_the_causal_kernel():
    """A unit impulse at token t0 comes out as the taps, oldest last: y[t0 + i]
    = w[3 - i] for i = 0..3, nothing before t0 (causal) and nothing after."""
    r = _rng(1)
    T, H, d, t0 = 12, 2, 6, 5
    w = r.standard_normal((H, d, 4))
    x = np.zeros((T, H, d))
    x[t0, 1, 4] = 1.0
    y = L.short_conv(x, w, [0, T])
    expect = np.zeros(T)
    for i in range(4):
        expect[t0 + i] = w[1, 4, 3 - i]
    np.testing.assert_array_equal(y[:, 1, 4], expect)
    assert np.count_nonzero(y) == 4


def test_short_conv_equals_numpy_convolve():
    """One sequence: per channel, the full discrete convolution with the reversed
    taps, truncated to the sequence (numpy.convolve)."""
    r = _rng(2)
    T, H, d = 17, 2, 5
    w = r.standard_normal((H, d, 4))
    x = r.standard_normal((T, H, d))
    y = L.short_conv(x, w, [0, T])
    for h in range(H):
        for c in range(d):
            ref = np.convolve(x[:, h, c], w[h, c, ::-1], mode="full")[:T]
            np.testing.assert_allclose(y[:, h, c], ref, rtol=1e-13, atol=1e-13)


def test_short_conv_restarts_at_every_sequence():
    """Packed sequences (including ones shorter than the kernel and an empty one)
    equal separate calls: nothing leaks across a boundary."""
    r = _rng(3)
    lengths = [2, 0, 5, 1, 7]
    H, d = 2, 3
    N = sum(lengths)
    w = r.standard_normal((H, d, 4))
    x = r.standard_normal((N, H, d))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    y = L.short_conv(x, w, cu)
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        np.testing.assert_array_equal(y[a:b], L.short_conv(x[a:b], w, [0, b - a]))


def test_swish_and_gates_closed_forms():
    assert L.swish(0.0) == 0.0
    np.testing.assert_allclose(L.swish(40.0), 40.0, rtol=1e-15)
    assert abs(L.swish(-40.0)) < 1e-15
    np.testing.assert_allclose(L.swish(1.0), 1.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)
    q = k = v = np.zeros((1, 1, 4))
    w = np.zeros((3, 1, 4, 4))
    a = np.array([[[0.0, 50.0, -50.0, 1.0]]])
    _, _, _, la, beta = L.prep(q, k, v, w, a, np.array([[0.0]]), [0, 1])
    np.testing.assert_allclose(la[0, 0, :3], [-2.5, -5.0, 0.0], atol=1e-12)
    assert -5.0 < la[0, 0, 3] < 0.0
    np.testing.assert_allclose(beta, [[0.5]], rtol=1e-15)


def test_l2norm_unit_length_and_scale_invariance():
    r = _rng(4)
    x = r.standard_normal((6, 3, 128))
    n = L.l2norm(x)
    unit = x / np.linalg.norm(x, axis=-1, keepdims=True)
    np.testing.assert_allclose(np.linalg.norm(n, axis=-1), 1.0, rtol=1e-6)
    # far above the epsilon the result is the exact unit vector (scale invariance)
    np.testing.assert_allclose(L.l2norm(1e4 * x), unit, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(n / np.linalg.norm(n, axis=-1, keepdims=True), unit, rtol=1e-12)


def test_post_closed_forms():
    """RMSNorm of a constant vector c is gamma * c / sqrt(c^2 + eps); a zero gate
    logit halves it; the result is invariant to the scale of o."""
    gamma = np.linspace(0.5, 1.5, 128)
    o = np.full((1, 1, 128), 3.0)
    out = L.post(o, np.zeros((1, 1, 128)), gamma)
    np.testing.assert_allclose(out[0, 0], 0.5 * gamma * 3.0 / np.sqrt(9.0 + L.RMS_EPS),
                               rtol=1e-14)
    r = _rng(5)
    o = r.standard_normal((4, 2, 128))
    g = r.standard_normal((4, 2, 128))
    exact = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True)) * gamma * L.sigmoid(g)
    # far above the epsilon the result no longer depends on the scale of o
    np.testing.assert_allclose(L.post(1e4 * o, g, gamma), exact, rtol=1e-12, atol=1e-15)
    big = L.post(o, np.full_like(g, 60.0), gamma)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + L.RMS_EPS)
    np.testing.assert_allclose(big, o / rms * gamma, rtol=1e-14)
