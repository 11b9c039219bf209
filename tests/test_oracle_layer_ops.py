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


# ---- the convolution window carried across calls, and the fused layer replay

def test_conv_window_of_zeros_equals_the_plain_convolution():
    r = _rng(11)
    lengths = [0, 1, 2, 3, 9]
    H, d = 2, 5
    cu = np.concatenate([[0], np.cumsum(lengths)])
    w = r.standard_normal((H, d, 4))
    x = r.standard_normal((cu[-1], H, d))
    y, win = L.short_conv_state(x, w, cu, np.zeros((len(lengths), 3, H, d)))
    np.testing.assert_array_equal(y, L.short_conv(x, w, cu))
    # the window after the call: the last three raw rows, zeros before the start
    for s, n in enumerate(lengths):
        for i in range(3):
            t = n - 3 + i
            want = x[cu[s] + t] if t >= 0 else np.zeros((H, d))
            np.testing.assert_array_equal(win[s, i], want)


def test_conv_window_closed_form_on_zero_input():
    """Zero input after a carried window s0, s1, s2 (oldest first): the taps read
    the window, y[0] = w0 s0 + w1 s1 + w2 s2, y[1] = w0 s1 + w1 s2, y[2] = w0 s2,
    then nothing; the window shifts in the zero rows."""
    r = _rng(12)
    H, d, T = 1, 3, 5
    w = r.standard_normal((H, d, 4))
    s = r.standard_normal((1, 3, H, d))
    y, win = L.short_conv_state(np.zeros((T, H, d)), w, [0, T], s)
    w0, w1, w2 = w[..., 0], w[..., 1], w[..., 2]
    np.testing.assert_allclose(y[0], w0 * s[0, 0] + w1 * s[0, 1] + w2 * s[0, 2], rtol=1e-15)
    np.testing.assert_allclose(y[1], w0 * s[0, 1] + w1 * s[0, 2], rtol=1e-15)
    np.testing.assert_allclose(y[2], w0 * s[0, 2], rtol=1e-15)
    assert not y[3:].any() and not win.any()
    # a one-token call keeps the newest two rows of the window, then the token
    x1 = r.standard_normal((1, H, d))
    _, win1 = L.short_conv_state(x1, w, [0, 1], s)
    np.testing.assert_array_equal(win1[0], np.stack([s[0, 1], s[0, 2], x1[0]]))


def test_prep_split_at_any_token_with_the_carried_window_equals_one_call():
    """prep of x[0:t] then prep of x[t:T] from the window the first call returned
    equals prep of x[0:T], for cuts inside, before and at the kernel width, and
    a two-call chain of one-token pieces."""
    r = _rng(13)
    T, H, d = 11, 2, 8
    x = {n: r.standard_normal((T, H, d)) for n in ("q", "k", "v", "a")}
    b = r.standard_normal((T, H))
    cw = r.standard_normal((3, H, d, 4))
    full = L.prep(x["q"], x["k"], x["v"], cw, x["a"], b, [0, T])
    zero = np.zeros((1, 3, 3, H, d))
    for cut in (0, 1, 2, 3, 4, 7, T):
        first = L.prep_state(x["q"][:cut], x["k"][:cut], x["v"][:cut], cw, x["a"][:cut], b[:cut],
                             [0, cut], zero)
        second = L.prep_state(x["q"][cut:], x["k"][cut:], x["v"][cut:], cw, x["a"][cut:],
                              b[cut:], [0, T - cut], first[5])
        for i in range(5):
            np.testing.assert_allclose(np.concatenate([first[i], second[i]]), full[i],
                                       rtol=1e-14, atol=1e-15)
    # token by token, as decode calls it
    win = zero
    for t in range(T):
        step = L.prep_state(x["q"][t:t + 1], x["k"][t:t + 1], x["v"][t:t + 1], cw,
                            x["a"][t:t + 1], b[t:t + 1], [0, 1], win)
        win = step[5]
        for i in range(5):
            np.testing.assert_allclose(step[i][0], full[i][t], rtol=1e-14, atol=1e-15)


def test_layer_replay_equals_prep_recurrence_post_chain():
    """The fused replay against the unfused chain run independently: prep with
    the window, the C oracle's chunk loop (a different code path from its
    decode step) from the state, then post; rejected tokens leave nothing,
    nothing accepted leaves state and window untouched, counts above T clamp."""
    import oracle
    r = _rng(14)
    B, T, H, d = 4, 5, 2, 128
    raw = {n: r.standard_normal((B, T, H, d)) for n in ("q", "k", "v", "a", "g")}
    bl = r.standard_normal((B, T, H))
    cw = 0.5 * r.standard_normal((3, H, d, 4))
    gamma = 1 + 0.1 * r.standard_normal(d)
    state0 = 0.02 * r.standard_normal((B, H, d, d))
    win0 = r.standard_normal((B, 3, 3, H, d))
    n = np.array([3, 0, 9, 1])
    state, win = state0.copy(), win0.copy()
    out = L.layer_replay(state, win, raw["q"], raw["k"], raw["v"], raw["a"], bl, raw["g"], cw,
                         gamma, n, oracle.decode_step)
    for b in range(B):
        nb = min(int(n[b]), T)
        if nb == 0:
            np.testing.assert_array_equal(state[b], state0[b])
            np.testing.assert_array_equal(win[b], win0[b])
            assert not out[b].any()
            continue
        q, k, v, la, be, w_ref = L.prep_state(raw["q"][b, :nb], raw["k"][b, :nb],
                                              raw["v"][b, :nb], cw, raw["a"][b, :nb],
                                              bl[b, :nb], [0, nb], win0[b:b + 1])
        o, fin = oracle.chunk_fwd(q, k, v, la, be, state0[b:b + 1], [0, nb])
        np.testing.assert_allclose(out[b, :nb], L.post(o, raw["g"][b, :nb], gamma),
                                   rtol=1e-10, atol=1e-12)
        assert not out[b, nb:].any()
        np.testing.assert_allclose(state[b], fin[0], rtol=1e-11, atol=1e-14)
        np.testing.assert_array_equal(win[b], w_ref[0])
