"""The per-token operations either side of the KDA recurrence, in fp64 numpy.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Before the recurrence ("Kimi K3: 架构、训练与系统全景解析", section 4.2.3, and the
"Kimi K3" study notes, section 3-2 "2) Kimi Delta Attention"): a short causal
convolution of kernel size 4 injects local context, Swish adds a smooth
non-linearity, q and k are L2-normalised, beta sets how strongly the token is
written and alpha how much of each channel of the old state is kept; the K3
decay is a lower-bounded scaled sigmoid with bound -5 (全景解析 sections 2.1 and
4.2.5).  After the recurrence (全景解析 section 4.2.6): a head-wise RMSNorm of the
recurrent output, then an input-dependent full-rank sigmoid output gate.

The pages print no formulas for these steps (they are stripped), so each
function states the reading it implements:
  * short_conv: causal depthwise convolution over time within each sequence,
    kernel size 4, y[t] = sum_j w[j] x[t - 3 + j], zero before the sequence start;
  * short_conv_state: the same convolution continuing a sequence across calls:
    the three raw rows before the call's first token come from a carried window
    (oldest first) instead of zeros, and the call returns the window after its
    last token (the last three raw rows of the sequence so far);
  * swish(x) = x * sigmoid(x);
  * l2norm(x) = x / sqrt(sum(x^2) + 1e-6) over the 128 channels of a head;
  * beta = sigmoid(b_logit), log_alpha = -5 * sigmoid(a_logit);
  * rmsnorm(o) = o / sqrt(mean(o^2) + 1e-5) * gamma, gamma one weight per channel
    of the head dimension shared by all heads; out = rmsnorm(o) * sigmoid(g).
"""
from __future__ import annotations

import numpy as np

CONV_K = 4
L2_EPS = 1e-6
RMS_EPS = 1e-5
DECAY_BOUND = -5.0


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def sigmoid(x):
    x = _f64(x)
    return 1.0 / (1.0 + np.exp(-x))


def swish(x):
    x = _f64(x)
    return x * sigmoid(x)


def short_conv(x, w, cu_seqlens):
    """Causal depthwise convolution of ``x`` ``[N, H, d]`` with ``w`` ``[H, d, 4]``
    inside each packed sequence (``cu_seqlens`` ``[n_seqs + 1]``)."""
    x, w = _f64(x), _f64(w)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    y = np.zeros_like(x)
    for s in range(cu.shape[0] - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        for t in range(a, b):
            for j in range(CONV_K):
                src = t - (CONV_K - 1) + j
                if src >= a:
                    y[t] += w[:, :, j] * x[src]
    return y


def short_conv_state(x, w, cu_seqlens, window):
    """``short_conv`` with a carried window: ``window`` ``[n_seqs, 3, H, d]``
    holds, per packed sequence, the three raw rows before its first token in
    this call, oldest first (a fresh sequence has zeros).  Returns ``(y,
    window_out)``, window_out the three raw rows before the token after the
    call: the sequence's last three rows, or, for one shorter than three, the
    old window's newest rows followed by all of its rows."""
    x, w = _f64(x), _f64(w)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    win = _f64(window)
    y = np.zeros_like(x)
    win_out = np.zeros_like(win)
    for s in range(cu.shape[0] - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        ext = np.concatenate([win[s], x[a:b]], axis=0)   # token a - 3 + i at row i
        for t in range(a, b):
            for j in range(CONV_K):
                y[t] += w[:, :, j] * ext[(t - a) + j]
        win_out[s] = ext[-(CONV_K - 1):]
    return y, win_out


def l2norm(x):
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)


def prep(q_raw, k_raw, v_raw, conv_w, a_logit, b_logit, cu_seqlens):
    """q, k, v, log_alpha, beta of the recurrence from the projected inputs.
    ``conv_w`` is ``[3, H, d, 4]`` (q, k, v)."""
    conv_w = _f64(conv_w)
    q = l2norm(swish(short_conv(q_raw, conv_w[0], cu_seqlens)))
    k = l2norm(swish(short_conv(k_raw, conv_w[1], cu_seqlens)))
    v = swish(short_conv(v_raw, conv_w[2], cu_seqlens))
    log_alpha = DECAY_BOUND * sigmoid(a_logit)
    beta = sigmoid(b_logit)
    return q, k, v, log_alpha, beta


def prep_state(q_raw, k_raw, v_raw, conv_w, a_logit, b_logit, cu_seqlens, conv_state):
    """``prep`` continuing each sequence from a carried convolution window:
    ``conv_state`` ``[n_seqs, 3, 3, H, d]`` = (q, k, v) x (three raw rows before
    the call, oldest first).  Returns q, k, v, log_alpha, beta and the window
    after the call, same layout."""
    conv_w = _f64(conv_w)
    st = _f64(conv_state)
    outs, wins = [], []
    for i, x in enumerate((q_raw, k_raw, v_raw)):
        y, wo = short_conv_state(x, conv_w[i], cu_seqlens, st[:, i])
        outs.append(swish(y))
        wins.append(wo)
    q, k = l2norm(outs[0]), l2norm(outs[1])
    v = outs[2]
    log_alpha = DECAY_BOUND * sigmoid(a_logit)
    beta = sigmoid(b_logit)
    return q, k, v, log_alpha, beta, np.stack(wins, axis=1)


def layer_replay(state, conv_state, q_raw, k_raw, v_raw, a_logit, b_logit, g, conv_w, gamma,
                 n_accept, decode_step):
    """Replay of the accepted draft tokens of a speculative step through the
    whole KDA layer between its projections ("Kimi K3: 架构、训练与系统全景解析",
    KDA state replay under speculative decoding: short convolution, norms,
    gates, the recurrence and the output norm are replayed on chip over the
    accepted prefix, and the state and convolution window are written once).
    Per sequence b with n_b = n_accept[b] clamped to [0, T]: ``prep_state`` of
    its first n_b cached raw rows from its window, ``decode_step`` (the oracle's
    token step) n_b times on its state, ``post`` of the outputs.  ``state``
    (C-contiguous fp64 ``[B, H, d, d]``) and ``conv_state`` (fp64
    ``[B, 3, 3, H, d]``) are updated in place; inputs ``[B, T, H, d]`` (b_logit
    ``[B, T, H]``).  Returns out ``[B, T, H, d]``, zero where t >= n_b."""
    q_raw, k_raw, v_raw, a_logit, b_logit, g = (_f64(t) for t in (q_raw, k_raw, v_raw,
                                                                   a_logit, b_logit, g))
    B, T, H, d = q_raw.shape
    n = np.clip(np.asarray(n_accept, dtype=np.int64).reshape(B), 0, T)
    out = np.zeros((B, T, H, d))
    for b in range(B):
        nb = int(n[b])
        if nb == 0:
            continue
        q, k, v, la, be, win = prep_state(q_raw[b, :nb], k_raw[b, :nb], v_raw[b, :nb], conv_w,
                                          a_logit[b, :nb], b_logit[b, :nb], [0, nb],
                                          conv_state[b:b + 1])
        sub = np.ascontiguousarray(state[b:b + 1])
        o = np.stack([decode_step(sub, q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1],
                                  be[t:t + 1])[0] for t in range(nb)])
        state[b] = sub[0]
        conv_state[b] = win[0]
        out[b, :nb] = post(o, g[b, :nb], gamma)
    return out


def post(o, g, gamma):
    """Head-wise RMSNorm of the recurrent output ``o`` ``[N, H, d]`` with weight
    ``gamma`` ``[d]``, times the sigmoid of the gate logits ``g`` ``[N, H, d]``."""
    o, g, gamma = _f64(o), _f64(g), _f64(gamma)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + RMS_EPS)
    return o / rms * gamma * sigmoid(g)
