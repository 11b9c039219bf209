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


def post(o, g, gamma):
    """Head-wise RMSNorm of the recurrent output ``o`` ``[N, H, d]`` with weight
    ``gamma`` ``[d]``, times the sigmoid of the gate logits ``g`` ``[N, H, d]``."""
    o, g, gamma = _f64(o), _f64(g), _f64(gamma)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + RMS_EPS)
    return o / rms * gamma * sigmoid(g)
