"""Brute-force KDA by explicit transition matrices (affine pairs).

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  Tiny sizes only: it builds
dense ``dk x dk`` matrices per token.

Every token acts on the incoming state as an affine map

    S_t = M_t S_{t-1} + B_t,   M_t = (I - beta_t k_t k_t^T) Diag(exp(log_alpha_t)),
                               B_t = beta_t k_t v_t^T

("Kimi K3" study notes, section 3-2 "2) Kimi Delta Attention", update
equation).  A run of tokens is therefore one pair (M, B) acting as
S_out = M S_in + B, and pairs compose associatively:

    (M2, B2) o (M1, B1) = (M2 M1, M2 B1 + B2)

("Kimi K3: 架构、训练与系统全景解析" section 7.1, cross-device KCP: each segment
is a cumulative transition plus the local write from a zero state, and a prefix
scan over such pairs recovers every segment's incoming state).  The state after
t tokens is read off the composed prefix pair, never by stepping S itself:

    S_t = (M_t ... M_1) S_0 + sum_i (M_t ... M_{i+1}) B_i,   o_t = S_t^T q_t.
"""
from __future__ import annotations

import numpy as np


def token_pair(k_t, v_t, log_alpha_t, beta_t):
    """The affine pair (M_t, B_t) of one token, materialised densely."""
    k_t = np.asarray(k_t, dtype=np.float64)
    v_t = np.asarray(v_t, dtype=np.float64)
    dk = k_t.shape[0]
    erase = np.eye(dk) - beta_t * np.outer(k_t, k_t)
    M = erase @ np.diag(np.exp(np.asarray(log_alpha_t, dtype=np.float64)))
    B = beta_t * np.outer(k_t, v_t)
    return M, B


def compose(later, earlier):
    """(M2, B2) o (M1, B1): apply ``earlier`` first, then ``later``."""
    M2, B2 = later
    M1, B1 = earlier
    return M2 @ M1, M2 @ B1 + B2


def identity_pair(dk, dv):
    return np.eye(dk), np.zeros((dk, dv))


def segment_pair(k, v, log_alpha, beta):
    """Composed pair of a whole segment ``[T, dk]`` / ``[T, dv]`` / ``[T]``."""
    dk, dv = k.shape[1], v.shape[1]
    acc = identity_pair(dk, dv)
    for t in range(k.shape[0]):
        acc = compose(token_pair(k[t], v[t], log_alpha[t], beta[t]), acc)
    return acc


def chain(q, k, v, log_alpha, beta, S0=None):
    """One (sequence, head) chain.  q, k, log_alpha ``[T, dk]``, v ``[T, dv]``,
    beta ``[T]``.  Returns (out ``[T, dv]``, S_T ``[dk, dv]``)."""
    q, k, v, log_alpha, beta = (np.asarray(x, dtype=np.float64)
                                for x in (q, k, v, log_alpha, beta))
    T, dk = k.shape
    dv = v.shape[1]
    S0 = np.zeros((dk, dv)) if S0 is None else np.asarray(S0, dtype=np.float64)
    prefix = identity_pair(dk, dv)
    out = np.zeros((T, dv))
    for t in range(T):
        prefix = compose(token_pair(k[t], v[t], log_alpha[t], beta[t]), prefix)
        S_t = prefix[0] @ S0 + prefix[1]
        out[t] = S_t.T @ q[t]
    S_T = prefix[0] @ S0 + prefix[1]
    return out, S_T


def segmented_state(k, v, log_alpha, beta, S0, boundaries):
    """Final state from segment pairs combined by an exclusive prefix scan.

    ``boundaries`` are token indices splitting ``[0, T)`` into segments; each
    segment's pair is built from a zero state on its own, then the pairs are
    composed left to right (the KCP combine), and the result applied to S0.
    """
    T = k.shape[0]
    cuts = [0, *boundaries, T]
    pairs = [segment_pair(k[a:b], v[a:b], log_alpha[a:b], beta[a:b])
             for a, b in zip(cuts[:-1], cuts[1:])]
    acc = identity_pair(k.shape[1], v.shape[1])
    incoming = []
    for p in pairs:
        incoming.append(acc[0] @ S0 + acc[1])
        acc = compose(p, acc)
    return acc[0] @ S0 + acc[1], incoming
