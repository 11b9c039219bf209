"""Pins for the fp64 oracle against what the pages and the mathematics fix.

Each ``pin_*`` function checks the oracle library it is given and raises
AssertionError on a mismatch.  The tests run them on the real oracle; the
mutation test compiles deliberately broken copies of the oracle source (on the
CPU, in a temporary directory) and checks that every plausible mistake trips at
least one pin.
"""
from __future__ import annotations

import json
import os
import tempfile

import numpy as np
import pytest

import oracle
from oracle import affine

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def random_case(seed, T=7, H=2, dk=5, dv=3, n_seqs=1, init=True, lengths=None):
    r = _rng(seed)
    lengths = lengths or [T] * n_seqs
    N = sum(lengths)
    q = _unit(r.standard_normal((N, H, dk)))
    k = _unit(r.standard_normal((N, H, dk)))
    v = r.standard_normal((N, H, dv))
    la = -5.0 / (1.0 + np.exp(-r.standard_normal((N, H, dk))))
    b = 1.0 / (1.0 + np.exp(-r.standard_normal((N, H))))
    s0 = 0.3 * r.standard_normal((len(lengths), H, dk, dv)) if init else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return dict(q=q, k=k, v=v, log_alpha=la, beta=b, init_state=s0, cu_seqlens=cu)


# --------------------------------------------------------------------------- pins

def pin_delta_rule_1d(lib):
    """AI-Workshop #15 section 7.2: read-out 0.7, target 0.9, beta 0.5 -> 0.8."""
    g = json.load(open(os.path.join(GOLDEN, "delta_rule_1d.json")))
    dk, dv = 4, 2
    k = np.zeros(dk); k[2] = 1.0                        # a unit key (one address)
    S0 = np.zeros((dk, dv)); S0[2, 0] = g["old_readout"]  # k^T S0 = [0.7, 0]
    S0[0, 1] = 5.0                                       # content at another address
    v = np.array([g["target"], 0.0])
    out, fin = oracle.chunk_fwd(q=k.reshape(1, 1, dk), k=k.reshape(1, 1, dk),
                                v=v.reshape(1, 1, dv), log_alpha=np.zeros((1, 1, dk)),
                                beta=np.array([[g["beta"]]]), init_state=S0[None, None],
                                lib=lib)
    np.testing.assert_allclose(out[0, 0, 0], g["new_readout"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(g["target"] - g["old_readout"], g["delta"], atol=1e-15)
    # The other address is untouched by a write along k.
    assert fin[0, 0, 0, 1] == 5.0
    # beta = 1 overwrites: the read-out along k becomes the target exactly.
    out1, _ = oracle.chunk_fwd(q=k.reshape(1, 1, dk), k=k.reshape(1, 1, dk),
                               v=v.reshape(1, 1, dv), log_alpha=np.zeros((1, 1, dk)),
                               beta=np.array([[1.0]]), init_state=S0[None, None], lib=lib)
    np.testing.assert_allclose(out1[0, 0], v, rtol=0, atol=1e-15)


def pin_orthogonal_write_query(lib):
    """AI-Workshop #15 section 7.2 two-address example: S = k1 v1^T + k2 v2^T,
    query k1 returns v1, query k2 returns v2, exactly."""
    g = json.load(open(os.path.join(GOLDEN, "orthogonal_write_query.json")))
    keys = np.array(g["keys"]); vals = np.array(g["values"])
    for qi, query in enumerate(g["queries"]):
        q = np.stack([keys[0], np.array(query)])[:, None, :]
        out, fin = oracle.chunk_fwd(q=q, k=keys[:, None, :], v=vals[:, None, :],
                                    log_alpha=np.full((2, 1, 2), g["log_alpha"]),
                                    beta=np.full((2, 1), g["beta"]), lib=lib)
        assert np.array_equal(out[1, 0], np.array(g["expected_readouts"][qi]))
        assert np.array_equal(fin[0, 0], np.array(g["expected_state"]))


def pin_orthogonal_write_query_d128(lib):
    """Same example lifted to d_k = d_v = 128 with keys e_0, e_1 (exact)."""
    r = _rng(3)
    d = 128
    keys = np.zeros((2, d)); keys[0, 0] = 1.0; keys[1, 1] = 1.0
    vals = np.round(r.standard_normal((2, d)) * 64) / 64  # exact in bf16 and fp64
    for which in (0, 1):
        q = np.stack([keys[0], keys[which]])[:, None, :]
        out, _ = oracle.chunk_fwd(q=q, k=keys[:, None, :], v=vals[:, None, :],
                                  log_alpha=np.zeros((2, 1, d)), beta=np.ones((2, 1)), lib=lib)
        assert np.array_equal(out[1, 0], vals[which])


def pin_beta_zero_closed_form(lib):
    """beta = 0 removes every write: S_t = Diag(exp(sum_{s<=t} log_alpha_s)) S_0."""
    c = random_case(11, T=9, H=2, dk=6, dv=4)
    c["beta"] = np.zeros_like(c["beta"])
    out, fin = oracle.chunk_fwd(**c, lib=lib)
    G = np.cumsum(c["log_alpha"], axis=0)              # [T, H, dk]
    for h in range(2):
        S0 = c["init_state"][0, h]
        for t in range(9):
            St = np.exp(G[t, h])[:, None] * S0
            np.testing.assert_allclose(out[t, h], St.T @ c["q"][t, h], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(fin[0, h], np.exp(G[-1, h])[:, None] * S0,
                                   rtol=1e-13, atol=1e-15)


def pin_alpha_one_orthonormal_linear_attention(lib):
    """alpha = 1, mutually orthonormal keys, S_0 = 0: the erase term never fires,
    so S_t = sum_{i<=t} beta_i k_i v_i^T and o_t = sum_{i<=t} beta_i (k_i.q_t) v_i."""
    r = _rng(5)
    dk, dv, T = 16, 8, 12
    Q, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    k = Q[:, :T].T                                       # T orthonormal keys
    q = _unit(r.standard_normal((T, dk)))
    v = r.standard_normal((T, dv))
    b = r.uniform(0.05, 1.0, T)
    out, fin = oracle.chunk_fwd(q=q[:, None], k=k[:, None], v=v[:, None],
                                log_alpha=np.zeros((T, 1, dk)), beta=b[:, None], lib=lib)
    S = np.zeros((dk, dv))
    for t in range(T):
        S += b[t] * np.outer(k[t], v[t])
        expect = sum(b[i] * (k[i] @ q[t]) * v[i] for i in range(t + 1))
        np.testing.assert_allclose(out[t, 0], expect, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fin[0, 0], S, rtol=1e-12, atol=1e-13)


def pin_bruteforce_affine(lib):
    """Token loop vs explicit transition matrices (prefix-composed affine pairs)."""
    for seed, (dk, dv) in enumerate([(5, 3), (3, 6), (8, 8)]):
        c = random_case(100 + seed, T=7, H=3, dk=dk, dv=dv, n_seqs=1)
        out, fin = oracle.chunk_fwd(**c, lib=lib)
        for h in range(3):
            o_ref, s_ref = affine.chain(c["q"][:, h], c["k"][:, h], c["v"][:, h],
                                        c["log_alpha"][:, h], c["beta"][:, h],
                                        c["init_state"][0, h])
            np.testing.assert_allclose(out[:, h], o_ref, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(fin[0, h], s_ref, rtol=1e-12, atol=1e-13)


def pin_split_invariance(lib):
    """fwd(x[0:t]) -> S_t -> fwd(x[t:T], init=S_t) equals fwd(x[0:T])."""
    c = random_case(21, T=13, H=2, dk=6, dv=5)
    out, fin = oracle.chunk_fwd(**c, lib=lib)
    for cut in (1, 5, 12):
        a = {k: (v[:cut] if k in ("q", "k", "v", "log_alpha", "beta") else v)
             for k, v in c.items()}
        a["cu_seqlens"] = np.array([0, cut])
        o1, s1 = oracle.chunk_fwd(**a, lib=lib)
        b = {k: (v[cut:] if k in ("q", "k", "v", "log_alpha", "beta") else v)
             for k, v in c.items()}
        b["cu_seqlens"] = np.array([0, 13 - cut]); b["init_state"] = s1
        o2, s2 = oracle.chunk_fwd(**b, lib=lib)
        np.testing.assert_allclose(np.concatenate([o1, o2]), out, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(s2, fin, rtol=1e-12, atol=1e-14)


def pin_varlen_equals_separate(lib):
    """A packed call over several sequences equals one call per sequence, and the
    per-sequence state never leaks across a boundary (zero-length sequences too)."""
    lengths = [4, 0, 7, 1]
    c = random_case(31, H=2, dk=5, dv=4, lengths=lengths)
    out, fin = oracle.chunk_fwd(**c, lib=lib)
    cu = c["cu_seqlens"]
    for s, n in enumerate(lengths):
        sl = slice(cu[s], cu[s + 1])
        o_s, f_s = oracle.chunk_fwd(q=c["q"][sl], k=c["k"][sl], v=c["v"][sl],
                                    log_alpha=c["log_alpha"][sl], beta=c["beta"][sl],
                                    init_state=c["init_state"][s:s + 1],
                                    cu_seqlens=np.array([0, n]), lib=lib)
        np.testing.assert_allclose(out[sl], o_s, rtol=0, atol=0)
        np.testing.assert_allclose(fin[s], f_s[0], rtol=0, atol=0)
        # and each sequence also agrees with the brute-force form
        for h in range(2):
            if n == 0:
                np.testing.assert_array_equal(fin[s, h], c["init_state"][s, h])
                continue
            o_ref, s_ref = affine.chain(c["q"][sl, h], c["k"][sl, h], c["v"][sl, h],
                                        c["log_alpha"][sl, h], c["beta"][sl, h],
                                        c["init_state"][s, h])
            np.testing.assert_allclose(o_s[:, h], o_ref, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(f_s[0, h], s_ref, rtol=1e-12, atol=1e-13)


def pin_contraction_bound(lib):
    """With unit keys, beta in [0,1] and alpha in (0,1], every transition has
    spectral norm <= 1, so ||S_t||_F <= ||S_0||_F + sum_i beta_i ||v_i||."""
    c = random_case(41, T=40, H=2, dk=8, dv=8)
    for cut in range(1, 41, 13):
        a = {k: (v[:cut] if k in ("q", "k", "v", "log_alpha", "beta") else v)
             for k, v in c.items()}
        a["cu_seqlens"] = np.array([0, cut])
        _, fin = oracle.chunk_fwd(**a, lib=lib)
        for h in range(2):
            bound = np.linalg.norm(c["init_state"][0, h]) + sum(
                c["beta"][i, h] * np.linalg.norm(c["v"][i, h]) for i in range(cut))
            assert np.linalg.norm(fin[0, h]) <= bound * (1 + 1e-12)


def pin_decode_step(lib):
    """The in-place decode step equals one token of the brute-force form, and T
    decode steps equal the forward pass over the same T tokens."""
    c = random_case(51, T=6, H=3, dk=5, dv=4)
    state = np.ascontiguousarray(c["init_state"].copy())
    outs = []
    for t in range(6):
        outs.append(oracle.decode_step(state, c["q"][t][None], c["k"][t][None], c["v"][t][None],
                                       c["log_alpha"][t][None], c["beta"][t][None], lib=lib)[0])
        if t == 0:
            for h in range(3):
                M, Bm = affine.token_pair(c["k"][0, h], c["v"][0, h], c["log_alpha"][0, h],
                                          c["beta"][0, h])
                S1 = M @ c["init_state"][0, h] + Bm
                np.testing.assert_allclose(state[0, h], S1, rtol=1e-13, atol=1e-15)
                np.testing.assert_allclose(outs[0][h], S1.T @ c["q"][0, h],
                                           rtol=1e-13, atol=1e-15)
    out, fin = oracle.chunk_fwd(**c, lib=lib)
    np.testing.assert_allclose(np.stack(outs), out, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(state, fin, rtol=1e-13, atol=1e-15)


def pin_segment_combine(lib):
    """Segments computed from zero states and combined by a prefix scan over
    affine pairs reproduce the sequential final state and every incoming state."""
    c = random_case(61, T=17, H=1, dk=6, dv=4)
    out, fin = oracle.chunk_fwd(**c, lib=lib)
    h = 0
    S_T, incoming = affine.segmented_state(c["k"][:, h], c["v"][:, h], c["log_alpha"][:, h],
                                           c["beta"][:, h], c["init_state"][0, h], [4, 9, 10])
    np.testing.assert_allclose(S_T, fin[0, h], rtol=1e-12, atol=1e-13)
    for cut, s_in in zip([4, 9, 10], incoming[1:]):
        a = {k: (v[:cut] if k in ("q", "k", "v", "log_alpha", "beta") else v)
             for k, v in c.items()}
        a["cu_seqlens"] = np.array([0, cut])
        _, f_cut = oracle.chunk_fwd(**a, lib=lib)
        np.testing.assert_allclose(s_in, f_cut[0, h], rtol=1e-12, atol=1e-13)


def pin_decode_replay(lib):
    """Replay of accepted draft tokens ("Kimi K3: 架构、训练与系统全景解析", KDA state
    replay under speculative decoding): per sequence, the accepted prefix replayed
    from the cached inputs gives the brute-force transition-matrix outputs and
    final state (oracle.affine); nothing accepted leaves the state untouched; an
    accepted count above T is clamped; rows of rejected tokens stay zero."""
    r = _rng(31)
    B, T, H, dk, dv = 4, 5, 2, 5, 3
    q = _unit(r.standard_normal((B, T, H, dk)))
    k = _unit(r.standard_normal((B, T, H, dk)))
    v = r.standard_normal((B, T, H, dv))
    la = -5.0 / (1.0 + np.exp(-r.standard_normal((B, T, H, dk))))
    b = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, H))))
    s0 = 0.3 * r.standard_normal((B, H, dk, dv))
    n = np.array([0, 2, 5, 7])
    state = s0.copy()
    out = oracle.decode_replay(state, q, k, v, la, b, n, lib=lib)
    for bi in range(B):
        nb = min(int(n[bi]), T)
        assert np.all(out[bi, nb:] == 0.0)
        for h in range(H):
            if nb == 0:
                assert np.array_equal(state[bi, h], s0[bi, h])
                continue
            o_ref, s_ref = affine.chain(q[bi, :nb, h], k[bi, :nb, h], v[bi, :nb, h],
                                        la[bi, :nb, h], b[bi, :nb, h], s0[bi, h])
            np.testing.assert_allclose(out[bi, :nb, h], o_ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(state[bi, h], s_ref, rtol=1e-12, atol=1e-12)


PINS = [pin_delta_rule_1d, pin_orthogonal_write_query, pin_orthogonal_write_query_d128,
        pin_beta_zero_closed_form, pin_alpha_one_orthonormal_linear_attention,
        pin_bruteforce_affine, pin_split_invariance, pin_varlen_equals_separate,
        pin_contraction_bound, pin_decode_step, pin_segment_combine, pin_decode_replay]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_affine_pair_is_associative():
    """The KCP combine is associative (checked on random pairs)."""
    r = _rng(7)
    pairs = [(r.standard_normal((4, 4)), r.standard_normal((4, 3))) for _ in range(3)]
    left = affine.compose(pairs[2], affine.compose(pairs[1], pairs[0]))
    right = affine.compose(affine.compose(pairs[2], pairs[1]), pairs[0])
    for a, b in zip(left, right):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_tile_log_decay_range():
    """With log_alpha >= -5, the cumulative log-decay over a 16-token tile lies in
    [-80, 0] and its inverse exp stays inside the fp32/bf16 exponent range
    ("Kimi K3: 架构、训练与系统全景解析" section 4.2.5)."""
    la = np.full(16, -5.0)
    g = np.cumsum(la)
    assert g.min() >= -80.0 and g.max() <= 0.0
    assert np.isfinite(np.float32(np.exp(-g.min())))          # e^80 < fp32 max
    assert np.exp(80.0) < float(np.finfo(np.float32).max)


# Plausible mistakes, planted in a copy of the oracle source compiled on the CPU.
MUTANTS = {
    "no_erase_term": ("tmp[n] = bt * (vt[n] - tmp[n]);", "tmp[n] = bt * vt[n];", 0),
    "beta_dropped": ("tmp[n] = bt * (vt[n] - tmp[n]);", "tmp[n] = (vt[n] - tmp[n]);", 0),
    "decay_sign": ("const double a = exp(lat[i]);", "const double a = exp(-lat[i]);", 0),
    "decay_skipped": ("for (int64_t n = 0; n < dv; ++n) S[i * dv + n] *= a;",
                      "for (int64_t n = 0; n < dv; ++n) S[i * dv + n] *= 1.0;", 0),
    "erase_with_query": ("const double ki = kt[i];\n            for (int64_t n = 0; n < dv; ++n) S[i * dv + n] += ki * tmp[n];",
                         "const double ki = qt[i];\n            for (int64_t n = 0; n < dv; ++n) S[i * dv + n] += ki * tmp[n];", 0),
    "readout_with_key": ("const double qi = qt[i];", "const double qi = kt[i];", 0),
    "predict_with_query": ("const double ki = kt[i];\n            for (int64_t n = 0; n < dv; ++n) tmp[n] += ki",
                           "const double ki = qt[i];\n            for (int64_t n = 0; n < dv; ++n) tmp[n] += ki", 0),
    "init_state_ignored": ("if (j->init_state) {", "if (0) {", 0),
    "sequence_start_wrong": ("const int64_t t0 = j->cu_seqlens[seq], t1",
                             "const int64_t t0 = j->cu_seqlens[seq > 0 ? seq - 1 : 0], t1", 0),
    "decode_decay_sign": ("const double a = exp(lat[i]);", "const double a = exp(-lat[i]);", 1),
    "decode_readout_before_update": (
        "for (int64_t n = 0; n < dv; ++n) {\n            double acc = 0.0;\n            for (int64_t i = 0; i < dk; ++i) acc += qt[i]",
        "for (int64_t n = 0; n < dv; ++n) {\n            double acc = 0.0;\n            for (int64_t i = 0; i < dk; ++i) acc += kt[i]", 0),
}


def _replace_nth(text, old, new, nth):
    pos = -1
    for _ in range(nth + 1):
        pos = text.find(old, pos + 1)
        if pos < 0:
            raise ValueError(f"pattern not found: {old!r} (occurrence {nth})")
    return text[:pos] + new + text[pos + len(old):]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new, nth = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()
    mutated = _replace_nth(src, old, new, nth)
    path = tmp_path / f"mut_{name}.c"
    path.write_text(mutated)
    lib = oracle.load_library(oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"
