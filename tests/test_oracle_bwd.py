"""Pins of the oracle's gradient (oracle/kda_oracle_bwd.c) against what fixes
it independently of its own code: central finite differences of the forward
oracle, the transposed transition product of the brute-force affine form, and
closed forms without writes.  A mutation test plants plausible mistakes in a
copy of the gradient source and checks that each fails a pin."""
from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from oracle import affine

HERE = os.path.dirname(os.path.abspath(__file__))


def _rng(seed):
    return np.random.default_rng(seed)


def _problem(seed, lengths=(7, 0, 3), H=2, dk=4, dv=3, init=True):
    """A tiny packed problem with unit keys, beta in (0, 1), log_alpha in
    (-1, 0) and random output / final-state gradients (dk != dv, so that a
    transposition shows)."""
    r = _rng(seed)
    N = int(sum(lengths))
    x = dict(q=r.standard_normal((N, H, dk)), k=r.standard_normal((N, H, dk)),
             v=r.standard_normal((N, H, dv)), la=-r.random((N, H, dk)),
             b=0.1 + 0.8 * r.random((N, H)),
             s0=r.standard_normal((len(lengths), H, dk, dv)) if init else None,
             cu=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64),
             do=r.standard_normal((N, H, dv)), df=r.standard_normal((len(lengths), H, dk, dv)))
    x["k"] /= np.linalg.norm(x["k"], axis=-1, keepdims=True)
    return x


def _grads(lib, x, do=None, df="same"):
    return oracle.chunk_bwd(x["q"], x["k"], x["v"], x["la"], x["b"], x["s0"], x["cu"],
                            x["do"] if do is None else do, x["df"] if df == "same" else df,
                            lib=lib)


def pin_finite_differences(lib):
    """Every gradient equals the central difference of the forward oracle's
    loss L = <d_out, out> + <d_final, final_state>, element by element."""
    x = _problem(1)
    g = _grads(lib, x)
    names = ("q", "k", "v", "la", "b", "s0")

    def loss(vals):
        o, f = oracle.chunk_fwd(vals["q"], vals["k"], vals["v"], vals["la"], vals["b"],
                                vals["s0"], x["cu"])
        return float((o * x["do"]).sum() + (f * x["df"]).sum())

    eps = 1e-6
    for name, grad in zip(names, g):
        base = x[name]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            vals = {n: x[n] for n in names}
            plus, minus = base.copy(), base.copy()
            plus[idx] += eps
            minus[idx] -= eps
            vals[name] = plus
            lp = loss(vals)
            vals[name] = minus
            num[idx] = (lp - loss(vals)) / (2 * eps)
        scale = 1.0 + np.abs(num).max()
        assert np.abs(num - grad).max() <= 1e-6 * scale, name


def pin_affine_transpose(lib):
    """With no output gradient, the gradient reaching the initial state is the
    transposed product of the transitions applied to d_final, and each value's
    gradient is beta_t (M_{T..t+1} k_t)^T d_final (v enters only through the
    write beta k v^T), both from explicit dense transition matrices."""
    x = _problem(2, lengths=(6,), H=1, dk=5, dv=3)
    g = _grads(lib, x, do=np.zeros_like(x["do"]))
    k, v, la, b = x["k"][:, 0], x["v"][:, 0], x["la"][:, 0], x["b"][:, 0]
    M, _ = affine.segment_pair(k, v, la, b)
    np.testing.assert_allclose(g[5][0, 0], M.T @ x["df"][0, 0], rtol=1e-12, atol=1e-12)
    T = k.shape[0]
    for t in range(T):
        later, _ = affine.segment_pair(k[t + 1:], v[t + 1:], la[t + 1:], b[t + 1:])
        want = b[t] * (later @ k[t]) @ x["df"][0, 0]
        np.testing.assert_allclose(g[2][t, 0], want, rtol=1e-11, atol=1e-12)
    assert not g[0].any()                                  # no read-out gradient, no dq


def pin_no_writes_closed_form(lib):
    """beta = 0: S_T = Diag(e^{sum_t log_alpha_t}) S_0, so with only a final-state
    gradient every token's log_alpha gradient is sum_n d_final Gamma S_0 (the
    same for every t), d_init = Diag(Gamma) d_final, and q, k, v get nothing."""
    x = _problem(3, lengths=(5,), H=1, dk=4, dv=3)
    x["b"] = np.zeros_like(x["b"])
    g = _grads(lib, x, do=np.zeros_like(x["do"]))
    gam = np.exp(x["la"][:, 0].sum(axis=0))                # [dk]
    s0, df = x["s0"][0, 0], x["df"][0, 0]
    want_la = (df * gam[:, None] * s0).sum(axis=1)
    for t in range(5):
        np.testing.assert_allclose(g[3][t, 0], want_la, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g[5][0, 0], gam[:, None] * df, rtol=1e-13, atol=1e-14)
    for i in (0, 1, 2):
        assert not g[i].any()


def pin_readout_gradient(lib):
    """Only the output of token t carries a gradient: dq_t = S_t do_t with S_t
    the forward oracle's final state of the prefix [0, t] (a separate run)."""
    x = _problem(4, lengths=(6,), H=1, dk=4, dv=3)
    t = 3
    do = np.zeros_like(x["do"])
    do[t] = x["do"][t]
    g = _grads(lib, x, do=do, df=None)
    _, s_t = oracle.chunk_fwd(x["q"][:t + 1], x["k"][:t + 1], x["v"][:t + 1], x["la"][:t + 1],
                              x["b"][:t + 1], x["s0"], [0, t + 1])
    np.testing.assert_allclose(g[0][t, 0], s_t[0, 0] @ do[t, 0], rtol=1e-12, atol=1e-13)
    assert not g[0][t + 1:].any() and not g[0][:t].any()


def pin_sequences_are_independent(lib):
    """Packed sequences (one of them empty) equal separate calls."""
    x = _problem(5, lengths=(4, 0, 3))
    g = _grads(lib, x)
    for s in range(3):
        a, e = x["cu"][s], x["cu"][s + 1]
        gs = oracle.chunk_bwd(x["q"][a:e], x["k"][a:e], x["v"][a:e], x["la"][a:e], x["b"][a:e],
                              x["s0"][s:s + 1], [0, e - a], x["do"][a:e], x["df"][s:s + 1], lib=lib)
        for i in range(5):
            np.testing.assert_allclose(g[i][a:e], gs[i], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(g[5][s], gs[5][0], rtol=1e-13, atol=1e-14)


PINS = [pin_finite_differences, pin_affine_transpose, pin_no_writes_closed_form,
        pin_readout_gradient, pin_sequences_are_independent]


@pytest.fixture(scope="module")
def bwd_lib():
    oracle.build()
    return oracle.load_bwd_library(oracle._LIB_BWD_PATH)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_gradient_pin(pin, bwd_lib):
    pin(bwd_lib)


def test_long_sequence_recomputation_blocks():
    """Sequences longer than the oracle's recomputation block (64 tokens): the
    gradient matches finite differences on a few sampled elements."""
    x = _problem(6, lengths=(150,), H=1, dk=4, dv=3)
    g = oracle.chunk_bwd(x["q"], x["k"], x["v"], x["la"], x["b"], x["s0"], x["cu"], x["do"],
                         x["df"])
    eps = 1e-6

    def loss(name, idx, delta):
        vals = {n: x[n].copy() if n == name else x[n] for n in ("q", "k", "v", "la", "b", "s0")}
        vals[name][idx] += delta
        o, f = oracle.chunk_fwd(vals["q"], vals["k"], vals["v"], vals["la"], vals["b"],
                                vals["s0"], x["cu"])
        return float((o * x["do"]).sum() + (f * x["df"]).sum())

    for name, gi, idx in (("q", 0, (10, 0, 2)), ("k", 1, (63, 0, 1)), ("k", 1, (64, 0, 3)),
                          ("v", 2, (127, 0, 0)), ("la", 3, (1, 0, 2)), ("b", 4, (149, 0))):
        num = (loss(name, idx, eps) - loss(name, idx, -eps)) / (2 * eps)
        assert abs(num - g[gi][idx]) <= 1e-6 * (1 + abs(num)), (name, idx)


MUTANTS = {
    "readout_grad_dropped": ("w->dS[i * dv + n] += q[i] * dout[n];", "w->dS[i * dv + n] += 0.0;"),
    "dq_from_decayed_state": ("acc += (X[i * dv + n] + k[i] * d[n]) * dout[n];",
                              "acc += X[i * dv + n] * dout[n];"),
    "dp_sign": ("const double dp = -b * dd[n];", "const double dp = b * dd[n];"),
    "no_decay_backprop": ("w->dS[i * dv + n] = al * w->dX[i * dv + n];",
                          "w->dS[i * dv + n] = w->dX[i * dv + n];"),
    "dla_wrong_operand": ("la_acc += dx * X[i * dv + n];",
                          "la_acc += w->dS[i * dv + n] * X[i * dv + n];"),
    "dbeta_without_prediction": ("db += dd[n] * (v[n] - p[n]);", "db += dd[n] * v[n];"),
    "dk_missing_prediction_term": ("dkk[i] += acc;", "dkk[i] += 0.0 * acc;"),
    "dv_without_beta": ("dvv[n] = b * dd[n];", "dvv[n] = dd[n];"),
    "dd_transposed_key": ("dd[n] += w->dS[i * dv + n] * k[i];", "dd[n] += w->dS[i * dv + n] * q[i];"),
    "final_grad_ignored": ("if (j->d_final) memcpy", "if (0) memcpy"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle_bwd.c")).read()
    assert src.count(old) == 1, old
    path = tmp_path / f"mut_{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load_bwd_library(oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"
