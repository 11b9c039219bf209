"""GPU parity of kda_decode_step against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _oracle_steps(d, steps, units=None):
    """Oracle decode over ``steps`` steps, on every flat (sequence, head) unit or
    only on the listed ones.  Returns (per-step outputs, final states), both with
    the units on axis 0 and a unit head axis of size 1."""
    B, H = d["state"].shape[:2]
    sel = slice(None) if units is None else units

    def flat(t, s=None):
        a = (t if s is None else t[s]).double().cpu().numpy()
        return np.ascontiguousarray(a.reshape((B * H, 1) + a.shape[2:])[sel])

    state = flat(d["state"])
    outs = [oracle.decode_step(state, flat(d["q"], s), flat(d["k"], s), flat(d["v"], s),
                               flat(d["log_alpha"], s), flat(d["beta"], s))
            for s in range(steps)]
    return outs, state


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_steps_match_oracle(dtype):
    d = inputs.decode_inputs(B=3, H=5, steps=4, dtype=dtype, device=DEV)
    state = d["state"].clone()
    outs = []
    for s in range(4):
        outs.append(kda.kda_decode_step(state, d["q"][s], d["k"][s], d["v"][s],
                                        d["log_alpha"][s], d["beta"][s]).clone())
    torch.cuda.synchronize()
    ref_outs, ref_state = _oracle_steps(d, 4)
    for s in range(4):
        assert rel_l2(outs[s].reshape(15, 1, 128), ref_outs[s]) <= TOL[dtype]
    assert rel_l2(state.reshape(15, 1, 128, 128), ref_state) <= TOL[dtype]


def test_decode_full_size_sampled_units():
    """512 sequences x 96 heads (the benchmark's launch configuration), one step;
    64 sampled (sequence, head) units checked against the oracle one by one."""
    d = inputs.decode_inputs(B=512, H=96, steps=1, dtype="bf16", device=DEV)
    state0 = d["state"]
    state = state0.clone()
    out = kda.kda_decode_step(state, d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0],
                              d["beta"][0])
    torch.cuda.synchronize()
    g = np.random.default_rng(0)
    units = np.sort(g.choice(512 * 96, size=64, replace=False))
    ref_outs, ref_state = _oracle_steps(d, 1, units=units)
    got_out = out.reshape(512 * 96, 1, 128)[torch.as_tensor(units, device=DEV)]
    got_state = state.reshape(512 * 96, 1, 128, 128)[torch.as_tensor(units, device=DEV)]
    assert rel_l2(got_out, ref_outs[0]) <= TOL["bf16"]
    assert rel_l2(got_state, ref_state) <= TOL["bf16"]
    # and every unit was written: the new state differs from the old one everywhere
    # a token with beta > 0 arrived (beta = sigmoid(N(0,1)) is never 0).
    changed = (state != state0).reshape(512 * 96, -1).any(dim=1)
    assert bool(changed.all())


@pytest.mark.parametrize("case", ["beta0", "beta1", "la0", "la_floor"])
def test_decode_edge_values(case):
    d = inputs.decode_inputs(B=4, H=3, steps=1, dtype="f32", device=DEV)
    if case == "beta0":
        d["beta"].zero_()
    elif case == "beta1":
        d["beta"].fill_(1.0)
    elif case == "la0":
        d["log_alpha"].zero_()
    else:
        d["log_alpha"].fill_(-5.0)
    state = d["state"].clone()
    out = kda.kda_decode_step(state, d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0],
                              d["beta"][0])
    torch.cuda.synchronize()
    ref_outs, ref_state = _oracle_steps(d, 1)
    assert rel_l2(out.reshape(12, 1, 128), ref_outs[0]) <= TOL["f32"]
    assert rel_l2(state.reshape(12, 1, 128, 128), ref_state) <= TOL["f32"]


def test_decode_deterministic():
    d = inputs.decode_inputs(B=8, H=4, steps=1, dtype="bf16", device=DEV)
    a, b = d["state"].clone(), d["state"].clone()
    oa = kda.kda_decode_step(a, d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0])
    ob = kda.kda_decode_step(b, d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0])
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(oa, ob)
