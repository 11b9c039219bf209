"""GPU parity of kda_decode_step against the fp64 oracle (whole tensor, every
(sequence, head) unit and every row)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, assert_parity

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


def _cmp(got, ref, tol, name):
    """Units on axis 0 (each its own sequence), a unit head axis."""
    got = got.reshape(ref.shape)
    return assert_parity(got, ref, tol, cu=None if got.ndim == 4 else np.arange(ref.shape[0] + 1),
                         name=name)


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
        _cmp(outs[s], ref_outs[s], TOL[dtype], f"out, step {s}")
    _cmp(state, ref_state, TOL[dtype], "state")


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
    _cmp(got_out, ref_outs[0], TOL["bf16"], "out")
    _cmp(got_state, ref_state, TOL["bf16"], "state")
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
    _cmp(out, ref_outs[0], TOL["f32"], "out")
    _cmp(state, ref_state, TOL["f32"], "state")


def test_decode_deterministic():
    d = inputs.decode_inputs(B=8, H=4, steps=1, dtype="bf16", device=DEV)
    a, b = d["state"].clone(), d["state"].clone()
    oa = kda.kda_decode_step(a, d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0])
    ob = kda.kda_decode_step(b, d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0])
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(oa, ob)


def test_decode_100_steps_in_place_sampled_units():
    """The decode workload as specified: 512 sequences x 96 heads, 100
    consecutive steps with fresh inputs each, the fp32 state advanced in place
    by every step.  48 sampled (sequence, head) units are replayed by the oracle
    over all 100 steps: every step's output and the final state must match."""
    steps = 100
    d = inputs.decode_inputs(B=512, H=96, steps=steps, dtype="bf16", device=DEV, seed=5)
    state = d["state"].clone()
    out = torch.empty(steps, 512, 96, 128, dtype=torch.bfloat16, device=DEV)
    for s in range(steps):
        kda.kda_decode_step(state, d["q"][s], d["k"][s], d["v"][s], d["log_alpha"][s],
                            d["beta"][s], out=out[s])
    torch.cuda.synchronize()
    g = np.random.default_rng(5)
    units = np.sort(g.choice(512 * 96, size=48, replace=False))
    usel = torch.as_tensor(units, device=DEV)
    ref_outs, ref_state = _oracle_steps(d, steps, units=units)
    got = out.reshape(steps, 512 * 96, 1, 128).index_select(1, usel)
    # all steps at once: rows = (step, unit), each unit's 100 rows one sequence
    got_all = got.permute(1, 0, 2, 3).reshape(48 * steps, 1, 128)
    ref_all = np.stack(ref_outs, axis=1).reshape(48 * steps, 1, 128)
    assert_parity(got_all, ref_all, TOL["bf16"], cu=np.arange(49) * steps, name="out, 100 steps")
    _cmp(state.reshape(512 * 96, 1, 128, 128)[usel], ref_state, TOL["bf16"], "state after 100 steps")
    del d, out, state
    torch.cuda.empty_cache()
