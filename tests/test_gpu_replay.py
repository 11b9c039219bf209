"""GPU parity of kda_decode_replay (replay of the accepted draft tokens of a
speculative decode step) against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, assert_parity, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def replay_inputs(B, T, H, dtype, seed=0):
    """Cached draft inputs [B, T, H, ...] (the decode generator's T steps)."""
    d = inputs.decode_inputs(B=B, H=H, steps=T, dtype=dtype, device=DEV, seed=seed)
    r = {name: d[name].transpose(0, 1).contiguous()
         for name in ("q", "k", "v", "log_alpha", "beta")}
    r["state"] = d["state"]
    return r


def _oracle(r, n):
    state = r["state"].double().cpu().numpy().copy()
    out = oracle.decode_replay(state, *(r[x].double().cpu().numpy()
                                        for x in ("q", "k", "v", "log_alpha", "beta")), n)
    return out, state


def _check(out, state, ref_out, ref_state, n, T, tol):
    """Accepted rows of every sequence (one row range per sequence, all heads)
    and the states of the sequences with an accepted token, against the oracle
    (whole tensor, every (sequence, head) slice, every row)."""
    nb = np.clip(n, 0, T)
    rows = [(b, t) for b in range(len(nb)) for t in range(int(nb[b]))]
    if rows:
        bi = torch.as_tensor([b for b, _ in rows], device=DEV)
        ti = torch.as_tensor([t for _, t in rows], device=DEV)
        got = out[bi, ti]                                   # [rows, H, 128]
        ref = np.stack([ref_out[b, t] for b, t in rows])
        assert_parity(got, ref, tol, cu=np.concatenate([[0], np.cumsum(nb)]), name="out")
    act = [b for b in range(len(nb)) if nb[b] > 0]
    if act:
        assert_parity(state[torch.as_tensor(act, device=DEV)], ref_state[act], tol, name="state")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_replay_matches_oracle(dtype):
    B, T, H = 5, 4, 3
    r = replay_inputs(B, T, H, dtype, seed=3)
    n = np.array([0, 1, 4, 2, 9], dtype=np.int32)          # 9 > T is clamped to T
    state = r["state"].clone()
    out = torch.full((B, T, H, 128), float("nan"), dtype=r["q"].dtype, device=DEV)
    kda.kda_decode_replay(state, r["q"], r["k"], r["v"], r["log_alpha"], r["beta"],
                          torch.as_tensor(n, device=DEV), out=out)
    torch.cuda.synchronize()
    ref_out, ref_state = _oracle(r, n)
    _check(out, state, ref_out, ref_state, n, T, TOL[dtype])
    for b in range(B):
        nb = min(int(n[b]), T)
        if nb == 0:
            assert torch.equal(state[b], r["state"][b])     # nothing accepted: untouched
        assert torch.isnan(out[b, nb:]).all()               # rejected rows never written


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_replay_more_tokens_than_one_group(dtype):
    """T = 11 drafts: the first 8 accepted tokens come staged with the state, the
    rest in a second group."""
    B, T, H = 4, 11, 2
    r = replay_inputs(B, T, H, dtype, seed=5)
    n = np.array([11, 9, 8, 3], dtype=np.int32)
    state = r["state"].clone()
    out = torch.full((B, T, H, 128), float("nan"), dtype=r["q"].dtype, device=DEV)
    kda.kda_decode_replay(state, r["q"], r["k"], r["v"], r["log_alpha"], r["beta"],
                          torch.as_tensor(n, device=DEV), out=out)
    torch.cuda.synchronize()
    ref_out, ref_state = _oracle(r, n)
    _check(out, state, ref_out, ref_state, n, T, TOL[dtype])
    for b in range(B):
        assert torch.isnan(out[b, int(n[b]):]).all()


def test_replay_each_cta_walks_units_across_skipped_runs():
    """More units than the persistent grid (two CTAs per SM), so every CTA walks
    several units, with a run of sequences that accept nothing longer than two
    grid strides and the last units empty: each CTA's next count is copied a
    unit ahead, and units without accepted tokens are crossed one by one.
    Every unit against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H, T = 1, 3
    B = 8 * sms + 37                                        # about four units per CTA
    g = np.random.default_rng(41)
    n = g.integers(1, T + 1, size=B).astype(np.int32)
    n[50:50 + 6 * sms] = 0
    n[-5:] = 0
    n[[7, 7 + 2 * sms]] = -3                                # clamped to 0
    n[[9, 9 + 2 * sms]] = T + 5                             # clamped to T
    r = replay_inputs(B, T, H, "f32", seed=41)
    state = r["state"].clone()
    out = torch.full((B, T, H, 128), float("nan"), dtype=r["q"].dtype, device=DEV)
    kda.kda_decode_replay(state, r["q"], r["k"], r["v"], r["log_alpha"], r["beta"],
                          torch.as_tensor(n, device=DEV), out=out)
    torch.cuda.synchronize()
    ref_out, ref_state = _oracle(r, n)
    _check(out, state, ref_out, ref_state, n, T, TOL["f32"])
    skipped = torch.as_tensor(np.flatnonzero(n <= 0), device=DEV)
    assert torch.equal(state[skipped], r["state"][skipped])
    assert torch.isnan(out[skipped]).all()


def test_replay_equals_consecutive_decode_steps():
    """Replaying every draft token equals that many kda_decode_step calls."""
    B, T, H = 3, 5, 4
    r = replay_inputs(B, T, H, "bf16", seed=5)
    s1 = r["state"].clone()
    out = kda.kda_decode_replay(s1, r["q"], r["k"], r["v"], r["log_alpha"], r["beta"],
                                torch.full((B,), T, dtype=torch.int32, device=DEV))
    s2 = r["state"].clone()
    outs = [kda.kda_decode_step(s2, *(r[x][:, t].contiguous()
                                      for x in ("q", "k", "v", "log_alpha", "beta")))
            for t in range(T)]
    torch.cuda.synchronize()
    assert rel_l2(s1, s2) <= 1e-6
    assert rel_l2(out, torch.stack(outs, dim=1)) <= 1e-6


def test_replay_without_output_updates_state():
    B, T, H = 2, 3, 2
    r = replay_inputs(B, T, H, "f32", seed=7)
    n = np.array([3, 1], dtype=np.int32)
    state = r["state"].clone()
    assert kda.kda_decode_replay(state, r["q"], r["k"], r["v"], r["log_alpha"], r["beta"],
                                 torch.as_tensor(n, device=DEV), output=False) is None
    torch.cuda.synchronize()
    _, ref_state = _oracle(r, n)
    assert_parity(state, ref_state, TOL["f32"], name="state")


def test_replay_full_size_sampled_units():
    """512 sequences x 96 heads x 4 draft tokens (the benchmark's launch
    configuration) with mixed accepted counts; 48 sampled units against the
    oracle one by one."""
    B, T, H = 512, 4, 96
    r = replay_inputs(B, T, H, "bf16", seed=11)
    g = np.random.default_rng(11)
    n = g.integers(0, T + 1, size=B).astype(np.int32)
    state = r["state"].clone()
    out = kda.kda_decode_replay(state, r["q"], r["k"], r["v"], r["log_alpha"], r["beta"],
                                torch.as_tensor(n, device=DEV))
    torch.cuda.synchronize()
    units = np.sort(g.choice(B * H, size=48, replace=False))
    got_o, ref_o, got_s, ref_s, lens = [], [], [], [], []
    for u in units:
        b, h = divmod(int(u), H)
        nb = int(n[b])
        sub = {x: r[x][b:b + 1, :, h:h + 1] for x in ("q", "k", "v", "log_alpha", "beta")}
        st = r["state"][b:b + 1, h:h + 1].double().cpu().numpy().copy()
        ref_out = oracle.decode_replay(st, *(sub[x].double().cpu().numpy()
                                             for x in ("q", "k", "v", "log_alpha", "beta")),
                                       np.array([nb]))
        if nb:
            got_s.append(state[b, h].double().cpu().numpy())
            ref_s.append(st[0, 0])
            got_o.append(out[b, :nb, h].double().cpu().numpy())
            ref_o.append(ref_out[0, :nb, 0])
            lens.append(nb)
        else:
            assert torch.equal(state[b, h], r["state"][b, h])
    # each sampled unit is its own (sequence, head) slice
    cu = np.concatenate([[0], np.cumsum(lens)])
    assert_parity(np.concatenate(got_o)[:, None], np.concatenate(ref_o)[:, None], TOL["bf16"],
                  cu=cu, name="out")
    assert_parity(np.stack(got_s)[:, None], np.stack(ref_s)[:, None], TOL["bf16"], name="state")
