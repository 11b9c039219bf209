"""The convolution window carried across calls (kda_prep_fwd_state) and the
fused layer replay over accepted draft tokens (kda_layer_replay), against the
fp64 oracle and against the unfused GPU path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import layer_ops as L
from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, assert_parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GATE_TOL = 1e-5


def _np(t):
    return t.double().cpu().numpy()


def _window(n_seqs, H, dtype, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(n_seqs, 3, 3, H, 128, generator=g, device=DEV).to(inputs.torch_dtype(dtype))


def _prep_state(x, cu, w_in, w_out):
    return kda.kda_prep_fwd_state(x["q_raw"], x["k_raw"], x["v_raw"], x["conv_w"], x["a_logit"],
                                  x["b_logit"], cu, w_in, w_out)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("with_window", [True, False])
def test_prep_state_matches_oracle(dtype, with_window):
    lengths = [0, 1, 2, 3, 5, 40, 70]
    H = 3
    x = inputs.layer_inputs(lengths, H=H, dtype=dtype, device=DEV, seed=51)
    cu = x["cu_seqlens"]
    w_in = _window(len(lengths), H, dtype, 52) if with_window else None
    w_out = torch.full((len(lengths), 3, 3, H, 128), float("nan"), device=DEV,
                       dtype=inputs.torch_dtype(dtype))
    q, k, v, la, beta = _prep_state(x, cu, w_in, w_out)
    torch.cuda.synchronize()
    ref_w = np.zeros((len(lengths), 3, 3, H, 128)) if w_in is None else _np(w_in)
    ref = L.prep_state(_np(x["q_raw"]), _np(x["k_raw"]), _np(x["v_raw"]), _np(x["conv_w"]),
                       _np(x["a_logit"]), _np(x["b_logit"]), _np(cu).astype(np.int64), ref_w)
    cu_np = _np(cu).astype(np.int64)
    for name, got, want in zip("qkv", (q, k, v), ref[:3]):
        assert_parity(got, want, TOL[dtype], cu=cu_np, name=name)
    assert_parity(la, ref[3], GATE_TOL, cu=cu_np, name="log_alpha")
    assert_parity(beta[..., None], ref[4][..., None], GATE_TOL, cu=cu_np, name="beta")
    # the window holds raw rows: exactly the oracle's (same values, same dtype)
    want_w = torch.as_tensor(ref[5]).to(device=DEV, dtype=w_out.dtype)
    assert torch.equal(w_out, want_w)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prep_split_across_calls_equals_one_call_bitwise(dtype):
    """One long sequence per slot, cut at several points: the calls with the
    carried window give the one-call results bit for bit, the window updated
    in place."""
    T, H = 150, 4
    x = inputs.layer_inputs([T, T], H=H, dtype=dtype, device=DEV, seed=53)
    full = kda.kda_prep_fwd(x["q_raw"], x["k_raw"], x["v_raw"], x["conv_w"], x["a_logit"],
                            x["b_logit"], x["cu_seqlens"])
    for cuts in ([0, 1, 2, 3, 150], [0, 64, 65, 127, 150], [0, 33, 150]):
        win = torch.zeros(2, 3, 3, H, 128, device=DEV, dtype=inputs.torch_dtype(dtype))
        parts = [[] for _ in range(5)]
        for a, b in zip(cuts[:-1], cuts[1:]):
            # both sequences advance by the same piece: rows [a, b) of each
            idx = torch.cat([torch.arange(a, b), T + torch.arange(a, b)]).to(DEV)
            y = {n: x[n].index_select(0, idx).contiguous() for n in
                 ("q_raw", "k_raw", "v_raw", "a_logit", "b_logit")}
            y["conv_w"] = x["conv_w"]
            cu = torch.tensor([0, b - a, 2 * (b - a)], dtype=torch.int32, device=DEV)
            out = _prep_state(y, cu, win, win)
            for i in range(5):
                parts[i].append((out[i][: b - a], out[i][b - a:]))
        torch.cuda.synchronize()
        for i in range(5):
            got = torch.cat([torch.cat([p[0] for p in parts[i]]), torch.cat([p[1] for p in parts[i]])])
            assert torch.equal(got, full[i]), (cuts, i)


def test_prep_state_one_token_calls_like_decode():
    """Decode-style calls: every sequence one token per call, the window in
    place; after T calls the outputs are those of one prefill, bit for bit."""
    B, T, H = 6, 9, 2
    x = inputs.layer_inputs([T] * B, H=H, dtype="bf16", device=DEV, seed=54)
    full = kda.kda_prep_fwd(x["q_raw"], x["k_raw"], x["v_raw"], x["conv_w"], x["a_logit"],
                            x["b_logit"], x["cu_seqlens"])
    win = torch.zeros(B, 3, 3, H, 128, device=DEV, dtype=torch.bfloat16)
    cu = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    for t in range(T):
        idx = (torch.arange(B) * T + t).to(DEV)
        y = {n: x[n].index_select(0, idx).contiguous() for n in
             ("q_raw", "k_raw", "v_raw", "a_logit", "b_logit")}
        y["conv_w"] = x["conv_w"]
        out = _prep_state(y, cu, win, win)
        for i in range(5):
            assert torch.equal(out[i], full[i].index_select(0, idx)), (t, i)


def replay_layer_inputs(B, T, H, dtype, seed):
    x = inputs.layer_inputs([T] * B, H=H, dtype=dtype, device=DEV, seed=seed)
    r = {n: x[n].reshape(B, T, H, *x[n].shape[2:]).contiguous()
         for n in ("q_raw", "k_raw", "v_raw", "a_logit", "b_logit", "g")}
    r["conv_w"], r["gamma"] = x["conv_w"], x["gamma"]
    g = torch.Generator(device=DEV).manual_seed(seed + 1)
    r["state"] = 0.02 * torch.randn(B, H, 128, 128, generator=g, device=DEV)
    r["window"] = _window(B, H, dtype, seed + 2)
    return r


def _oracle_replay(r, n):
    state = _np(r["state"]).copy()
    win = _np(r["window"]).copy()
    out = L.layer_replay(state, win, *(_np(r[x]) for x in ("q_raw", "k_raw", "v_raw", "a_logit",
                                                             "b_logit", "g", "conv_w", "gamma")),
                         n, oracle.decode_step)
    return out, state, win


def _check_replay(r, n, out, state, win, T, tol):
    ref_out, ref_state, ref_win = _oracle_replay(r, n)
    nb = np.clip(n, 0, T)
    rows = [(b, t) for b in range(len(nb)) for t in range(int(nb[b]))]
    bi = torch.as_tensor([b for b, _ in rows], device=DEV)
    ti = torch.as_tensor([t for _, t in rows], device=DEV)
    assert_parity(out[bi, ti], np.stack([ref_out[b, t] for b, t in rows]), tol,
                  cu=np.concatenate([[0], np.cumsum(nb)]), name="layer output")
    act = [b for b in range(len(nb)) if nb[b] > 0]
    assert_parity(state[torch.as_tensor(act, device=DEV)], ref_state[act], tol, name="state")
    want_w = torch.as_tensor(ref_win).to(device=DEV, dtype=win.dtype)
    assert torch.equal(win, want_w)                      # raw rows, exactly
    for b in range(len(nb)):
        assert torch.isnan(out[b, int(nb[b]):]).all()     # rejected rows never written
        if nb[b] == 0:
            assert torch.equal(state[b], r["state"][b]) and torch.equal(win[b], r["window"][b])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [4, 7])
def test_layer_replay_matches_oracle(dtype, T):
    B, H = 5, 3
    r = replay_layer_inputs(B, T, H, dtype, seed=55 + T)
    n = np.array([0, 1, T, 2, 9], dtype=np.int32)        # 9 > T is clamped to T
    state, win = r["state"].clone(), r["window"].clone()
    out = torch.full((B, T, H, 128), float("nan"), device=DEV, dtype=r["q_raw"].dtype)
    kda.kda_layer_replay(state, win, r["q_raw"], r["k_raw"], r["v_raw"], r["a_logit"],
                         r["b_logit"], r["g"], r["conv_w"], r["gamma"],
                         torch.as_tensor(n, device=DEV), out=out)
    torch.cuda.synchronize()
    _check_replay(r, n, out, state, win, T, TOL[dtype])


def test_layer_replay_each_cta_walks_units_across_skipped_runs():
    """More units than the persistent grid (two CTAs per SM), so every CTA walks
    several units, with a run of sequences that accept nothing longer than two
    grid strides and the last units empty.  Every unit against the oracle;
    skipped units keep their state and window."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H, T = 1, 3
    B = 8 * sms + 37
    g = np.random.default_rng(43)
    n = g.integers(1, T + 1, size=B).astype(np.int32)
    n[50:50 + 6 * sms] = 0
    n[-5:] = 0
    n[[7, 7 + 2 * sms]] = -3                                # clamped to 0
    n[[9, 9 + 2 * sms]] = T + 5                             # clamped to T
    r = replay_layer_inputs(B, T, H, "f32", seed=43)
    state, win = r["state"].clone(), r["window"].clone()
    out = torch.full((B, T, H, 128), float("nan"), device=DEV, dtype=r["q_raw"].dtype)
    kda.kda_layer_replay(state, win, r["q_raw"], r["k_raw"], r["v_raw"], r["a_logit"],
                         r["b_logit"], r["g"], r["conv_w"], r["gamma"],
                         torch.as_tensor(n, device=DEV), out=out)
    torch.cuda.synchronize()
    _check_replay(r, n, out, state, win, T, TOL["f32"])


def test_layer_replay_equals_the_unfused_gpu_chain():
    """prep with the window, the decode replay, then post (three kernels, with
    bf16 rounding between them) against the fused kernel: each is within the
    bf16 tolerance of the exact result (the fused one is checked against the
    oracle above), so they are within twice that of each other; the window is
    the same bit for bit."""
    B, T, H = 4, 5, 2
    r = replay_layer_inputs(B, T, H, "bf16", seed=61)
    n = np.array([5, 3, 1, 4], dtype=np.int32)
    s1, w1 = r["state"].clone(), r["window"].clone()
    fused = kda.kda_layer_replay(s1, w1, r["q_raw"], r["k_raw"], r["v_raw"], r["a_logit"],
                                 r["b_logit"], r["g"], r["conv_w"], r["gamma"],
                                 torch.as_tensor(n, device=DEV))
    s2, w2 = r["state"].clone(), r["window"].clone()
    for b in range(B):
        nb = int(n[b])
        y = {x: r[x][b, :nb].contiguous() for x in ("q_raw", "k_raw", "v_raw", "a_logit", "b_logit")}
        y["conv_w"] = r["conv_w"]
        cu = torch.tensor([0, nb], dtype=torch.int32, device=DEV)
        wb = w2[b:b + 1].clone()
        q, k, v, la, be = _prep_state(y, cu, wb, wb)
        w2[b] = wb[0]
        st = s2[b:b + 1]
        o = kda.kda_decode_replay(st, q[None], k[None], v[None], la[None], be[None],
                                  torch.tensor([nb], dtype=torch.int32, device=DEV))
        s2[b] = st[0]
        post = kda.kda_post_fwd(o[0], r["g"][b, :nb].contiguous(), r["gamma"])
        assert_parity(fused[b, :nb], post, 2 * TOL["bf16"], name=f"output of sequence {b}")
    torch.cuda.synchronize()
    assert_parity(s1, s2, 2 * TOL["bf16"], name="state")
    assert torch.equal(w1, w2)


def test_layer_replay_full_size_sampled_units():
    """512 sequences x 96 heads x 4 drafts (the benchmark's configuration),
    seeded accepted counts; 32 sampled units replayed by the oracle."""
    B, T, H = 512, 4, 96
    r = replay_layer_inputs(B, T, H, "bf16", seed=63)
    g = np.random.default_rng(63)
    n = g.integers(0, T + 1, size=B).astype(np.int32)
    state, win = r["state"].clone(), r["window"].clone()
    out = kda.kda_layer_replay(state, win, r["q_raw"], r["k_raw"], r["v_raw"], r["a_logit"],
                               r["b_logit"], r["g"], r["conv_w"], r["gamma"],
                               torch.as_tensor(n, device=DEV))
    torch.cuda.synchronize()
    got_o, ref_o, got_s, ref_s, lens = [], [], [], [], []
    for u in np.sort(g.choice(B * H, size=32, replace=False)):
        b, h = divmod(int(u), H)
        nb = int(n[b])
        sub = {x: r[x][b:b + 1, :, h:h + 1] for x in ("q_raw", "k_raw", "v_raw", "a_logit",
                                                       "b_logit", "g")}
        st = _np(r["state"][b:b + 1, h:h + 1]).copy()
        wn = _np(r["window"][b:b + 1, :, :, h:h + 1]).copy()
        ro = L.layer_replay(st, wn, *(_np(sub[x]) for x in ("q_raw", "k_raw", "v_raw", "a_logit",
                                                             "b_logit", "g")),
                            _np(r["conv_w"][:, h:h + 1]), _np(r["gamma"]), [nb], oracle.decode_step)
        if nb:
            got_o.append(_np(out[b, :nb, h]))
            ref_o.append(ro[0, :nb, 0])
            got_s.append(_np(state[b, h]))
            ref_s.append(st[0, 0])
            lens.append(nb)
        assert torch.equal(win[b, :, :, h], torch.as_tensor(wn[0, :, :, 0]).to(DEV, win.dtype))
    cu = np.concatenate([[0], np.cumsum(lens)])
    assert_parity(np.concatenate(got_o)[:, None], np.concatenate(ref_o)[:, None], TOL["bf16"],
                  cu=cu, name="layer output")
    assert_parity(np.stack(got_s)[:, None], np.stack(ref_s)[:, None], TOL["bf16"], name="state")
