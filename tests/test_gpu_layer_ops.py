"""GPU parity of kda_prep_fwd / kda_post_fwd (the per-token steps around the
recurrence) against the fp64 oracle, alone and chained with kda_chunk_fwd."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import layer_ops as L
from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, assert_parity, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GATE_TOL = 1e-5   # fp32 gates (sigmoid through expf) in both dtypes


def _np(t):
    return t.double().cpu().numpy()


PREP_CASES = [
    # sequences shorter than the convolution window, an empty one, ragged longer ones
    ([0, 1, 3, 4, 37, 130], 3),
    # many tiny and empty sequences inside one run of tokens; H not a multiple of 8
    ([1, 0, 0, 2, 1, 5, 0, 3, 33, 1, 2, 0, 70], 9),
    # sequence starts just before, at and after the boundaries of 128-token runs,
    # and one sequence across several runs
    ([127, 1, 129, 0, 2, 300], 3),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("lengths,H", PREP_CASES)
def test_prep_matches_oracle(dtype, lengths, H):
    x = inputs.layer_inputs(lengths, H=H, dtype=dtype, device=DEV, seed=21)
    q, k, v, la, beta = kda.kda_prep_fwd(x["q_raw"], x["k_raw"], x["v_raw"], x["conv_w"],
                                         x["a_logit"], x["b_logit"], x["cu_seqlens"])
    torch.cuda.synchronize()
    ref = L.prep(_np(x["q_raw"]), _np(x["k_raw"]), _np(x["v_raw"]), _np(x["conv_w"]),
                 _np(x["a_logit"]), _np(x["b_logit"]), _np(x["cu_seqlens"]).astype(np.int64))
    cu = _np(x["cu_seqlens"]).astype(np.int64)
    for name, got, want in zip("qkv", (q, k, v), ref[:3]):
        assert_parity(got, want, TOL[dtype], cu=cu, name=name)
    assert_parity(la, ref[3], GATE_TOL, cu=cu, name="log_alpha")
    assert_parity(beta[..., None], ref[4][..., None], GATE_TOL, cu=cu, name="beta")
    norms = q.float().norm(dim=-1)
    assert torch.allclose(norms, torch.ones_like(norms), atol=2e-2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_post_matches_oracle_and_runs_in_place(dtype):
    x = inputs.layer_inputs([50, 77], H=4, dtype=dtype, device=DEV, seed=22)
    o = x["v_raw"]
    out = kda.kda_post_fwd(o, x["g"], x["gamma"])
    torch.cuda.synchronize()
    ref = L.post(_np(o), _np(x["g"]), _np(x["gamma"]))
    assert_parity(out, ref, TOL[dtype], cu=_np(x["cu_seqlens"]).astype(np.int64), name="post")
    o2 = o.clone()
    kda.kda_post_fwd(o2, x["g"], x["gamma"], out=o2)
    torch.cuda.synchronize()
    assert torch.equal(o2, out)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_layer_chain_matches_oracle(dtype):
    """prep -> chunked recurrence -> post against the oracle's own chain."""
    lengths = [70, 3, 129]
    H = 2
    x = inputs.layer_inputs(lengths, H=H, dtype=dtype, device=DEV, seed=23)
    q, k, v, la, beta = kda.kda_prep_fwd(x["q_raw"], x["k_raw"], x["v_raw"], x["conv_w"],
                                         x["a_logit"], x["b_logit"], x["cu_seqlens"])
    o, fin = kda.kda_chunk_fwd(q, k, v, la, beta, None, x["cu_seqlens"])
    y = kda.kda_post_fwd(o, x["g"], x["gamma"])
    torch.cuda.synchronize()
    cu = _np(x["cu_seqlens"]).astype(np.int64)
    rq, rk, rv, rla, rb = L.prep(_np(x["q_raw"]), _np(x["k_raw"]), _np(x["v_raw"]),
                                 _np(x["conv_w"]), _np(x["a_logit"]), _np(x["b_logit"]), cu)
    ro, rfin = oracle.chunk_fwd(rq, rk, rv, rla, rb, None, cu)
    ry = L.post(ro, _np(x["g"]), _np(x["gamma"]))
    assert_parity(y, ry, TOL[dtype], cu=cu, name="layer output")
    assert_parity(fin, rfin, TOL[dtype], name="final state")


def test_prep_and_post_full_size_sampled_rows():
    """The benchmark's shape (one sequence of 32768 tokens, 96 heads, bf16): 64
    sampled (token, head) rows of every output against the oracle row by row
    (a row's convolution needs only the three tokens before it)."""
    T, H = 32768, 96
    x = inputs.layer_inputs([T], H=H, dtype="bf16", device=DEV, seed=24)
    q, k, v, la, beta = kda.kda_prep_fwd(x["q_raw"], x["k_raw"], x["v_raw"], x["conv_w"],
                                         x["a_logit"], x["b_logit"], x["cu_seqlens"])
    y = kda.kda_post_fwd(v, x["g"], x["gamma"])
    torch.cuda.synchronize()
    g = np.random.default_rng(24)
    for t, h in zip(g.integers(0, T, 64), g.integers(0, H, 64)):
        t, h = int(t), int(h)
        a = max(0, t - 3)
        sl = slice(a, t + 1)
        win = {n: _np(x[n][sl, h:h + 1]) for n in ("q_raw", "k_raw", "v_raw", "a_logit")}
        rq, rk, rv, rla, rb = L.prep(win["q_raw"], win["k_raw"], win["v_raw"],
                                     _np(x["conv_w"][:, h:h + 1]), win["a_logit"],
                                     _np(x["b_logit"][sl, h:h + 1]), [0, t + 1 - a])
        assert rel_l2(q[t, h], rq[-1, 0]) <= TOL["bf16"]
        assert rel_l2(k[t, h], rk[-1, 0]) <= TOL["bf16"]
        assert rel_l2(v[t, h], rv[-1, 0]) <= TOL["bf16"]
        assert rel_l2(la[t, h], rla[-1, 0]) <= GATE_TOL
        assert abs(float(beta[t, h]) - float(rb[-1, 0])) <= 1e-6
        ry = L.post(_np(v[t:t + 1, h:h + 1]), _np(x["g"][t:t + 1, h:h + 1]), _np(x["gamma"]))
        assert rel_l2(y[t, h], ry[0, 0]) <= TOL["bf16"]
