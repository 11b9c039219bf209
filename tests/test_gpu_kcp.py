"""The KCP building blocks on the GPU: each segment's affine pair
(kda_chunk_fwd_transitions) and their composition (kda_state_combine) against
the oracle, and a three-rank context-parallel prefill emulated on one GPU (the
ranks' steps run in turn; the exchange is a list) against the oracle over the
whole sequences."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_13_gb300 import inputs, kda
from gated_delta_rule_13_gb300.kcp import KernelOps, stack_pairs, start_state
from kcp_util import OracleOps, rank_segments
from parity_util import TOL, assert_parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(lengths, H, seed, decay):
    x = inputs.prefill_inputs(lengths, H=H, dtype="bf16", init_state=True, device=DEV, seed=seed)
    x["log_alpha"].mul_(decay)
    return x


@pytest.mark.parametrize("decay", [0.0, 0.02])
def test_transitions_match_oracle_pairs(decay):
    x = _inputs([700, 0, 130], H=3, seed=61, decay=decay)
    b, m = kda.kda_chunk_fwd_transitions(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                         x["cu_seqlens"])
    torch.cuda.synchronize()
    rb, rm = OracleOps.pairs(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"])
    assert_parity(b, rb, TOL["bf16"], name="B")
    assert_parity(m, rm, TOL["bf16"], name="M")
    # an empty sequence maps every state to itself
    assert torch.equal(b[1], torch.zeros_like(b[1]))
    assert torch.equal(m[1], torch.eye(128, device=DEV).expand(3, 128, 128))


def test_state_combine_matches_numpy():
    g = torch.Generator(device=DEV).manual_seed(62)
    n_seqs, K, H = 2, 5, 3
    b = 0.1 * torch.randn(n_seqs * K, H, 128, 128, device=DEV, generator=g)
    m = torch.randn(n_seqs * K, H, 128, 128, device=DEV, generator=g) / 128 ** 0.5
    init = torch.randn(n_seqs, H, 128, 128, device=DEV, generator=g)
    for s0 in (init, None):
        starts, end = kda.kda_state_combine(b, m, K, s0)
        torch.cuda.synchronize()
        rs, re = OracleOps.combine(b, m, K, s0)
        assert_parity(starts, rs, 1e-5, name="start states")
        assert_parity(end, re, 1e-5, name="end states")


@pytest.mark.parametrize("decay", [0.0, 0.02, 1.0])
def test_three_rank_kcp_matches_oracle(decay):
    world = 3
    x = _inputs([5000, 2500, 90], H=4, seed=63, decay=decay)
    locs = [rank_segments(x, world, r) for r in range(world)]
    pairs = [KernelOps.pairs(l["q"], l["k"], l["v"], l["log_alpha"], l["beta"], l["cu_seqlens"])
             for l, _ in locs]
    state_b, state_m = stack_pairs(pairs)
    out = torch.empty_like(x["v"])
    end = None
    for r, (l, idx) in enumerate(locs):
        start, end_r = start_state(state_b, state_m, r, world, x["init_state"])
        o = KernelOps.forward(l["q"], l["k"], l["v"], l["log_alpha"], l["beta"], start,
                              l["cu_seqlens"])
        out.index_copy_(0, idx, o)
        if end is not None:
            assert torch.equal(end, end_r)  # every rank composes the same final states
        end = end_r
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                    x["init_state"], x["cu_seqlens"])
    assert_parity(out, o_ref, TOL["bf16"], cu=x["cu_seqlens"].cpu().numpy(), name="out")
    assert_parity(end, s_ref, TOL["bf16"], name="final state")
