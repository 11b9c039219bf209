"""Helper CTAs of the bf16 prefill: when a call has fewer chains than the GPU
has SMs, the idle SMs precompute the state-independent half of later chunks and
the chain CTAs use those packages instead of computing them.  The results must
be bitwise those of a run without helpers (same arithmetic, same order), and
still match the oracle."""
from __future__ import annotations

import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, check_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(x, helpers):
    """kda_chunk_fwd with the split off (these calls are small enough for it,
    and it takes precedence over helpers) and helpers on (the library's count)
    or off; returns the outputs and the helper counters of the call."""
    n_seqs = x["cu_seqlens"].shape[0] - 1
    N, H = x["q"].shape[0], x["q"].shape[1]
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(n_seqs, N, H, dtype=kda.KDA_BF16),
                     dtype=torch.uint8, device=DEV)
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                 x["init_state"], x["cu_seqlens"], workspace=ws, max_split=0,
                                 max_helpers=None if helpers else 0)
    stats = kda.kda_read_chunk_stats(ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    return out.clone(), fin.clone(), stats


def _sampled_parity(x, out, fin, heads):
    check_prefill(x, out, fin, TOL["bf16"], heads=heads)


def test_long_chains_use_packages_bitwise():
    """8 chains of 128 chunks: helpers publish packages and the chains use some;
    outputs and final states equal the helper-free run bit for bit."""
    x = inputs.prefill_inputs([8192], H=8, dtype="bf16", init_state=True, device=DEV, seed=31)
    o0, s0, st0 = _run(x, helpers=False)
    o1, s1, st1 = _run(x, helpers=True)
    assert st0 == (0, 0)
    published, consumed = st1
    assert published > 0 and 0 < consumed <= published
    assert torch.equal(o0, o1) and torch.equal(s0, s1)
    _sampled_parity(x, o1, s1, heads=[0, 7])


def test_mixed_lengths_bitwise_and_oracle():
    """Short, empty and long sequences with ragged last chunks: chains that end
    early, chains helpers can help and packages of partial chunks."""
    lengths = [3000, 1, 0, 65, 2111, 640]
    x = inputs.prefill_inputs(lengths, H=3, dtype="bf16", init_state=True, device=DEV, seed=32)
    o0, s0, _ = _run(x, helpers=False)
    o1, s1, st1 = _run(x, helpers=True)
    assert torch.equal(o0, o1) and torch.equal(s0, s1)
    assert st1[1] <= st1[0]
    _sampled_parity(x, o1, s1, heads=[0, 1, 2])


def test_repeated_calls_same_workspace():
    """The helper header is reset per call: back-to-back calls on one workspace
    give identical results and consistent counters."""
    x = inputs.prefill_inputs([4096, 4096], H=4, dtype="bf16", device=DEV, seed=33)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(2, 8192, 4, dtype=kda.KDA_BF16),
                     dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(3):
        out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None,
                                     x["cu_seqlens"], workspace=ws, max_split=0)
        pub, con = kda.kda_read_chunk_stats(ws)
        assert 0 <= con <= pub
        outs.append((out.clone(), fin.clone()))
    for o, s in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(s, outs[0][1])


def test_noalloc_runs_without_helpers_bitwise():
    """The no-workspace entry point has no room for the ring: same bits."""
    x = inputs.prefill_inputs([4096], H=6, dtype="bf16", init_state=True, device=DEV, seed=34)
    o1, s1, _ = _run(x, helpers=True)
    o2, s2 = kda.kda_chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                       x["init_state"], x["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
