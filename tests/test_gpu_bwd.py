"""GPU parity of the backward pass (kda_chunk_bwd) against the fp64 gradient
oracle (oracle/kda_oracle_bwd.c, itself pinned by finite differences of the
forward oracle): every gradient, whole tensor, every (sequence, head) slice and
every row."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, assert_parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _grads_in(x, seed, d_final=True):
    g = torch.Generator(device=DEV).manual_seed(seed)
    N, H, _ = x["q"].shape
    do = torch.randn(N, H, 128, generator=g, device=DEV).to(x["q"].dtype)
    n_seqs = x["cu_seqlens"].shape[0] - 1
    df = torch.randn(n_seqs, H, 128, 128, generator=g, device=DEV) if d_final else None
    return do, df


def _check(x, do, df, dtype, heads=None, every=None):
    got = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                            x["cu_seqlens"], do, df, ckpt_every=every)
    torch.cuda.synchronize()
    hs = list(range(x["q"].shape[1])) if heads is None else heads
    hsel = torch.as_tensor(hs, device=DEV)

    def sub(t):
        return t.detach().index_select(1, hsel).cpu() if t is not None else None

    ref = oracle.chunk_bwd(sub(x["q"]), sub(x["k"]), sub(x["v"]), sub(x["log_alpha"]),
                           sub(x["beta"]), sub(x["init_state"]), x["cu_seqlens"].cpu(), sub(do),
                           sub(df))
    cu = x["cu_seqlens"].cpu().numpy()
    tol = TOL[dtype]
    for name, gt, rf in zip(("dq", "dk", "dv", "d_log_alpha"), got[:4], ref[:4]):
        assert_parity(sub(gt), rf, tol, cu=cu, name=name)
    assert_parity(sub(got[4])[..., None], ref[4][..., None], tol, cu=cu, name="d_beta")
    assert_parity(sub(got[5]), ref[5], tol, name="d_init_state")
    return got


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("init,final", [(True, True), (False, True), (True, False)])
def test_bwd_matches_oracle_ragged(dtype, init, final):
    lengths = [0, 1, 15, 16, 17, 33, 64, 100]
    x = inputs.prefill_inputs(lengths, H=2, dtype=dtype, init_state=init, device=DEV, seed=91)
    do, df = _grads_in(x, 92, d_final=final)
    _check(x, do, df, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", ["la0", "la_floor", "beta1"])
def test_bwd_edge_values(case, dtype):
    """No decay, the decay floor (log alpha = -5 on every channel: a 16-token
    chunk spans e^-80, the chunked pass's factors e^+-40 around its middle row)
    and beta = 1."""
    x = inputs.prefill_inputs([70, 45], H=2, dtype=dtype, init_state=True, device=DEV, seed=93)
    if case == "la0":
        x["log_alpha"].zero_()
    elif case == "la_floor":
        x["log_alpha"].fill_(-5.0)
    else:
        x["beta"].fill_(1.0)
    do, df = _grads_in(x, 94)
    _check(x, do, df, dtype)


def test_bwd_bf16_token_loop_pass():
    """An explicit checkpoint interval selects the token-loop pass for bf16
    too: the same oracle parity on ragged lengths."""
    lengths = [0, 1, 15, 16, 17, 33, 64, 100]
    x = inputs.prefill_inputs(lengths, H=2, dtype="bf16", init_state=True, device=DEV, seed=97)
    do, df = _grads_in(x, 98)
    _check(x, do, df, "bf16", every=8)


@pytest.mark.parametrize("every", [None, 4])
def test_bwd_host_cu_seqlens_and_deterministic_dv(every):
    """A host cu_seqlens gives the results of a device one.  The chunked pass
    (bf16 default) writes every gradient element once: all of them bitwise
    repeatable.  The token-loop pass: dv and the initial-state gradient (one
    column block each, no atomics) bitwise, the atomically summed ones to their
    last bits."""
    x = inputs.prefill_inputs([40, 90], H=3, dtype="bf16", init_state=True, device=DEV, seed=95)
    do, df = _grads_in(x, 96)
    a = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                          x["cu_seqlens"], do, df, ckpt_every=every)
    b = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                          x["cu_seqlens"].cpu(), do, df, ckpt_every=every)
    torch.cuda.synchronize()
    assert torch.equal(a[2], b[2]) and torch.equal(a[5], b[5])
    for i in (0, 1, 3, 4):
        if every is None:
            assert torch.equal(a[i], b[i]), i
        assert_parity(a[i] if i != 4 else a[i][..., None], b[i] if i != 4 else b[i][..., None],
                      1e-5, cu=x["cu_seqlens"].cpu().numpy(), name=f"gradient {i}")


def test_bwd_two_calls_chain_through_the_state():
    """Backward of two calls with the state handed over equals the backward of
    one call: the second call's initial-state gradient is the first call's
    final-state gradient."""
    T, cut = 300, 129
    x = inputs.prefill_inputs([T], H=2, dtype="f32", init_state=True, device=DEV, seed=97)
    do, df = _grads_in(x, 98)
    whole = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                              x["init_state"], x["cu_seqlens"], do, df)
    first = {n: x[n][:cut].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    second = {n: x[n][cut:].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    _, mid = kda.kda_chunk_fwd(first["q"], first["k"], first["v"], first["log_alpha"],
                               first["beta"], x["init_state"])
    g2 = kda.kda_chunk_bwd(second["q"], second["k"], second["v"], second["log_alpha"],
                           second["beta"], mid, None, do[cut:].contiguous(), df)
    g1 = kda.kda_chunk_bwd(first["q"], first["k"], first["v"], first["log_alpha"],
                           first["beta"], x["init_state"], None, do[:cut].contiguous(), g2[5])
    torch.cuda.synchronize()
    for i, name in enumerate(("dq", "dk", "dv", "d_log_alpha")):
        assert_parity(torch.cat([g1[i], g2[i]]), whole[i], 1e-4, name=name)
    assert_parity(g1[5], whole[5], 1e-4, name="d_init_state")


def test_bwd_one_cta_per_chain():
    """With more chains than half the SMs the chunked pass takes one CTA per
    chain (with fewer, a two-CTA cluster splits each chain's value columns):
    80 chains of ragged lengths, 6 heads against the oracle."""
    lengths = [0, 1, 37, 16, 130]
    x = inputs.prefill_inputs(lengths, H=20, dtype="bf16", init_state=True, device=DEV, seed=103)
    do, df = _grads_in(x, 104)
    assert len(lengths) * 20 * 2 > torch.cuda.get_device_properties(0).multi_processor_count
    _check(x, do, df, "bf16", heads=[0, 3, 7, 11, 16, 19])


@pytest.mark.parametrize("every,H", [(None, 2), (None, 80), (4, 2)])
def test_bwd_invalid_device_cu_seqlens_reports_status(every, H):
    """A malformed device cu_seqlens: every kernel of the pass (a two-CTA
    cluster per chain, one CTA per chain, the token loop) records
    KDA_ERR_INVALID_ARG in the workspace (both CTAs of a cluster leave before
    their first cluster barrier); the same workspace then serves a valid call,
    which reports OK."""
    x = inputs.prefill_inputs([100, 50], H=H, dtype="bf16", init_state=True, device=DEV, seed=8)
    do, df = _grads_in(x, 9)
    ws = torch.zeros(kda.kda_chunk_bwd_workspace_size(2, 150, H, ckpt_every=every or 0),
                     dtype=torch.uint8, device=DEV)
    bad = torch.tensor([0, 120, 110], dtype=torch.int32, device=DEV)
    kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"], bad, do,
                      df, workspace=ws, ckpt_every=every)
    assert kda.kda_read_device_status(ws) == kda.KDA_ERR_INVALID_ARG
    kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                      x["cu_seqlens"], do, df, workspace=ws, ckpt_every=every)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK


def test_bwd_b4_h16_t4096_sampled_heads():
    """The B=4, H=16, T=4096 prefill workload (random initial states): heads 0
    and 15 of every sequence against the oracle."""
    x = inputs.workload_inputs("b4_h16_t4096", device=DEV)
    do, df = _grads_in(x, 99)
    _check(x, do, df, "bf16", heads=[0, 15])


def test_bwd_checkpoint_interval_changes_nothing():
    """Every checkpoint interval gives the default's gradients: the states
    replayed from a stored one are the forward sweep's own, so dv and the
    initial-state gradient (no atomics) are bitwise equal and the atomically
    summed ones equal to their last bits.  Sequences shorter and longer than
    the intervals, one of them empty, cover the recomputation of whole and
    partial groups."""
    lengths = [0, 3, 16, 47, 130, 300]
    x = inputs.prefill_inputs(lengths, H=2, dtype="f32", init_state=True, device=DEV, seed=101)
    do, df = _grads_in(x, 102)
    base = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                             x["cu_seqlens"], do, df)
    cu = x["cu_seqlens"].cpu().numpy()
    for every in (4, 8, 16, 64, 1024):
        g = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                              x["cu_seqlens"], do, df, ckpt_every=every)
        torch.cuda.synchronize()
        assert torch.equal(g[2], base[2]) and torch.equal(g[5], base[5]), every
        for i in (0, 1, 3):
            assert_parity(g[i], base[i], 1e-5, cu=cu, name=f"gradient {i}, every {every}")
        assert_parity(g[4][..., None], base[4][..., None], 1e-5, cu=cu, name=f"d_beta, every {every}")
