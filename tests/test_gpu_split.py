"""In-device split of the bf16 prefill: with few chains, every sequence is cut
into K segments that run side by side (pass 1: each segment's B from a zero
state and its transition M from the identity with v = 0; combine
S_{j+1} = M_j S_j + B_j; pass 2: the outputs from the true start states).  The
results change rounding but must meet the oracle tolerance like the unsplit
path."""
from __future__ import annotations

import os

import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, oracle_prefill, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(x, split=True, host_cu=False, final=True):
    old = os.environ.get("KDA_CHUNK_SPLIT")
    try:
        if split:
            os.environ.pop("KDA_CHUNK_SPLIT", None)
        else:
            os.environ["KDA_CHUNK_SPLIT"] = "0"
        n_seqs = x["cu_seqlens"].shape[0] - 1
        N, H = x["q"].shape[0], x["q"].shape[1]
        ws = torch.empty(kda.kda_chunk_fwd_workspace_size(n_seqs, N, H, dtype=kda.KDA_BF16),
                         dtype=torch.uint8, device=DEV)
        cu = x["cu_seqlens"].cpu() if host_cu else x["cu_seqlens"]
        out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                     x["init_state"], cu, workspace=ws,
                                     output_final_state=final)
        assert kda.kda_read_device_status(ws) == kda.KDA_OK
        return out.clone(), (fin.clone() if fin is not None else None), ws.numel()
    finally:
        if old is None:
            os.environ.pop("KDA_CHUNK_SPLIT", None)
        else:
            os.environ["KDA_CHUNK_SPLIT"] = old


def _parity(x, out, fin, heads=None):
    o_ref, s_ref, idx = oracle_prefill(x, heads=heads)
    H = x["q"].shape[1]
    hsel = torch.as_tensor(heads if heads is not None else list(range(H)), device=DEV)
    got_o = out.index_select(0, torch.as_tensor(idx, device=DEV)).index_select(1, hsel)
    eo = rel_l2(got_o, o_ref)
    assert eo <= TOL["bf16"], eo
    if fin is not None:
        es = rel_l2(fin.index_select(1, hsel), s_ref)
        assert es <= TOL["bf16"], es
    return eo


def _slow_decay(x, scale):
    """With the workload's decay (log alpha = -5 sigmoid(N(0,1))) a chunk's
    total decay underflows to 0 in fp32, so states remember nothing older than
    a chunk and every M_j is exactly 0: the split is then bitwise the unsplit
    path.  Scaling log alpha down makes the segments' transitions matter."""
    x["log_alpha"].mul_(scale)
    return x


def test_workload_decay_split():
    """Under the workload's own decay (see _slow_decay) the final states are bit
    for bit the unsplit ones (every M_j is 0 and B_j the true state), and the
    outputs differ only where the correction is not zero yet: the first tokens
    of each segment, before their transition underflows."""
    x = inputs.prefill_inputs([16384], H=8, dtype="bf16", init_state=True, device=DEV, seed=41)
    o1, s1, ws_split = _run(x)
    o0, s0, ws_plain = _run(x, split=False)
    assert ws_split > ws_plain  # the split's scratch was provided
    assert torch.equal(s0, s1)
    assert rel_l2(o1, o0) <= 2e-3
    _parity(x, o1, s1, heads=[3])


@pytest.mark.parametrize("scale", [0.0, 0.01])
def test_long_sequence_split_matches_oracle(scale):
    """One sequence of 16384 tokens over 8 heads (split 9 ways on a GB300) with
    an initial state, with no decay (scale 0: M_j is the whole product of the
    segment's (I - beta k k^T)) and with a decay 100 times weaker."""
    x = _slow_decay(inputs.prefill_inputs([16384], H=8, dtype="bf16", init_state=True,
                                          device=DEV, seed=41), scale)
    o1, s1, _ = _run(x)
    o0, s0, _ = _run(x, split=False)
    _parity(x, o1, s1, heads=[0, 5])
    # close to the unsplit result (both within the oracle tolerance)
    assert rel_l2(o1, o0) <= 1e-2
    assert rel_l2(s1, s0) <= 1e-2


def test_several_sequences_with_short_and_empty_ones():
    """Sequences shorter than the split (empty segments), an empty sequence and
    ragged ends, each with its own initial state, no decay: every head against
    the oracle."""
    lengths = [5000, 70, 0, 3011]
    x = _slow_decay(inputs.prefill_inputs(lengths, H=2, dtype="bf16", init_state=True,
                                          device=DEV, seed=42), 0.0)
    o1, s1, _ = _run(x)
    _parity(x, o1, s1)
    # the empty sequence's final state is its initial state
    assert torch.equal(s1[2], x["init_state"][2])


def test_host_cu_seqlens_and_no_final_state():
    x = _slow_decay(inputs.prefill_inputs([6000, 4000], H=3, dtype="bf16", device=DEV, seed=43),
                    0.01)
    o1, s1, _ = _run(x, host_cu=True, final=False)
    assert s1 is None
    _parity(x, o1, None, heads=[1])


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("scale", [0.0, 0.01])
def test_zero_init_split_takes_more_segments(scale):
    """Without an initial state the first segment needs no transition run, so a
    sequence over 16 heads is cut into K = (SMs + 16) // 32 segments (5 on a
    GB300, one more than with an initial state): every M_j of a later segment
    and the combine from S_0 = 0 against the oracle."""
    x = _slow_decay(inputs.prefill_inputs([16384], H=16, dtype="bf16", device=DEV, seed=44),
                    scale)
    o1, s1, ws_split = _run(x)
    o0, s0, ws_plain = _run(x, split=False)
    assert ws_split > ws_plain
    _parity(x, o1, s1, heads=[0, 9, 15])
    assert rel_l2(o1, o0) <= 1e-2
    assert rel_l2(s1, s0) <= 1e-2


def test_zero_init_split_beyond_the_init_bound():
    """40 chains: 2 K - 1 = 3 blocks per chain fit the SMs, 2 K = 4 do not, so
    the call without an initial state is split in two and the one with an
    initial state is not (bitwise the plain path)."""
    sms = _sms()
    if not ((sms + 40) // 80 >= 2 and sms // 80 < 2):
        pytest.skip(f"{sms} SMs: not the case this test is about")
    x = _slow_decay(inputs.prefill_inputs([4096], H=40, dtype="bf16", device=DEV, seed=45), 0.01)
    o1, s1, ws_split = _run(x)
    o0, s0, ws_plain = _run(x, split=False)
    assert ws_split > ws_plain
    assert not torch.equal(o1, o0)  # the split ran (its rounding differs)
    _parity(x, o1, s1)
    y = _slow_decay(inputs.prefill_inputs([4096], H=40, dtype="bf16", init_state=True,
                                          device=DEV, seed=45), 0.01)
    o2, s2, _ = _run(y)
    o3, s3, _ = _run(y, split=False)
    assert torch.equal(o2, o3) and torch.equal(s2, s3)
    _parity(y, o2, s2, heads=[0, 39])
