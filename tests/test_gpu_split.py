"""In-device split of the bf16 prefill: with few chains, every sequence is cut
into K segments that run side by side (pass 1: each segment's B from a zero
state and its transition M from the identity with v = 0; combine
S_{j+1} = M_j S_j + B_j; pass 2: the outputs from the true start states).  The
results change rounding but must meet the oracle tolerance like the unsplit
path."""
from __future__ import annotations

import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, assert_parity, check_prefill, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(x, split=True, host_cu=False, final=True):
    """The library's schedule (the split, for these shapes), or the plain one;
    returns the outputs and the split's segment count."""
    n_seqs = x["cu_seqlens"].shape[0] - 1
    N, H = x["q"].shape[0], x["q"].shape[1]
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(n_seqs, N, H, dtype=kda.KDA_BF16),
                     dtype=torch.uint8, device=DEV)
    cu = x["cu_seqlens"].cpu() if host_cu else x["cu_seqlens"]
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                 x["init_state"], cu, workspace=ws, output_final_state=final,
                                 max_split=None if split else 0, max_helpers=0)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    return out.clone(), (fin.clone() if fin is not None else None)


def _parity(x, out, fin, heads=None):
    """Oracle parity on the chosen heads: whole tensor, every (sequence, head)
    slice and every row, which covers each segment's first tokens (where the
    output correction applies) and the ragged ends."""
    check_prefill(x, out, fin, TOL["bf16"], heads=heads)


def _close(o1, o0, s1, s0, x, tol):
    """Split against plain: within `tol` over the whole tensor, and within the
    bf16 tolerance for every (sequence, head) slice and row."""
    cu = x["cu_seqlens"].cpu().numpy()
    assert rel_l2(o1, o0) <= tol
    assert_parity(o1, o0, TOL["bf16"], cu=cu, name="out, split vs plain")
    if s1 is not None:
        assert rel_l2(s1, s0) <= tol
        assert_parity(s1, s0, TOL["bf16"], name="final state, split vs plain")


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
    o1, s1 = _run(x)
    o0, s0 = _run(x, split=False)
    assert not torch.equal(o1, o0)  # the split ran (its rounding differs)
    assert torch.equal(s0, s1)
    _close(o1, o0, None, None, x, 2e-3)
    _parity(x, o1, s1, heads=[3])


@pytest.mark.parametrize("scale", [0.0, 0.01])
def test_long_sequence_split_matches_oracle(scale):
    """One sequence of 16384 tokens over 8 heads (split 9 ways on a GB300) with
    an initial state, with no decay (scale 0: M_j is the whole product of the
    segment's (I - beta k k^T)) and with a decay 100 times weaker."""
    x = _slow_decay(inputs.prefill_inputs([16384], H=8, dtype="bf16", init_state=True,
                                          device=DEV, seed=41), scale)
    o1, s1 = _run(x)
    o0, s0 = _run(x, split=False)
    _parity(x, o1, s1, heads=[0, 5])
    # close to the unsplit result (both within the oracle tolerance)
    _close(o1, o0, s1, s0, x, 1e-2)


def test_several_sequences_with_short_and_empty_ones():
    """Sequences shorter than the split (empty segments), an empty sequence and
    ragged ends, each with its own initial state, no decay: every head against
    the oracle."""
    lengths = [5000, 70, 0, 3011]
    x = _slow_decay(inputs.prefill_inputs(lengths, H=2, dtype="bf16", init_state=True,
                                          device=DEV, seed=42), 0.0)
    o1, s1 = _run(x)
    _parity(x, o1, s1)
    # the empty sequence's final state is its initial state
    assert torch.equal(s1[2], x["init_state"][2])


def test_host_cu_seqlens_and_no_final_state():
    x = _slow_decay(inputs.prefill_inputs([6000, 4000], H=3, dtype="bf16", device=DEV, seed=43),
                    0.01)
    o1, s1 = _run(x, host_cu=True, final=False)
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
    o1, s1 = _run(x)
    o0, s0 = _run(x, split=False)
    assert not torch.equal(o1, o0)
    _parity(x, o1, s1, heads=[0, 9, 15])
    _close(o1, o0, s1, s0, x, 1e-2)


def test_zero_init_split_beyond_the_init_bound():
    """40 chains: 2 K - 1 = 3 blocks per chain fit the SMs, 2 K = 4 do not, so
    the call without an initial state is split in two and the one with an
    initial state is not (bitwise the plain path)."""
    sms = _sms()
    if not ((sms + 40) // 80 >= 2 and sms // 80 < 2):
        pytest.skip(f"{sms} SMs: not the case this test is about")
    x = _slow_decay(inputs.prefill_inputs([4096], H=40, dtype="bf16", device=DEV, seed=45), 0.01)
    o1, s1 = _run(x)
    o0, s0 = _run(x, split=False)
    assert not torch.equal(o1, o0)  # the split ran (its rounding differs)
    _parity(x, o1, s1)
    y = _slow_decay(inputs.prefill_inputs([4096], H=40, dtype="bf16", init_state=True,
                                          device=DEV, seed=45), 0.01)
    o2, s2 = _run(y)
    o3, s3 = _run(y, split=False)
    assert torch.equal(o2, o3) and torch.equal(s2, s3)
    _parity(y, o2, s2, heads=[0, 39])
