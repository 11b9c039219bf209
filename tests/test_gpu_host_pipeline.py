"""kda_chunk_fwd_host: one sequence from host memory in token pieces, the copies
overlapping the prefill, each piece starting from the previous piece's final
state.  It must give exactly the results of one kda_chunk_fwd call."""
from __future__ import annotations

import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("N,piece,init", [(1000, 256, True), (4096, 4096, False),
                                          (5000, 1024, True), (64, 64, False)])
def test_pieces_equal_one_call(N, piece, init):
    """Bitwise: the pieces and the whole call run the plain schedule (few heads
    would otherwise take the in-device split for long calls only)."""
    x = inputs.prefill_inputs([N], H=3, dtype="bf16", init_state=init, device=DEV, seed=71)
    o_ref, s_ref = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                     x["init_state"], x["cu_seqlens"], max_split=0,
                                     max_helpers=0)
    host = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "log_alpha", "beta")}
    h_init = x["init_state"].cpu() if init else None
    out, fin = kda.kda_chunk_fwd_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                      host["beta"], h_init, piece_tokens=piece, device=DEV,
                                      max_split=0, max_helpers=0)
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref.cpu()) and torch.equal(fin, s_ref.cpu())


def test_default_schedules_match_oracle():
    """With the split allowed (long pieces over few heads take it), against the oracle."""
    import oracle
    from parity_util import TOL, assert_parity
    x = inputs.prefill_inputs([9000], H=2, dtype="bf16", init_state=True, device=DEV, seed=73)
    host = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "log_alpha", "beta")}
    out, fin = kda.kda_chunk_fwd_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                      host["beta"], x["init_state"].cpu(), piece_tokens=4096,
                                      device=DEV)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                    x["init_state"], x["cu_seqlens"])
    assert_parity(out, o_ref, TOL["bf16"], name="out")
    assert_parity(fin, s_ref, TOL["bf16"], name="final state")


def test_empty_sequence_and_bad_piece():
    x = inputs.prefill_inputs([64], H=2, dtype="bf16", init_state=True, device=DEV, seed=72)
    z = {n: x[n][:0].cpu() for n in ("q", "k", "v", "log_alpha", "beta")}
    out, fin = kda.kda_chunk_fwd_host(z["q"], z["k"], z["v"], z["log_alpha"], z["beta"],
                                      x["init_state"].cpu(), device=DEV)
    assert out.shape[0] == 0 and torch.equal(fin, x["init_state"].cpu())
    with pytest.raises(ValueError):
        kda.kda_chunk_fwd_host(z["q"], z["k"], z["v"], z["log_alpha"], z["beta"],
                               piece_tokens=100, device=DEV)
