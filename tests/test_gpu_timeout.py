"""The bounded-wait path of the bf16 prefill, exercised without faulting or
hanging anything: the workspace's test control makes one chain's CTA wait at
most 1 ms and withholds one warp's arrival on the barrier that releases a
chunk's Gram products.  That CTA's wait gives up, records KDA_ERR_TIMEOUT with
its chain and chunk, drains its copies and MMAs, frees its tensor memory and
returns; every other chain is unaffected, and the next ordinary call on the
same workspace is KDA_OK with oracle parity."""
from __future__ import annotations

import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, check_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H = 3
LENGTHS = [512, 300]        # 8 and 5 chunks


def _call(x, ws):
    # the plain schedule: the control acts only there
    return kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                             x["cu_seqlens"], workspace=ws, max_split=0, max_helpers=0)


@pytest.mark.parametrize("seq,head,chunk", [(1, 1, 2), (0, 2, 0), (1, 0, 4)])
def test_withheld_arrival_times_out_and_reports(seq, head, chunk):
    x = inputs.prefill_inputs(LENGTHS, H=H, dtype="bf16", init_state=True, device=DEV, seed=81)
    ws = torch.zeros(kda.kda_chunk_fwd_workspace_size(2, sum(LENGTHS), H), dtype=torch.uint8,
                     device=DEV)
    chain = seq * H + head
    kda.kda_test_arm_timeout(ws, chain, chunk, wait_us=1000)
    out, fin = _call(x, ws)
    torch.cuda.synchronize()
    code, detail, got_chain, got_chunk = kda.kda_read_device_status_detail(ws)
    assert code == kda.KDA_ERR_TIMEOUT, kda.status_string(code)
    assert (got_chain, got_chunk) == (chain, chunk), (detail, got_chain, got_chunk)
    # the other chains of both sequences ran to completion, correctly
    for s in range(2):
        heads = [h for h in range(H) if (s, h) != (seq, head)]
        check_prefill(x, out, fin, TOL["bf16"], heads=heads, seqs=[s])
    # the control was consumed; the next call on the same workspace is clean
    out2, fin2 = _call(x, ws)
    torch.cuda.synchronize()
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    check_prefill(x, out2, fin2, TOL["bf16"])


def test_disarmed_control_changes_nothing():
    x = inputs.prefill_inputs(LENGTHS, H=H, dtype="bf16", init_state=True, device=DEV, seed=82)
    ws = torch.zeros(kda.kda_chunk_fwd_workspace_size(2, sum(LENGTHS), H), dtype=torch.uint8,
                     device=DEV)
    o0, s0 = _call(x, ws)
    o0, s0 = o0.clone(), s0.clone()
    kda.kda_test_arm_timeout(ws, 1, 1, wait_us=1000)
    kda.kda_test_arm_timeout(ws, -1, 0)               # disarm
    o1, s1 = _call(x, ws)
    torch.cuda.synchronize()
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    assert torch.equal(o0, o1) and torch.equal(s0, s1)
