"""Parity at the workloads' full sizes, in the launch configuration bench.py
times: every output and final state of the B=4, H=16, T=4096 workload, and a
head (and sequence) sample of the K3-layout and million-token varlen workloads,
each compared with the fp64 oracle run on exactly the sampled chains (whole
tensor, every (sequence, head) slice and every row)."""
from __future__ import annotations

import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, check_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run_and_compare(x, heads=None, seqs=None):
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                 x["init_state"], x["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    return check_prefill(x, out, fin, TOL["bf16"], heads=heads, seqs=seqs)


def test_b4_h16_t4096_full():
    x = inputs.workload_inputs("b4_h16_t4096", device=DEV)
    _run_and_compare(x)


def test_k3_h96_t32768_head_sample():
    x = inputs.workload_inputs("k3_h96_t32768", device=DEV)
    _run_and_compare(x, heads=[0, 31, 63, 95])


def test_varlen_h96_1m_sample():
    """8 packed sequences of 1k-262k tokens (about 1M tokens), per-sequence
    initial and final states; heads 0 and 95 of every sequence checked."""
    x = inputs.workload_inputs("varlen_h96_1m", device=DEV)
    try:
        _run_and_compare(x, heads=[0, 95])
    finally:
        del x
        torch.cuda.empty_cache()
