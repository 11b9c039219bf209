"""Parity at the workloads' full sizes, in the launch configuration bench.py
times: every output and final state of the B=4, H=16, T=4096 workload, and a
head (and sequence) sample of the K3-layout and million-token varlen workloads,
each compared with the fp64 oracle run on exactly the sampled chains."""
from __future__ import annotations

import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, oracle_prefill, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run_and_compare(x, heads=None, seqs=None):
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                 x["init_state"], x["cu_seqlens"])
    torch.cuda.synchronize()
    o_ref, s_ref, idx = oracle_prefill(x, heads=heads, seqs=seqs)
    H = x["q"].shape[1]
    hsel = torch.as_tensor(heads if heads is not None else list(range(H)), device=DEV)
    n_seqs = x["cu_seqlens"].shape[0] - 1
    ssel = torch.as_tensor(seqs if seqs is not None else list(range(n_seqs)), device=DEV)
    got_o = out.index_select(0, torch.as_tensor(idx, device=DEV)).index_select(1, hsel)
    got_s = fin.index_select(0, ssel).index_select(1, hsel)
    eo, es = rel_l2(got_o, o_ref), rel_l2(got_s, s_ref)
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    return eo, es


def test_b4_h16_t4096_full():
    x = inputs.workload_inputs("b4_h16_t4096", device=DEV)
    eo, es = _run_and_compare(x)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)


def test_k3_h96_t32768_head_sample():
    x = inputs.workload_inputs("k3_h96_t32768", device=DEV)
    eo, es = _run_and_compare(x, heads=[0, 31, 63, 95])
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)


def test_varlen_h96_1m_sample():
    """8 packed sequences of 1k-262k tokens (about 1M tokens), per-sequence
    initial and final states; heads 0 and 95 of every sequence checked."""
    x = inputs.workload_inputs("varlen_h96_1m", device=DEV)
    eo, es = _run_and_compare(x, heads=[0, 95])
    del x
    torch.cuda.empty_cache()
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)
