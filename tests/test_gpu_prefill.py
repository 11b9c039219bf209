"""GPU parity of kda_chunk_fwd against the fp64 oracle, plus properties and
device-side error reporting.  fp32 inputs take the CUDA-core path (1e-4), bf16
inputs the tcgen05 tensor-core path (2e-2)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, assert_parity, check_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DTYPES = ["f32", "bf16"]


def run(x, **kw):
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                 x["init_state"], x["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return out, fin


def check(x, dtype, heads=None, seqs=None):
    """Whole-tensor, per-(sequence, head) and per-row parity with the oracle."""
    out, fin = run(x)
    return check_prefill(x, out, fin, TOL[dtype], heads=heads, seqs=seqs)


@pytest.mark.parametrize("dtype", DTYPES)
def test_tiny_workload(dtype):
    """B=1, H=1, T=512 (fp32 is the tiny workload itself)."""
    x = inputs.prefill_inputs([512], H=1, dtype=dtype, device=DEV)
    check(x, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("with_init", [False, True])
def test_ragged_lengths(dtype, with_init):
    lengths = [0, 1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200]
    x = inputs.prefill_inputs(lengths, H=3, dtype=dtype, init_state=with_init, device=DEV, seed=1)
    check(x, dtype)


@pytest.mark.parametrize("H", [2, 20, 40])
def test_f32_value_columns_split_over_ctas(H):
    """The fp32 path runs a chain on 4, 2 or 1 CTAs (32, 64 or 128 value columns
    each) by how many chains fit the SMs: 4, 40 and 80 chains here.  Every form
    against the oracle, with ragged last chunks and random initial states."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 4 * 4 <= sms and 2 * 40 <= sms < 4 * 40 and sms < 2 * 80
    x = inputs.prefill_inputs([37, 70], H=H, dtype="f32", init_state=True, device=DEV, seed=7)
    check(x, "f32", heads=None if H == 2 else [0, H // 2, H - 1])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("case", ["la0", "la_floor", "beta0", "beta1"])
def test_edge_values(dtype, case):
    x = inputs.prefill_inputs([300, 77], H=2, dtype=dtype, init_state=True, device=DEV, seed=2)
    if case == "la0":
        x["log_alpha"].zero_()
    elif case == "la_floor":
        x["log_alpha"].fill_(-5.0)          # worst case for the e^80 tile factors
    elif case == "beta0":
        # No writes: the state only decays.  Mild decay keeps the exact final
        # state (fp64) inside fp32 range, where a relative error means something.
        x["beta"].zero_()
        x["log_alpha"].mul_(0.01)
    else:
        x["beta"].fill_(1.0)
    check(x, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_init_state_is_read_only_and_zero_length(dtype):
    x = inputs.prefill_inputs([0, 70, 0], H=2, dtype=dtype, init_state=True, device=DEV, seed=3)
    s0 = x["init_state"].clone()
    out, fin = run(x)
    assert torch.equal(x["init_state"], s0)
    assert torch.equal(fin[0], s0[0]) and torch.equal(fin[2], s0[2])
    x["init_state"] = None
    _, fin0 = run(x)
    assert bool((fin0[0] == 0).all()) and bool((fin0[2] == 0).all())


@pytest.mark.parametrize("dtype", DTYPES)
def test_deterministic(dtype):
    x = inputs.prefill_inputs([257, 64], H=2, dtype=dtype, init_state=True, device=DEV, seed=4)
    o1, s1 = run(x)
    o1, s1 = o1.clone(), s1.clone()
    o2, s2 = run(x)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("dtype", DTYPES)
def test_split_with_state_handoff(dtype):
    """One call over T tokens equals two calls with the state handed over at a
    chunk-aligned cut (a prefix-cache resume) and at a ragged cut."""
    T = 1024
    x = inputs.prefill_inputs([T], H=2, dtype=dtype, init_state=True, device=DEV, seed=5)
    out, fin = run(x)
    for cut in (512, 389):
        a = {k: (v[:cut] if k in ("q", "k", "v", "log_alpha", "beta") else v)
             for k, v in x.items()}
        a["cu_seqlens"] = torch.tensor([0, cut], dtype=torch.int32, device=DEV)
        o1, s1 = run(a)
        b = {k: (v[cut:] if k in ("q", "k", "v", "log_alpha", "beta") else v)
             for k, v in x.items()}
        b["cu_seqlens"] = torch.tensor([0, T - cut], dtype=torch.int32, device=DEV)
        b["init_state"] = s1
        o2, s2 = run(b)
        tol = TOL[dtype]
        assert_parity(torch.cat([o1, o2]), out, tol, name=f"out, cut at {cut}")
        assert_parity(s2, fin, tol, name=f"final state, cut at {cut}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_steps_equal_prefill(dtype):
    T = 40
    x = inputs.prefill_inputs([T], H=2, dtype=dtype, init_state=True, device=DEV, seed=6)
    out, fin = run(x)
    state = x["init_state"].clone()
    outs = []
    for t in range(T):
        outs.append(kda.kda_decode_step(state, x["q"][t:t + 1], x["k"][t:t + 1],
                                        x["v"][t:t + 1], x["log_alpha"][t:t + 1],
                                        x["beta"][t:t + 1]))
    torch.cuda.synchronize()
    tol = TOL[dtype]
    assert_parity(torch.cat(outs), out, tol, name="out")
    assert_parity(state, fin, tol, name="state")


@pytest.mark.parametrize("dtype", DTYPES)
def test_host_cu_seqlens(dtype):
    x = inputs.prefill_inputs([100, 50], H=2, dtype=dtype, init_state=True, device=DEV, seed=7)
    o_dev, s_dev = run(x)
    o_dev, s_dev = o_dev.clone(), s_dev.clone()
    x["cu_seqlens"] = x["cu_seqlens"].cpu()
    o_host, s_host = run(x)
    assert torch.equal(o_dev, o_host) and torch.equal(s_dev, s_host)
    bad = dict(x)
    bad["cu_seqlens"] = torch.tensor([0, 120, 110], dtype=torch.int32)
    with pytest.raises(kda.KDAError) as e:
        run(bad)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", DTYPES)
def test_invalid_device_cu_seqlens_reports_status(dtype):
    x = inputs.prefill_inputs([100, 50], H=2, dtype=dtype, device=DEV, seed=8)
    x["cu_seqlens"] = torch.tensor([0, 120, 110], dtype=torch.int32, device=DEV)
    ws = torch.zeros(kda.kda_chunk_fwd_workspace_size(2, 150, 2, dtype=
                                                      kda.KDA_BF16 if dtype == "bf16" else
                                                      kda.KDA_F32),
                     dtype=torch.uint8, device=DEV)
    run(x, workspace=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_read_device_status(ws) == kda.KDA_OK  # cleared by the read
    # a valid call afterwards on the same workspace reports OK
    x["cu_seqlens"] = torch.tensor([0, 100, 150], dtype=torch.int32, device=DEV)
    run(x, workspace=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
