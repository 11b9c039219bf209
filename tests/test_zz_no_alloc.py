"""kda_chunk_fwd_noalloc: the prefill entry point for callers that cannot give
the library device memory (their framework allocator owns all of it), checked
through the C ABI against the fp64 oracle and against kda_chunk_fwd on two
consecutive calls, and its status reader on a malformed device cu_seqlens.

Collected last on purpose: the entry point's device scratch is shared by every
call, so this file must also pass after all other tests ran in the process.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from gated_delta_rule_13_gb300 import inputs, kda
from parity_util import TOL, assert_parity, check_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _noalloc_c_call(x, out, fin, cu):
    """Raw C-ABI call: no workspace argument, raw device pointers."""
    lib = kda.library()
    vp = ctypes.c_void_p
    N, H, dk = x["q"].shape
    n_seqs = cu.shape[0] - 1
    p = lambda t: vp(t.data_ptr()) if t is not None else vp(None)  # noqa: E731
    code = kda.KDA_BF16 if x["q"].dtype == torch.bfloat16 else kda.KDA_F32
    return lib.kda_chunk_fwd_noalloc(p(x["q"]), p(x["k"]), p(x["v"]), p(x["log_alpha"]),
                                     p(x["beta"]), p(x["init_state"]), p(cu), n_seqs, N, H, dk,
                                     x["v"].shape[2], code, p(out), p(fin),
                                     vp(torch.cuda.current_stream().cuda_stream))


def _status_c_call():
    st = ctypes.c_int32(-1)
    rc = kda.library().kda_noalloc_read_status(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), 1, ctypes.byref(st))
    assert rc == kda.KDA_OK
    return st.value


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(dtype):
    for call, (lengths, seed, host_cu) in enumerate([([300, 0, 129, 64], 11, False),
                                                     ([77, 1024, 5], 12, True)]):
        x = inputs.prefill_inputs(lengths, H=3, dtype=dtype, init_state=True, device=DEV,
                                  seed=seed)
        ref_out, ref_fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                             x["init_state"], x["cu_seqlens"])
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        cu = x["cu_seqlens"].cpu() if host_cu else x["cu_seqlens"]
        rc = _noalloc_c_call(x, out, fin, cu)
        torch.cuda.synchronize()
        assert rc == kda.KDA_OK, f"call {call}: {kda.status_string(rc)}"
        assert _status_c_call() == kda.KDA_OK
        assert torch.isfinite(out).all() and torch.isfinite(fin).all()
        check_prefill(x, out, fin, TOL[dtype])
        cu_np = x["cu_seqlens"].cpu().numpy()
        assert_parity(out, ref_out, TOL[dtype], cu=cu_np, name=f"out vs kda_chunk_fwd, call {call}")
        assert_parity(fin, ref_fin, TOL[dtype], name=f"final state vs kda_chunk_fwd, call {call}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_status_reports_malformed_device_cu_seqlens(dtype):
    """The call returns KDA_OK (the kernel validates a device cu_seqlens); the
    status reader returns what the kernel recorded, then the cleared status."""
    x = inputs.prefill_inputs([100, 50], H=2, dtype=dtype, device=DEV, seed=13)
    bad = torch.tensor([0, 120, 110], dtype=torch.int32, device=DEV)
    out = torch.empty_like(x["v"])
    assert _noalloc_c_call(x, out, None, bad) == kda.KDA_OK
    assert _status_c_call() == kda.KDA_ERR_INVALID_ARG
    assert _status_c_call() == kda.KDA_OK
    assert _noalloc_c_call(x, out, None, x["cu_seqlens"]) == kda.KDA_OK
    assert _status_c_call() == kda.KDA_OK


def test_noalloc_rejects_too_many_sequences():
    x = inputs.prefill_inputs([1] * 8, H=1, dtype="bf16", device=DEV)
    cu = torch.arange(4097, dtype=torch.int32, device=DEV)   # 4096 sequences
    x["cu_seqlens"] = cu
    x["q"] = x["q"].new_zeros(4096, 1, 128)
    x["k"] = x["k"].new_zeros(4096, 1, 128)
    x["v"] = x["v"].new_zeros(4096, 1, 128)
    x["log_alpha"] = x["log_alpha"].new_zeros(4096, 1, 128)
    x["beta"] = x["beta"].new_zeros(4096, 1)
    x["init_state"] = None
    out = torch.empty(4096, 1, 128, dtype=torch.bfloat16, device=DEV)
    assert _noalloc_c_call(x, out, None, cu) == kda.KDA_ERR_WORKSPACE
