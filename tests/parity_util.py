"""Shared helpers for the GPU parity tests (comparison with the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances on relative L2 error, per element type of q/k/v/out (fp32 state and
# accumulation in both cases).
TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_l2(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 over the whole tensor, in fp64."""
    if isinstance(x, torch.Tensor):
        x = x.detach().double().cpu().numpy()
    if isinstance(ref, torch.Tensor):
        ref = ref.detach().double().cpu().numpy()
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


def oracle_prefill(x, heads=None, seqs=None, n_threads=None):
    """Run the oracle on the prefill inputs ``x`` (from ``inputs.prefill_inputs``),
    optionally on a subset of heads and sequences.  Returns (out, final_state,
    token_index) where token_index maps oracle rows back to packed rows."""
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    n_seqs = cu.shape[0] - 1
    seqs = list(range(n_seqs)) if seqs is None else list(seqs)
    H = x["q"].shape[1]
    heads = list(range(H)) if heads is None else list(heads)
    idx = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]) if seqs else np.zeros(0, np.int64)
    lens = [int(cu[s + 1] - cu[s]) for s in seqs]
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tidx = torch.as_tensor(idx, dtype=torch.long)
    hidx = torch.as_tensor(heads, dtype=torch.long)

    def take(t):
        return t.detach().cpu().index_select(0, tidx).index_select(1, hidx)

    s0 = None
    if x["init_state"] is not None:
        s0 = x["init_state"].detach().cpu()[torch.as_tensor(seqs)][:, hidx]
    out, fin = oracle.chunk_fwd(take(x["q"]), take(x["k"]), take(x["v"]), take(x["log_alpha"]),
                                take(x["beta"]), s0, sub_cu, n_threads=n_threads)
    return out, fin, idx
