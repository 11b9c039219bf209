"""Shared helpers for the GPU parity tests (comparison with the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances on relative L2 error, per element type of q/k/v/out (fp32 state and
# accumulation in both cases).
TOL = {"f32": 1e-4, "bf16": 2e-2}

# A (sequence, head) slice gets its own relative-L2 check when its reference
# energy is at least this fraction of what an average row of its head would
# give it.  Below that (a one-token sequence whose q is nearly orthogonal to
# its k, say) the relative error measures the rounding floor of a tiny
# quantity rather than the slice; such slices are still bounded row by row.
SLICE_ENERGY_FLOOR = 0.25

# Each row's error is bounded by ROW_FACTOR x tol x max(||reference row||, RMS
# row norm of its head).  On the bf16 path the per-row error, in units of the
# head's RMS, has a median near 0.0033, a 99.9th percentile near 0.021 and a
# maximum of 0.026-0.046 over 10^4-10^6 rows (K3 layout, the 8192 x 8 helper
# case, the ragged case and the varlen sample, measured on a GB300): a row
# where the chunk's two output terms (pre-chunk state and intra-chunk causal)
# nearly cancel keeps the absolute rounding of the larger terms, and a large
# row keeps an error proportional to itself.  A bound of 1 x tol per row would
# therefore reject correct results; 5 x tol (10 % for bf16) still fails any
# row that is actually wrong (an error of the order of the row or the head).
ROW_FACTOR = 5.0


def _np(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_l2(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 over the whole tensor, in fp64."""
    x = _np(x)
    ref = _np(ref)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


def _rows(x, cu):
    """Normalise to rows [R, H, d] and the row bounds of the sequences."""
    if x.ndim == 4:            # states [S, H, dk, dv]: sequence s = rows s*dk .. s*dk + dk - 1
        S, H, dk, dv = x.shape
        return x.transpose(0, 2, 1, 3).reshape(S * dk, H, dv), np.arange(S + 1) * dk
    if x.ndim != 3:
        raise ValueError("expected [rows, H, d] or [S, H, dk, dv]")
    bounds = np.array([0, x.shape[0]]) if cu is None else np.asarray(cu, dtype=np.int64)
    if bounds[0] != 0 or bounds[-1] != x.shape[0] or np.any(np.diff(bounds) < 0):
        raise ValueError("cu must be row bounds from 0 to the row count")
    return x, bounds


def parity_report(got, ref, cu=None) -> dict:
    """Error of ``got`` against ``ref`` at three granularities.

    ``got`` and ``ref`` are outputs ``[rows, H, d]`` whose sequences are the
    row ranges ``cu`` (None: one sequence), or states ``[S, H, dk, dv]`` (one
    sequence per leading index, its rows the dk key rows).  Returns:
      whole      relative L2 over the whole tensor;
      row        the largest ||row error||_2 / max(||reference row||_2, RMS row
                 norm of the row's head (the RMS over every compared row of that
                 head)), and where;
      slice      the largest relative L2 of a (sequence, head) slice whose
                 reference energy passes SLICE_ENERGY_FLOOR, and where.
    A head whose reference is all zero must match exactly (its row ratio is
    the error norm itself)."""
    g, bounds = _rows(_np(got), cu)
    r, _ = _rows(_np(ref), cu)
    if g.shape != r.shape:
        raise ValueError(f"shape mismatch {g.shape} vs {r.shape}")
    R, H, _ = g.shape
    rep = {"whole": rel_l2(g, r), "row": 0.0, "row_at": None, "slice": 0.0, "slice_at": None}
    if R == 0:
        return rep
    err = np.linalg.norm(g - r, axis=2)               # [R, H]
    rn2 = np.sum(r * r, axis=2)                        # [R, H]
    rms = np.sqrt(np.mean(rn2, axis=0))                # [H]
    scale = np.maximum(np.sqrt(rn2), rms[None, :])
    ratio = np.where(scale > 0, err / np.where(scale > 0, scale, 1.0), err)
    ratio = np.where(np.isfinite(ratio), ratio, np.inf)
    i = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    seq = int(np.searchsorted(bounds, i[0], side="right") - 1)
    rep["row"] = float(ratio[i])
    rep["row_at"] = {"sequence": seq, "row_in_sequence": int(i[0] - bounds[seq]), "head": int(i[1])}
    for s in range(len(bounds) - 1):
        a, b = int(bounds[s]), int(bounds[s + 1])
        if b == a:
            continue
        e2 = np.sum(err[a:b] ** 2, axis=0)             # [H]
        n2 = np.sum(rn2[a:b], axis=0)
        for h in range(H):
            if rms[h] == 0 or n2[h] < SLICE_ENERGY_FLOOR * (b - a) * rms[h] ** 2:
                continue
            q = float(np.sqrt(e2[h] / n2[h])) if np.isfinite(e2[h]) else float("inf")
            if not q <= rep["slice"]:
                rep["slice"] = q
                rep["slice_at"] = {"sequence": s, "head": h}
    return rep


def assert_parity(got, ref, tol, cu=None, name="out"):
    """Asserts the errors of ``parity_report``: the whole tensor's relative L2
    and every (sequence, head) slice's relative L2 within ``tol``, and every
    row's error within ROW_FACTOR x ``tol`` of the larger of its own norm and
    its head's RMS row norm.  A single wrong token row, a wrong short sequence
    or a wrong head fails it even where the whole-tensor figure would hide it.
    Returns the report."""
    rep = parity_report(got, ref, cu)
    assert rep["whole"] <= tol, f"{name}: rel L2 {rep['whole']:.3e} > {tol:g}"
    assert rep["slice"] <= tol, (f"{name}: (sequence, head) slice rel L2 {rep['slice']:.3e} > "
                                 f"{tol:g} at {rep['slice_at']}")
    assert rep["row"] <= ROW_FACTOR * tol, (
        f"{name}: row error {rep['row']:.3e} x max(row, head RMS) > {ROW_FACTOR * tol:g} at "
        f"{rep['row_at']}")
    return rep


def oracle_prefill(x, heads=None, seqs=None, n_threads=None):
    """Run the oracle on the prefill inputs ``x`` (from ``inputs.prefill_inputs``),
    optionally on a subset of heads and sequences.  Returns (out, final_state,
    token_index, sub_cu) where token_index maps oracle rows back to packed rows
    and sub_cu holds the row bounds of the chosen sequences in ``out``."""
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
    return out, fin, idx, sub_cu


def check_prefill(x, out, fin, tol, heads=None, seqs=None):
    """Oracle parity of a prefill's outputs and final states (``assert_parity``
    on both) on the chosen heads and sequences; returns the two reports."""
    o_ref, s_ref, idx, sub_cu = oracle_prefill(x, heads=heads, seqs=seqs)
    dev = out.device
    H = x["q"].shape[1]
    hsel = torch.as_tensor(heads if heads is not None else list(range(H)), device=dev)
    got_o = out.index_select(0, torch.as_tensor(idx, device=dev)).index_select(1, hsel)
    ro = assert_parity(got_o, o_ref, tol, cu=sub_cu, name="out")
    rs = None
    if fin is not None:
        n_seqs = x["cu_seqlens"].shape[0] - 1
        ssel = torch.as_tensor(seqs if seqs is not None else list(range(n_seqs)), device=dev)
        got_s = fin.index_select(0, ssel).index_select(1, hsel)
        rs = assert_parity(got_s, s_ref, tol, name="final state")
    return ro, rs
