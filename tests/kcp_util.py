"""Test helpers for context parallelism: the oracle as the compute of the KCP
steps (any head size, fp64, CPU), and the split of packed inputs into the
per-rank segments a KCP caller holds."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def _np(t):
    return t.detach().double().cpu().numpy()


class OracleOps:
    """The three compute steps of ``kcp_chunk_fwd`` by the fp64 oracle."""

    @staticmethod
    def pairs(q, k, v, log_alpha, beta, cu_seqlens):
        cu = _np(cu_seqlens).astype(np.int64)
        n_seqs, H, dk = cu.shape[0] - 1, q.shape[1], q.shape[2]
        _, b = oracle.chunk_fwd(_np(q), _np(k), _np(v), _np(log_alpha), _np(beta), None, cu)
        eye = np.broadcast_to(np.eye(dk), (n_seqs, H, dk, dk)).copy()
        zero_v = np.zeros(q.shape, dtype=np.float64)
        _, m = oracle.chunk_fwd(_np(q), _np(k), zero_v, _np(log_alpha), _np(beta), eye, cu)
        return torch.from_numpy(b), torch.from_numpy(m)

    @staticmethod
    def combine(state_b, state_m, n_segments, init_state):
        b, m = _np(state_b), _np(state_m)
        n_seqs = b.shape[0] // n_segments
        starts = np.zeros_like(b)
        end = np.zeros((n_seqs,) + b.shape[1:])
        for s in range(n_seqs):
            st = np.zeros(b.shape[1:]) if init_state is None else _np(init_state)[s]
            for j in range(n_segments):
                starts[s * n_segments + j] = st
                st = np.einsum("hck,hkn->hcn", m[s * n_segments + j], st) + b[s * n_segments + j]
            end[s] = st
        return torch.from_numpy(starts), torch.from_numpy(end)

    @staticmethod
    def forward(q, k, v, log_alpha, beta, init_state, cu_seqlens):
        out, _ = oracle.chunk_fwd(_np(q), _np(k), _np(v), _np(log_alpha), _np(beta),
                                  _np(init_state), _np(cu_seqlens).astype(np.int64))
        return torch.from_numpy(out)


def rank_segments(x, world, rank):
    """Rank ``rank``'s inputs: the rank-th of ``world`` contiguous pieces of
    every sequence (equal whole-chunk pieces; trailing ones may be empty),
    packed, with the token indices they came from."""
    cu = [int(c) for c in x["cu_seqlens"].tolist()]
    idx, lens = [], []
    for s in range(len(cu) - 1):
        a, n = cu[s], cu[s + 1] - cu[s]
        chunks = -(-n // 64)
        per = -(-chunks // world) * 64  # whole chunks per piece
        lo, hi = min(n, rank * per), min(n, (rank + 1) * per)
        idx.extend(range(a + lo, a + hi))
        lens.append(hi - lo)
    it = torch.tensor(idx, dtype=torch.long, device=x["q"].device)
    local = {n: x[n].index_select(0, it).contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    c = [0]
    for n in lens:
        c.append(c[-1] + n)
    local["cu_seqlens"] = torch.tensor(c, dtype=torch.int32, device=x["q"].device)
    return local, it
