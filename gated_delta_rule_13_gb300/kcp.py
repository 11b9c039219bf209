"""Context parallelism of the prefill across devices (KCP).

"Kimi K3: 架构、训练与系统全景解析", section 7.1: the recurrence maps the state a
sequence segment starts from to the one it ends with affinely,
S_end = M S_start + B (the segment's "affine pair"), and the pairs of
consecutive segments compose.  So devices that each hold one segment of the
same sequences need a single exchange:
  1. every rank computes its segment's pair (B, M)      kda_chunk_fwd_transitions
  2. all ranks all-gather the pairs (2 x 64 KiB per head and sequence)
  3. every rank composes the pairs of the ranks before it with the initial
     state into its start state, and all of them into the final state
                                                         kda_state_combine
  4. every rank runs its segment from its start state    kda_chunk_fwd
The compute of steps 1, 3 and 4 is the library's kernels (``ops``); the
exchange is one ``torch.distributed.all_gather`` (NCCL between GPUs).

Layout: rank r holds, for each of the same n_seqs sequences, the r-th
contiguous piece of its tokens (possibly empty), packed token-major with its
own cu_seqlens, like any kda_chunk_fwd input; all ranks have the same H.
"""
from __future__ import annotations

from . import kda


class KernelOps:
    """The library's kernels for the three compute steps."""

    @staticmethod
    def pairs(q, k, v, log_alpha, beta, cu_seqlens):
        return kda.kda_chunk_fwd_transitions(q, k, v, log_alpha, beta, cu_seqlens)

    @staticmethod
    def combine(state_b, state_m, n_segments, init_state):
        return kda.kda_state_combine(state_b, state_m, n_segments, init_state)

    @staticmethod
    def forward(q, k, v, log_alpha, beta, init_state, cu_seqlens):
        out, _ = kda.kda_chunk_fwd(q, k, v, log_alpha, beta, init_state, cu_seqlens,
                                   output_final_state=False)
        return out


def stack_pairs(pairs_by_rank):
    """Pairs gathered per rank (lists of ``[n_seqs, H, d, d]``) to the segment
    order the combine takes: segment r of sequence s at index ``s * W + r``."""
    import torch
    b = torch.stack([p[0] for p in pairs_by_rank], dim=1)
    m = torch.stack([p[1] for p in pairs_by_rank], dim=1)
    n_seqs, world = b.shape[0], b.shape[1]
    return (b.reshape(n_seqs * world, *b.shape[2:]).contiguous(),
            m.reshape(n_seqs * world, *m.shape[2:]).contiguous())


def start_state(state_b, state_m, rank, world, init_state=None, ops=KernelOps):
    """Start state of ``rank``'s segments ``[n_seqs, H, d, d]`` and the
    sequences' final states, from the stacked pairs of all ranks."""
    starts, end = ops.combine(state_b, state_m, world, init_state)
    n_seqs = end.shape[0]
    return starts.reshape(n_seqs, world, *starts.shape[1:])[:, rank].contiguous(), end


def kcp_chunk_fwd(q, k, v, log_alpha, beta, init_state=None, cu_seqlens=None, *, group=None,
                  ops=KernelOps):
    """KCP prefill of this rank's segment.  ``init_state`` is the sequences'
    initial state (the same on every rank, or None).  Returns this rank's
    outputs and the sequences' final states (the same on every rank)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    b, m = ops.pairs(q, k, v, log_alpha, beta, cu_seqlens)
    bs = [b.new_empty(b.shape) for _ in range(world)]
    ms = [m.new_empty(m.shape) for _ in range(world)]
    dist.all_gather(bs, b.contiguous(), group=group)
    dist.all_gather(ms, m.contiguous(), group=group)
    state_b, state_m = stack_pairs(list(zip(bs, ms)))
    start, end = start_state(state_b, state_m, rank, world, init_state, ops)
    out = ops.forward(q, k, v, log_alpha, beta, start, cu_seqlens)
    return out, end
