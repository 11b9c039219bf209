"""Context parallelism across ranks (KCP) on the host: two and three gloo
processes each hold one segment of every sequence and run ``kcp_chunk_fwd``
with the oracle as the compute of its three steps, so the test covers the
exchange and the composition, not the kernels.  The stitched result must be
the oracle's over the whole sequences (fp64 throughout)."""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LENGTHS = [300, 70, 0, 513]
H, D = 2, 8


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    from gated_delta_rule_13_gb300 import inputs
    x = inputs.prefill_inputs(LENGTHS, H=H, dtype="f32", init_state=True, device="cpu", seed=51,
                              dk=D, dv=D)
    x["log_alpha"].mul_(0.05)  # slow decay: the segments' transitions matter
    return x


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    from gated_delta_rule_13_gb300.kcp import kcp_chunk_fwd
    from kcp_util import OracleOps, rank_segments
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = _inputs()
        local, idx = rank_segments(x, world, rank)
        out, end = kcp_chunk_fwd(local["q"], local["k"], local["v"], local["log_alpha"],
                                 local["beta"], x["init_state"], local["cu_seqlens"],
                                 ops=OracleOps)
        q.put((rank, idx.numpy(), out.numpy(), end.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_kcp_gloo_ranks_match_whole_sequences(world):
    import torch.multiprocessing as mp
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x = _inputs()
    o_ref, s_ref = oracle.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                    x["init_state"], x["cu_seqlens"])
    out = np.full_like(o_ref, np.nan)
    for _, idx, o, end in results:
        out[idx] = o
        np.testing.assert_allclose(end, s_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out, o_ref, rtol=1e-10, atol=1e-12)
