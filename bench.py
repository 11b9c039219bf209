"""Benchmark of the KDA recurrence hot path on GB300.

One step = one chunked prefill (kda_chunk_fwd) over the K3 head layout
(B=1, H=96, T=32768, d=128, bf16 q/k/v, fp32 log_alpha/beta, fp32 final state)
plus one in-place decode step (kda_decode_step) over 512 sequences x 96 heads.
``value`` is prefill tokens/s (the prefill kernel's CUDA-event time over the
timed steps); the decode step is reported beside it in GB/s against the HBM
peak.  Inputs are synthetic (seeded, ``gated_delta_rule_13_gb300.inputs``) and
larger than L2, so no flush is needed between iterations.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica on its own GPU (the path has no exchange step): value = all ranks'
tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (H=96,d=128, % tensor roofline); decode GB/s vs HBM peak"
PREFILL_FLOP_PER_TOKEN_HEAD = 139264      # 5*C*d + 6*d^2 at C = 64, d = 128
PREFILL_BYTES_PER_TOKEN_HEAD = 1540       # bf16 q,k,v,out + fp32 log_alpha + fp32 beta
STATE_BYTES = 128 * 128 * 4
DECODE_BYTES_PER_UNIT = 2 * STATE_BYTES + 3 * 256 + 512 + 4 + 256
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def recorded_traffic(kernel: str, source: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.txt),
    or None when the kernel source changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = os.path.join(ROOT, "gated_delta_rule_13_gb300", "csrc", source)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for line in open(path):
        f = line.split()
        if len(f) == 4 and not line.startswith("#") and f[0] == kernel and f[2] == workload:
            return int(f[3]) if f[1] == digest else None
    return None


def max_over_ranks(values, world: int, device="cpu"):
    """Element-wise maximum of this rank's floats over all ranks (one all_reduce
    MAX; the identity for a single process).  Used for every time the JSON line
    reports, so that N replicas are timed by their slowest rank."""
    values = [float(v) for v in values]
    if world == 1:
        return values
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"kda_clocks_{gpu_index}_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- oracle (CPU)
def oracle_rate(workload, n_heads_sample: int, n_tokens_sample: int, seed=0):
    """Times the fp64 oracle on `n_heads_sample` heads x the first
    `n_tokens_sample` tokens of the workload; returns (token-heads/s, threads, desc)."""
    import numpy as np
    import oracle
    from gated_delta_rule_13_gb300 import inputs
    w = inputs.WORKLOADS[workload]
    x = inputs.prefill_inputs([n_tokens_sample], H=n_heads_sample, dtype=w.dtype,
                              init_state=w.init_state, device="cpu", seed=seed)
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                     np.array([0, n_tokens_sample]), n_threads=threads)
    dt = time.perf_counter() - t0
    th = n_heads_sample * n_tokens_sample
    desc = (f"oracle on {n_heads_sample} heads x {n_tokens_sample} tokens of {workload} "
            f"(same value distributions), {threads} threads, {dt:.2f} s")
    return th / dt, threads, desc, dt


def calibrated_sample(workload, target_s: float):
    """Chooses (heads, tokens) of the workload so that one multi-threaded oracle
    run takes about `target_s` seconds: first one head per host thread, growing
    the token count up to the sequence length, then more heads."""
    import oracle
    from gated_delta_rule_13_gb300 import inputs
    w = inputs.WORKLOADS[workload]
    threads = oracle.default_threads()
    rate1, _, _, _ = oracle_rate(workload, 1, 256)        # single chain = single thread
    heads = min(w.H, threads)
    T = int(max(256, min(w.seq_lengths[0], target_s * rate1)))
    if T >= w.seq_lengths[0]:
        rounds = max(1, int(target_s * rate1 / T))
        heads = min(w.H, threads * rounds)
    return heads, T


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from gated_delta_rule_13_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    budget = args.ref_step_s if args.ref_step_s > 0 else max(0.5, 150.0 / (args.steps + args.warmup))
    heads, T = calibrated_sample(args.workload, budget)
    rates = []
    desc = ""
    threads = 1
    for s in range(args.warmup + args.steps):
        rate, threads, desc, dt = oracle_rate(args.workload, heads, T, seed=s)
        if s >= args.warmup:
            rates.append(rate)
    th_rate = statistics.median(rates)
    value = th_rate / w.H                      # tokens/s of the H-head workload
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * heads * T / th_rate, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": args.workload, "note": w.note},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- GPU arm
def replay_bench(dev, peaks, steps: int = 20, warmup: int = 3, T: int = 4, B: int = 512):
    """kda_decode_replay on B (default 512) sequences x 96 heads x T cached draft tokens with
    seeded accepted counts in [0, T] (the step after a speculative verification).
    Algorithmic bytes: one state read and write per unit with an accepted token,
    plus the accepted tokens' inputs and outputs."""
    import torch
    from gated_delta_rule_13_gb300 import inputs, kda
    H = 96
    d = inputs.decode_inputs(B=B, H=H, steps=T, dtype="bf16", device=dev, seed=17)
    r = {x: d[x].transpose(0, 1).contiguous() for x in ("q", "k", "v", "log_alpha", "beta")}
    state = d["state"]
    g = torch.Generator(device="cpu").manual_seed(17)
    n = torch.randint(0, T + 1, (B,), generator=g, dtype=torch.int32)
    n_dev = n.to(dev)
    out = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)

    def run():
        kda.kda_decode_replay(state, r["q"], r["k"], r["v"], r["log_alpha"], r["beta"], n_dev,
                              out=out)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        run()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    accepted = int(n.sum())
    active = int((n > 0).sum())
    nbytes = H * (active * 2 * STATE_BYTES + accepted * (DECODE_BYTES_PER_UNIT - 2 * STATE_BYTES))
    gbs = nbytes / (ms / 1000.0) / 1e9
    del d, r, state, out
    return {"value": gbs, "unit": "GB/s", "ms_per_launch": ms,
            "workload": f"{B} sequences x 96 heads, {T} cached draft tokens, accepted counts "
                        f"seeded uniform in [0, {T}] (mean {accepted / B:.2f})",
            "accepted_tokens_per_s": accepted / (ms / 1000.0),
            "roofline": {"bound": "hbm", "kernel": "kda_decode_replay_kernel", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("kda_decode_replay_kernel", "kda_decode.cu",
                                                     f"replay_b{B}_h{H}_t{T}"),
                         "bytes_per_launch": nbytes}}


def layer_replay_bench(dev, peaks, steps: int = 20, warmup: int = 3, T: int = 4, B: int = 512):
    """kda_layer_replay (the layer between its projections, fused, over the
    accepted drafts) on B (default 512) sequences x 96 heads x T cached drafts, accepted
    counts seeded uniform in [0, T].  Algorithmic bytes per unit with an
    accepted token: the state and the bf16 convolution window read and written
    once, plus per accepted token the raw q, k, v and gate logits (bf16), the
    decay logits (fp32), the beta logit and the bf16 output."""
    import torch
    from gated_delta_rule_13_gb300 import inputs, kda
    H = 96
    x = inputs.layer_inputs([T] * B, H=H, dtype="bf16", device=dev, seed=19)
    r = {n: x[n].reshape(B, T, H, *x[n].shape[2:]) for n in
         ("q_raw", "k_raw", "v_raw", "a_logit", "b_logit", "g")}
    gen = torch.Generator(device=dev).manual_seed(19)
    state = 0.02 * torch.randn(B, H, 128, 128, generator=gen, device=dev)
    win = torch.randn(B, 3, 3, H, 128, generator=gen, device=dev).to(torch.bfloat16)
    g = torch.Generator(device="cpu").manual_seed(19)
    n = torch.randint(0, T + 1, (B,), generator=g, dtype=torch.int32)
    n_dev = n.to(dev)
    out = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)

    def run():
        kda.kda_layer_replay(state, win, r["q_raw"], r["k_raw"], r["v_raw"], r["a_logit"],
                             r["b_logit"], r["g"], x["conv_w"], x["gamma"], n_dev, out=out)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        run()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    accepted = int(n.sum())
    active = int((n > 0).sum())
    per_tok = 3 * 256 + 512 + 4 + 256 + 256
    nbytes = H * (active * (2 * STATE_BYTES + 2 * 9 * 256) + accepted * per_tok)
    gbs = nbytes / (ms / 1000.0) / 1e9
    del x, r, state, win, out
    return {"value": gbs, "unit": "GB/s", "ms_per_launch": ms,
            "workload": f"{B} sequences x 96 heads, {T} cached drafts (raw projections, bf16), "
                        f"accepted counts seeded uniform in [0, {T}] (mean {accepted / B:.2f})",
            "accepted_tokens_per_s": accepted / (ms / 1000.0),
            "roofline": {"bound": "hbm", "kernel": "kda_layer_replay_kernel", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("kda_layer_replay_kernel",
                                                     "kda_layer_ops.cu", f"b{B}_h{H}_t{T}"),
                         "bytes_per_launch": nbytes}}


def layer_ops_bench(dev, peaks, steps: int = 20, warmup: int = 3, T: int = 32768):
    """kda_prep_fwd and kda_post_fwd on the K3 layout (one sequence of T = 32768
    tokens, 96 heads, bf16).  Algorithmic bytes per token-head: prep reads
    q, k, v (bf16) and both gate logits and writes q, k, v, log_alpha and beta
    (2568 B); post reads o and the gate logits and writes the output (768 B)."""
    import torch
    from gated_delta_rule_13_gb300 import inputs, kda
    H = 96
    x = inputs.layer_inputs([T], H=H, dtype="bf16", device=dev, seed=29)
    o = x["v_raw"]

    def prep():
        return kda.kda_prep_fwd(x["q_raw"], x["k_raw"], x["v_raw"], x["conv_w"], x["a_logit"],
                                x["b_logit"], x["cu_seqlens"])

    y = torch.empty_like(o)

    def post():
        kda.kda_post_fwd(o, x["g"], x["gamma"], out=y)

    res = {}
    stream = torch.cuda.current_stream()
    for name, fn, per_th in (("prep", prep, 2568), ("post", post, 768)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        nbytes = T * H * per_th
        gbs = nbytes / (ms / 1000.0) / 1e9
        res[name] = {"value": gbs, "unit": "GB/s", "ms_per_launch": ms,
                     "tokens_per_s": T / (ms / 1000.0),
                     "roofline": {"bound": "hbm", "kernel": f"kda_{name}_kernel", "achieved": gbs,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": gbs / peaks["hbm_gbs"],
                                  "traffic": recorded_traffic(f"kda_{name}_kernel",
                                                              "kda_layer_ops.cu", f"t{T}_h{H}"),
                                  "bytes_per_launch": nbytes}}
    del x, o, y
    res["workload"] = f"one sequence of {T} tokens x 96 heads, bf16"
    return res


def few_chains_bench(dev, peaks, steps: int = 20, warmup: int = 3, T: int = 65536, H: int = 8):
    """Prefill of one long sequence over few heads (8 of K3's 96: the share of a
    GPU under head-sharded tensor parallelism), three ways: each (sequence, head)
    chain on one SM ("plain"), with helper CTAs on the idle SMs ("helpers"),
    and with the in-device split of the sequence into segments ("split", what
    kda_chunk_fwd picks for this shape)."""
    import torch
    from gated_delta_rule_13_gb300 import inputs, kda
    x = inputs.prefill_inputs([T], H=H, dtype="bf16", device=dev, seed=35)
    out = torch.empty_like(x["v"])
    fin = torch.empty(1, H, 128, 128, device=dev)
    res = {"workload": f"one sequence of {T} tokens x {H} heads, bf16"}
    stream = torch.cuda.current_stream()
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(1, T, H, dtype=kda.KDA_BF16),
                     dtype=torch.uint8, device=dev)
    # (max_split, max_helpers) of kda_chunk_fwd_sched; None: the library's choice
    variants = (("plain", (0, 0)), ("helpers", (0, None)), ("split", (None, None)))
    for name, (max_split, max_helpers) in variants:

        def run():
            kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None,
                              x["cu_seqlens"], out=out, final_state=fin, workspace=ws,
                              max_split=max_split, max_helpers=max_helpers)

        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            run()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        pub, used = kda.kda_read_chunk_stats(ws)
        gbs = prefill_bytes(x, H) / (ms / 1000.0) / 1e9
        res[name] = {"tokens_per_s": T / (ms / 1000.0), "ms_per_launch": ms,
                     "hbm_frac": gbs / peaks["hbm_gbs"]}
        if name == "helpers":
            res[name].update({"chunks_from_helpers": used, "packages_published": pub,
                              "chunks": H * ((T + 63) // 64)})
    for name in ("helpers", "split"):
        res[name]["speedup_vs_plain"] = res["plain"]["ms_per_launch"] / res[name]["ms_per_launch"]
    del x, out, fin, ws
    return res


def prefill_config_bench(dev, peaks, workload: str, steps: int, warmup: int = 3):
    """One prefill workload timed on its own (CUDA events over `steps` launches
    after `warmup`), with its roofline: the algorithmic bytes per token-head
    (bf16 q, k, v, out, fp32 log_alpha and beta) plus the states read and
    written, against the measured HBM copy peak."""
    import torch
    from gated_delta_rule_13_gb300 import inputs, kda
    w = inputs.WORKLOADS[workload]
    x = inputs.workload_inputs(workload, device=dev)
    n_tok, H = int(x["q"].shape[0]), w.H
    n_seqs = len(x["lengths"])
    bf16 = x["q"].dtype == torch.bfloat16
    out = torch.empty(n_tok, H, 128, dtype=x["q"].dtype, device=dev)
    fin = torch.empty(n_seqs, H, 128, 128, dtype=torch.float32, device=dev)
    ws = torch.zeros(kda.kda_chunk_fwd_workspace_size(
        n_seqs, n_tok, H, dtype=kda.KDA_BF16 if bf16 else kda.KDA_F32), dtype=torch.uint8,
        device=dev)

    def run():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                          x["cu_seqlens"], out=out, final_state=fin, workspace=ws)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        run()
    b.record(stream)
    torch.cuda.synchronize()
    ok = kda.kda_read_device_status(ws) == kda.KDA_OK
    ms = a.elapsed_time(b) / steps
    nbytes = prefill_bytes(x, H)
    gbs = nbytes / (ms / 1000.0) / 1e9
    flop = n_tok * H * PREFILL_FLOP_PER_TOKEN_HEAD
    res = {"workload": f"{workload}: {w.note}", "tokens": n_tok, "heads": H,
           "tokens_per_s": n_tok / (ms / 1000.0), "ms_per_launch": ms, "launches": steps,
           "device_status_ok": ok,
           "roofline": {"bound": "hbm",
                        "kernel": "kda_chunk_fwd_tc_kernel" if bf16 else "kda_chunk_fwd_f32_kernel",
                        "achieved": gbs,
                        "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                        "traffic": recorded_traffic("kda_chunk_fwd_tc_kernel", "kda_chunk_tc.cu",
                                                    workload) if bf16 else None,
                        "bytes_per_launch": nbytes,
                        "tensor_frac": flop / (ms / 1000.0) / 1e12 / peaks["bf16_tflops"]}}
    del x, out, fin, ws
    torch.cuda.empty_cache()
    return res


def decode_sequence_bench(dev, peaks, steps: int = 100, warmup_steps: int = 3, seed: int = 0):
    """The decode workload as specified: 512 sequences x 96 heads, `steps`
    consecutive steps, each with fresh inputs, the fp32 state advanced in place
    by every step.  CUDA events around every step; algorithmic bytes per step:
    each state read and written once plus the token's q, k, v, log_alpha, beta
    and output."""
    import torch
    from gated_delta_rule_13_gb300 import inputs, kda
    dw = inputs.WORKLOADS["decode_b512_h96"]
    d = inputs.decode_inputs(B=dw.B, H=dw.H, steps=steps, dtype=dw.dtype, device=dev, seed=seed)
    state = d["state"]
    out = torch.empty(dw.B, dw.H, 128, dtype=torch.bfloat16, device=dev)

    def step(s):
        kda.kda_decode_step(state, d["q"][s], d["k"][s], d["v"][s], d["log_alpha"][s],
                            d["beta"][s], out=out)

    for s in range(warmup_steps):          # warm-up on a copy of the state
        st0 = state.clone()
        step(s % steps)
        state.copy_(st0)
        del st0
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for s in range(steps):
        step(s)
        ev[s + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[s].elapsed_time(ev[s + 1]) for s in range(steps)]
    ms = sum(per) / steps
    nbytes = dw.B * dw.H * DECODE_BYTES_PER_UNIT
    gbs = nbytes / (ms / 1000.0) / 1e9
    res = {"value": gbs, "unit": "GB/s", "ms_per_step": ms,
           "ms_per_step_median": statistics.median(per), "ms_per_step_max": max(per),
           "steps_in_sequence": steps, "tokens_per_s": dw.B / (ms / 1000.0),
           "workload": f"decode_b512_h96: {dw.note}; fresh inputs each step, "
                       f"{steps * d['q'][0].numel() * 2 * 3 / 1e9:.1f} GB of q, k, v in HBM",
           "roofline": {"bound": "hbm", "kernel": "kda_decode_step_kernel", "achieved": gbs,
                        "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                        "traffic": recorded_traffic("kda_decode_step_kernel", "kda_decode.cu",
                                                    "decode_b512_h96"),
                        "bytes_per_launch": nbytes}}
    del d, state, out
    torch.cuda.empty_cache()
    return res


# Backward pass: flops per token-head of the minimal chain rule with the states
# at hand (X, p and S_t of the forward step, 3 d^2 multiply-adds; dS += q do^T,
# dq, dd, dk (two terms), dX, dlog_alpha and dS_{t-1}, 8 d^2), 2 flops each.
BWD_FLOP_PER_TOKEN_HEAD = 2 * 11 * 128 * 128
# Bytes per token-head (bf16): q, k, v, d_out in, dq, dk, dv out (7 x 256), fp32
# log_alpha in and its gradient out (2 x 512), beta and its gradient (8).
BWD_BYTES_PER_TOKEN_HEAD = 7 * 256 + 2 * 512 + 8


def fp32_alu_peak_tflops(dev):
    """FP32 FMA peak from the unit counts: SMs x 128 FP32 lanes x 2 flops x the
    maximum SM clock (2,070 MHz on a GB300)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return sms * 128 * 2 * 2.07e9 / 1e12


def backward_bench(dev, peaks, workload: str = "b4_h16_t4096", steps: int = 5, warmup: int = 2):
    """kda_chunk_bwd on a prefill workload (every gradient, random output and
    final-state gradients): for bf16 the chunked pass (its checkpoint kernel and
    the reverse chunk kernel, warp-level bf16 MMAs), CUDA events around each
    call.  Roofline: the token form's flops against the measured bf16 tensor
    peak (the pass is bound by its serial chunk steps, not by either roof)."""
    import torch
    from gated_delta_rule_13_gb300 import inputs, kda
    w = inputs.WORKLOADS[workload]
    x = inputs.workload_inputs(workload, device=dev)
    n_tok, H = int(x["q"].shape[0]), w.H
    n_seqs = len(x["lengths"])
    g = torch.Generator(device=dev).manual_seed(7)
    do = torch.randn(n_tok, H, 128, generator=g, device=dev).to(x["q"].dtype)
    df = torch.randn(n_seqs, H, 128, 128, generator=g, device=dev)
    ws = torch.empty(kda.kda_chunk_bwd_workspace_size(n_seqs, n_tok, H), dtype=torch.uint8,
                     device=dev)

    def run():
        kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                          x["cu_seqlens"], do, df, workspace=ws)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        run()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    th = n_tok * H
    tflops = th * BWD_FLOP_PER_TOKEN_HEAD / (ms / 1000.0) / 1e12
    peak = peaks["bf16_tflops"]
    nbytes = th * BWD_BYTES_PER_TOKEN_HEAD + n_seqs * H * 3 * STATE_BYTES
    del x, do, df, ws
    torch.cuda.empty_cache()
    return {"workload": f"{workload}: {w.note}", "ms_per_launch": ms,
            "tokens_per_s": n_tok / (ms / 1000.0),
            "hbm_gbs": nbytes / (ms / 1000.0) / 1e9,
            "chunk_steps_per_chain": -(-n_tok // n_seqs // 16),
            "roofline": {"bound": "tensor", "kernel": "kda_bwd_chunk_kernel", "achieved": tflops,
                         "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "peak_source": "measured bf16 burst (MEASURED_PEAKS.json)",
                         "alu_frac": tflops / fp32_alu_peak_tflops(dev),
                         "traffic": recorded_traffic("kda_bwd_chunk_kernel", "kda_bwd_chunk.cu",
                                                     workload),
                         "flop_per_launch": th * BWD_FLOP_PER_TOKEN_HEAD}}


def prefill_bytes(x, H):
    """Algorithmic bytes of one prefill launch: per token-head q, k, v and the
    output in the input type, fp32 log_alpha and beta (1,540 B for bf16, 2,564 B
    for fp32), plus the states read and written."""
    import torch
    n_tok = int(x["q"].shape[0])
    n_seqs = int(x["cu_seqlens"].shape[0] - 1)
    states = n_seqs * H * (2 if x["init_state"] is not None else 1)
    per_th = PREFILL_BYTES_PER_TOKEN_HEAD if x["q"].dtype == torch.bfloat16 else 4 * 128 * 4 + 512 + 4
    return n_tok * H * per_th + states * STATE_BYTES


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from gated_delta_rule_13_gb300 import inputs, kda

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (use --impl reference for the CPU oracle)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    w = inputs.WORKLOADS[args.workload]
    H = w.H

    # ---- inputs resident in HBM
    x = inputs.workload_inputs(args.workload, device=dev, seed=rank)
    n_tok = int(x["q"].shape[0])
    out = torch.empty(n_tok, H, 128, dtype=torch.bfloat16, device=dev)
    fin = torch.empty(len(x["lengths"]), H, 128, 128, dtype=torch.float32, device=dev)
    ws = torch.zeros(kda.kda_chunk_fwd_workspace_size(len(x["lengths"]), n_tok, H),
                     dtype=torch.uint8, device=dev)
    dw = inputs.WORKLOADS["decode_b512_h96"]
    n_dec_steps = args.warmup + args.steps     # fresh decode inputs for every step
    d = inputs.decode_inputs(B=dw.B, H=dw.H, steps=n_dec_steps, dtype=dw.dtype, device=dev,
                             seed=rank)
    state = d["state"]
    dout = torch.empty(dw.B, dw.H, 128, dtype=torch.bfloat16, device=dev)

    def prefill():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                          x["cu_seqlens"], out=out, final_state=fin, workspace=ws)

    def decode(s):
        i = s % n_dec_steps
        kda.kda_decode_step(state, d["q"][i], d["k"][i], d["v"][i], d["log_alpha"][i],
                            d["beta"][i], out=dout)

    for s in range(args.warmup):
        prefill()
        decode(s)
    torch.cuda.synchronize()
    if kda.kda_read_device_status(ws) != kda.KDA_OK:
        raise RuntimeError("prefill kernel reported a device error during warm-up")

    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for s in range(args.steps):
            e0, e1, e2 = ev[s]
            e0.record(stream)
            prefill()
            e1.record(stream)
            decode(args.warmup + s)
            e2.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    pre_ms = [a.elapsed_time(b) for a, b, _ in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    tot_ms = sum(step_ms)
    pre_avg = sum(pre_ms) / len(pre_ms)
    dec_avg = sum(dec_ms) / len(dec_ms)
    tot_ms, pre_avg, dec_avg = max_over_ranks([tot_ms, pre_avg, dec_avg], world, dev)
    status_ok = kda.kda_read_device_status(ws) == kda.KDA_OK

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        host = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "log_alpha", "beta")}
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_fin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
        dev_bufs = {k: torch.empty_like(x[k]) for k in host}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = h_out.numel() * h_out.element_size() + h_fin.numel() * h_fin.element_size()

        one_seq = int(x["cu_seqlens"].shape[0]) == 2
        h_init = x["init_state"].cpu().pin_memory() if x["init_state"] is not None else None

        def e2e_step():
            if one_seq:  # pieces of 4096 tokens, copies overlapping the prefill
                kda.kda_chunk_fwd_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                       host["beta"], h_init, out=h_out, final_state=h_fin,
                                       device=dev)
                return
            for k2 in host:
                dev_bufs[k2].copy_(host[k2], non_blocking=True)
            kda.kda_chunk_fwd(dev_bufs["q"], dev_bufs["k"], dev_bufs["v"], dev_bufs["log_alpha"],
                              dev_bufs["beta"], x["init_state"], x["cu_seqlens"], out=out,
                              final_state=fin, workspace=ws)
            h_out.copy_(out, non_blocking=True)
            h_fin.copy_(fin, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(1, min(args.steps, 5))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms, = max_over_ranks([a.elapsed_time(b) / n_e2e], world, dev)
        e2e = {"value": world * n_tok / (e2e_ms / 1000.0), "unit": "tokens/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        del host, dev_bufs

    pbytes = prefill_bytes(x, H)
    del x, out, fin, ws, d, state, dout
    torch.cuda.empty_cache()
    decode_seq = decode_sequence_bench(dev, peaks, steps=args.decode_steps, seed=rank)
    replay = replay_bench(dev, peaks, steps=args.sub_steps, B=args.replay_batch)
    few_chains = few_chains_bench(dev, peaks, steps=args.sub_steps)
    layer_ops = layer_ops_bench(dev, peaks, steps=args.sub_steps, T=args.layer_tokens)
    layer_replay = layer_replay_bench(dev, peaks, steps=args.sub_steps, B=args.replay_batch)
    backward = backward_bench(dev, peaks) if args.backward else None
    configs = {}
    for wl, n in (("tiny_f32", args.sub_steps), ("b4_h16_t4096", args.sub_steps),
                  ("varlen_h96_1m", args.varlen_steps)):
        if n > 0:
            configs[wl] = prefill_config_bench(dev, peaks, wl, steps=n)
    if world > 1:
        replay["ms_per_launch"], = max_over_ranks([replay["ms_per_launch"]], world, dev)
        layer_replay["ms_per_launch"], = max_over_ranks([layer_replay["ms_per_launch"]], world,
                                                        dev)
        decode_seq["ms_per_step"], = max_over_ranks([decode_seq["ms_per_step"]], world, dev)
        for c in configs.values():
            c["ms_per_launch"], = max_over_ranks([c["ms_per_launch"]], world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        heads, T = calibrated_sample(args.workload, args.cpu_seconds)
        rate, threads, desc, _ = oracle_rate(args.workload, heads, T)
        cpu = {"value": rate / H, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": desc}

    if rank != 0:
        return 0
    pflop = n_tok * H * PREFILL_FLOP_PER_TOKEN_HEAD
    achieved_gbs = pbytes / (pre_avg / 1000.0) / 1e9
    dbytes = dw.B * dw.H * DECODE_BYTES_PER_UNIT
    dec_gbs = dbytes / (dec_avg / 1000.0) / 1e9
    tokens_per_s = world * n_tok / (pre_avg / 1000.0)
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "note": w.note, "tokens": n_tok, "heads": H,
                   "decode_workload": "decode_b512_h96: 512 sequences x 96 heads, fp32 state",
                   "l2": f"inputs {pbytes / 1e9:.1f} GB and decode state "
                         f"{dbytes / 1e9:.1f} GB exceed the {L2_BYTES >> 20} MiB L2; no flush",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "kda_chunk_fwd_tc_kernel",
                     "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved_gbs / peaks["hbm_gbs"],
                     "traffic": recorded_traffic("kda_chunk_fwd_tc_kernel", "kda_chunk_tc.cu",
                                                 args.workload),
                     "peak_source": peaks["source"], "bytes_per_launch": pbytes,
                     "ms_per_launch": pre_avg,
                     "tensor_tflops": pflop / (pre_avg / 1000.0) / 1e12,
                     "tensor_frac": pflop / (pre_avg / 1000.0) / 1e12 / peaks["bf16_tflops"]},
        "decode": dict(decode_seq, in_step={
            "ms_per_step": dec_avg, "value": dec_gbs, "unit": "GB/s",
            "frac": dec_gbs / peaks["hbm_gbs"],
            "note": "the decode step inside each timed step, after the prefill"}),
        "prefill_configs": configs,
        "replay": replay,
        "prefill_few_chains": few_chains,
        "layer_ops": layer_ops,
        "layer_replay": layer_replay,
        "backward": backward,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
        "device_status_ok": status_ok,
        "wall_s_timed": t_wall,
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="k3_h96_t32768",
                    choices=["k3_h96_t32768", "b4_h16_t4096", "varlen_h96_1m"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target duration of the CPU oracle baseline sample")
    ap.add_argument("--ref-step-s", type=float, default=0.0,
                    help="target duration of one reference-arm step (default: about 150 s "
                         "spread over all steps)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sub-steps", type=int, default=20,
                    help="timed launches of the replay and per-token-step sub-benchmarks")
    ap.add_argument("--layer-tokens", type=int, default=32768,
                    help="tokens of the per-token-step sub-benchmark (96 heads)")
    ap.add_argument("--replay-batch", type=int, default=512,
                    help="sequences of the two replay sub-benchmarks (96 heads, 4 drafts)")
    ap.add_argument("--decode-steps", type=int, default=100,
                    help="consecutive in-place steps of the decode sub-benchmark")
    ap.add_argument("--no-backward", dest="backward", action="store_false",
                    help="skip the backward-pass sub-benchmark")
    ap.add_argument("--varlen-steps", type=int, default=5,
                    help="timed launches of the million-token varlen prefill (0: skip it)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
