"""Seeded synthetic inputs for the KDA recurrence.

This module only draws random tensors with the value distributions of the
workloads below; it holds none of the recurrence's arithmetic.  Tests, the
oracle comparison and ``bench.py`` all take their inputs from here, so the CUDA
path and the oracle always see identical values.

Value recipe (shared by every workload):
  * q, k ~ N(0, 1), then L2-normalised per (token, head) in fp32 and cast to the
    workload dtype (the KDA layer normalises q and k before the recurrence:
    "Kimi K3: 架构、训练与系统全景解析" section 4.2.3);
  * v ~ N(0, 1);
  * log_alpha = -5 * sigmoid(z), z ~ N(0, 1) per channel, fp32 (decay bounded
    below by -5: same page, sections 2.1 and 4.2.5);
  * beta = sigmoid(N(0, 1)), fp32;
  * initial states, where a workload has them, ~ N(0, 0.02^2), fp32.
Tensors are drawn slice by slice along the token axis (``SLICE`` tokens at a
time, order q, k, v, z_alpha, z_beta inside a slice) from one generator seeded
with ``seed``, then the initial state; this bounds the temporary memory of the
million-token workload and keeps small and large cases on the same recipe.
"""
from __future__ import annotations

import itertools

from dataclasses import dataclass, field

import torch

DK = 128
DV = 128
SLICE = 1 << 16
LOG_ALPHA_FLOOR = -5.0
STATE_STD = 0.02


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prefill" or "decode"
    H: int
    dtype: str                # "f32" or "bf16": dtype of q, k, v and out
    B: int = 1                # sequences (prefill, fixed length) or decode batch
    T: int = 0                # tokens per sequence (fixed-length prefill)
    lengths: tuple = ()       # explicit per-sequence lengths (varlen prefill)
    init_state: bool = False  # draw random initial states
    steps: int = 1            # decode steps
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def seq_lengths(self) -> list[int]:
        return list(self.lengths) if self.lengths else [self.T] * self.B

    @property
    def n_tokens(self) -> int:
        return int(sum(self.seq_lengths))


def varlen_lengths(n_seqs: int = 8, lo: int = 1024, hi: int = 262144, seed: int = 0):
    """Sequence lengths drawn uniformly from [lo, hi] on a CPU generator."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n_seqs,), generator=g))


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "prefill", H=1, dtype="f32", B=1, T=512,
                         note="B=1, H=1, T=512, fp32, zero initial state"),
    "b4_h16_t4096": Workload("b4_h16_t4096", "prefill", H=16, dtype="bf16", B=4, T=4096,
                             init_state=True,
                             note="B=4, H=16, T=4096, bf16, random fp32 initial state"),
    "k3_h96_t32768": Workload("k3_h96_t32768", "prefill", H=96, dtype="bf16", B=1, T=32768,
                              note="K3 head layout: B=1, H=96, T=32768, bf16, zero initial state"),
    "varlen_h96_1m": Workload("varlen_h96_1m", "prefill", H=96, dtype="bf16",
                              lengths=varlen_lengths(), init_state=True,
                              note="8 packed sequences of 1k-262k tokens (about 1M), H=96, bf16"),
    "decode_b512_h96": Workload("decode_b512_h96", "decode", H=96, dtype="bf16", B=512,
                                init_state=True, steps=100,
                                note="decode: 512 sequences x 96 heads, fp32 state, 100 steps"),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def cu_seqlens_of(lengths, device="cpu") -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def _fill_token_major(n_tokens, H, dtype, device, gen, dk=DK, dv=DV):
    qd = torch.empty(n_tokens, H, dk, dtype=dtype, device=device)
    kd = torch.empty(n_tokens, H, dk, dtype=dtype, device=device)
    vd = torch.empty(n_tokens, H, dv, dtype=dtype, device=device)
    la = torch.empty(n_tokens, H, dk, dtype=torch.float32, device=device)
    bt = torch.empty(n_tokens, H, dtype=torch.float32, device=device)
    for t0 in range(0, n_tokens, SLICE):
        n = min(SLICE, n_tokens - t0)
        sl = slice(t0, t0 + n)
        x = torch.randn(n, H, dk, generator=gen, device=device)
        qd[sl] = (x / x.norm(dim=-1, keepdim=True)).to(dtype)
        x = torch.randn(n, H, dk, generator=gen, device=device)
        kd[sl] = (x / x.norm(dim=-1, keepdim=True)).to(dtype)
        vd[sl] = torch.randn(n, H, dv, generator=gen, device=device).to(dtype)
        la[sl] = LOG_ALPHA_FLOOR * torch.sigmoid(
            torch.randn(n, H, dk, generator=gen, device=device))
        bt[sl] = torch.sigmoid(torch.randn(n, H, generator=gen, device=device))
        del x
    return qd, kd, vd, la, bt


def prefill_inputs(lengths, H: int, dtype: str = "bf16", init_state: bool = False,
                   device="cpu", seed: int = 0, dk: int = DK, dv: int = DV) -> dict:
    """Packed varlen prefill inputs: q, k, v ``[N, H, d]``, log_alpha ``[N, H, dk]``,
    beta ``[N, H]``, cu_seqlens int32 ``[n_seqs + 1]``, init_state or None."""
    lengths = [int(n) for n in lengths]
    N = sum(lengths)
    gen = torch.Generator(device=device).manual_seed(seed)
    q, k, v, la, bt = _fill_token_major(N, H, torch_dtype(dtype), device, gen, dk, dv)
    s0 = None
    if init_state:
        s0 = STATE_STD * torch.randn(len(lengths), H, dk, dv, generator=gen, device=device)
    return dict(q=q, k=k, v=v, log_alpha=la, beta=bt,
                cu_seqlens=cu_seqlens_of(lengths, device), init_state=s0, lengths=lengths)


def workload_inputs(name: str, device="cpu", seed: int = 0) -> dict:
    w = WORKLOADS[name]
    if w.kind != "prefill":
        raise ValueError(f"{name} is not a prefill workload")
    return prefill_inputs(w.seq_lengths, w.H, w.dtype, w.init_state, device, seed)


def decode_inputs(B: int, H: int, steps: int, dtype: str = "bf16", device="cpu",
                  seed: int = 0, dk: int = DK, dv: int = DV) -> dict:
    """Decode inputs: state ``[B, H, dk, dv]`` fp32 and per-step q, k, v
    ``[steps, B, H, d]``, log_alpha ``[steps, B, H, dk]``, beta ``[steps, B, H]``."""
    gen = torch.Generator(device=device).manual_seed(seed)
    dt = torch_dtype(dtype)
    qs, ks, vs, las, bts = [], [], [], [], []
    for _ in range(steps):
        q, k, v, la, bt = _fill_token_major(B, H, dt, device, gen, dk, dv)
        qs.append(q); ks.append(k); vs.append(v); las.append(la); bts.append(bt)
    state = STATE_STD * torch.randn(B, H, dk, dv, generator=gen, device=device)
    return dict(state=state, q=torch.stack(qs), k=torch.stack(ks), v=torch.stack(vs),
                log_alpha=torch.stack(las), beta=torch.stack(bts))


def layer_inputs(lengths, H: int, dtype: str = "bf16", device="cpu", seed: int = 0,
                 d: int = DK) -> dict:
    """Inputs of the per-token steps around the recurrence for packed sequences of
    the given lengths: projected q, k, v ``[N, H, d]`` ~ N(0, 1) in ``dtype``,
    depthwise convolution weights ``[3, H, d, 4]`` ~ N(0, 0.5^2), decay and beta
    logits ~ N(0, 1), output-gate logits ``[N, H, d]`` ~ N(0, 1) in ``dtype`` and
    an RMSNorm weight ``[d]`` ~ 1 + N(0, 0.1^2)."""
    gen = torch.Generator(device=device).manual_seed(seed)
    dt = torch_dtype(dtype)
    N = int(sum(lengths))

    def randn(*shape, std=1.0):
        return std * torch.randn(*shape, generator=gen, device=device)

    cu = torch.tensor([0] + list(itertools.accumulate(lengths)), dtype=torch.int32,
                      device=device)
    return dict(q_raw=randn(N, H, d).to(dt), k_raw=randn(N, H, d).to(dt),
                v_raw=randn(N, H, d).to(dt), conv_w=randn(3, H, d, 4, std=0.5),
                a_logit=randn(N, H, d), b_logit=randn(N, H), g=randn(N, H, d).to(dt),
                gamma=1.0 + randn(d, std=0.1), cu_seqlens=cu, lengths=list(lengths))
