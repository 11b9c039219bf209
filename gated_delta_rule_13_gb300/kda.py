"""Thin Python binding of libkda (argument marshalling only).

Every function here has the name of the C entry point it wraps (include/kda.h)
and does nothing but check tensor shapes, dtypes and devices, allocate outputs
when the caller did not pass them, and forward raw device pointers plus the
current CUDA stream.  All arithmetic runs in the CUDA kernels of libkda.so.
There is no fallback: if the library is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_ERR_TIMEOUT = 5
KDA_F32 = 0
KDA_BF16 = 1
HEAD_DIM = 128

# Symbols declared in include/kda.h.
EXPORTED = ("kda_status_string", "kda_version", "kda_chunk_fwd_workspace_size",
            "kda_chunk_fwd", "kda_chunk_fwd_sched", "kda_read_device_status",
            "kda_read_device_status_detail", "kda_test_arm_timeout", "kda_decode_step",
            "kda_chunk_fwd_noalloc", "kda_noalloc_read_status", "kda_decode_replay",
            "kda_prep_fwd", "kda_prep_fwd_state", "kda_layer_replay", "kda_post_fwd",
            "kda_read_chunk_stats", "kda_chunk_fwd_transitions", "kda_state_combine",
            "kda_chunk_bwd", "kda_chunk_bwd_workspace_size", "kda_chunk_bwd_sched",
            "kda_chunk_bwd_workspace_size_sched")

_lib = None


class KDAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (code {code})")


def library_path() -> str:
    return _build.LIB_PATH


def library() -> ctypes.CDLL:
    """Load libkda.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"libkda.so is not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_version.restype = ctypes.c_int
        lib.kda_version.argtypes = []
        lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_int
        lib.kda_chunk_fwd_workspace_size.argtypes = [i32, i64, i32, i32, i32, ctypes.c_int,
                                                     ctypes.POINTER(sz)]
        lib.kda_chunk_fwd.restype = ctypes.c_int
        lib.kda_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                      ctypes.c_int, vp, vp, vp, sz, vp]
        lib.kda_chunk_fwd_sched.restype = ctypes.c_int
        lib.kda_chunk_fwd_sched.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                            ctypes.c_int, vp, vp, i32, i32, vp, sz, vp]
        lib.kda_read_device_status.restype = ctypes.c_int
        lib.kda_read_device_status.argtypes = [vp, vp, ctypes.c_int, ctypes.POINTER(i32)]
        lib.kda_read_device_status_detail.restype = ctypes.c_int
        lib.kda_read_device_status_detail.argtypes = [vp, vp, ctypes.c_int, ctypes.POINTER(i32)]
        lib.kda_test_arm_timeout.restype = ctypes.c_int
        lib.kda_test_arm_timeout.argtypes = [vp, i32, i32, ctypes.c_uint32, vp]
        lib.kda_noalloc_read_status.restype = ctypes.c_int
        lib.kda_noalloc_read_status.argtypes = [vp, ctypes.c_int, ctypes.POINTER(i32)]
        lib.kda_read_chunk_stats.restype = ctypes.c_int
        lib.kda_read_chunk_stats.argtypes = [vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.kda_chunk_fwd_transitions.restype = ctypes.c_int
        lib.kda_chunk_fwd_transitions.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                                  ctypes.c_int, vp, vp, vp, sz, vp]
        lib.kda_state_combine.restype = ctypes.c_int
        lib.kda_state_combine.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
        lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.kda_chunk_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                              ctypes.c_int, vp, vp, vp]
        lib.kda_decode_replay.restype = ctypes.c_int
        lib.kda_decode_replay.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                          ctypes.c_int, vp, vp]
        lib.kda_prep_fwd.restype = ctypes.c_int
        lib.kda_prep_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                     ctypes.c_int, vp, vp, vp, vp, vp, vp]
        lib.kda_prep_fwd_state.restype = ctypes.c_int
        lib.kda_prep_fwd_state.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                           ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.kda_layer_replay.restype = ctypes.c_int
        lib.kda_layer_replay.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                         i32, i32, ctypes.c_int, vp, vp]
        lib.kda_chunk_bwd.restype = ctypes.c_int
        lib.kda_chunk_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                      ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_chunk_bwd_workspace_size.restype = ctypes.c_int
        lib.kda_chunk_bwd_workspace_size.argtypes = [i32, i64, i32, i32, i32, ctypes.c_int,
                                                     ctypes.POINTER(sz)]
        lib.kda_chunk_bwd_sched.restype = ctypes.c_int
        lib.kda_chunk_bwd_sched.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                            ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                            vp, sz, vp]
        lib.kda_chunk_bwd_workspace_size_sched.restype = ctypes.c_int
        lib.kda_chunk_bwd_workspace_size_sched.argtypes = [i32, i64, i32, i32, i32, ctypes.c_int,
                                                           i32, ctypes.POINTER(sz)]
        lib.kda_post_fwd.restype = ctypes.c_int
        lib.kda_post_fwd.argtypes = [vp, vp, vp, i64, i32, i32, ctypes.c_int, vp, vp]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                        ctypes.c_int, vp, vp]
        _lib = lib
    return _lib


def status_string(code: int) -> str:
    return library().kda_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != KDA_OK:
        raise KDAError(rc, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(name, t, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def kda_version() -> int:
    return library().kda_version()


def kda_chunk_fwd_workspace_size(n_seqs: int, n_tokens: int, H: int, dk: int = HEAD_DIM,
                                 dv: int = HEAD_DIM, dtype: int = KDA_BF16) -> int:
    out = ctypes.c_size_t(0)
    _check(library().kda_chunk_fwd_workspace_size(n_seqs, n_tokens, H, dk, dv, dtype,
                                                  ctypes.byref(out)),
           "kda_chunk_fwd_workspace_size")
    return out.value


def kda_chunk_fwd(q, k, v, log_alpha, beta, init_state=None, cu_seqlens=None, *, out=None,
                  final_state=None, workspace=None, output_final_state=True, max_split=None,
                  max_helpers=None, stream=None):
    """Chunked KDA prefill.  q, k ``[N, H, 128]`` and v ``[N, H, 128]`` (bf16 or
    fp32, same dtype); log_alpha ``[N, H, 128]`` fp32; beta ``[N, H]`` fp32;
    init_state ``[n_seqs, H, 128, 128]`` fp32 or None; cu_seqlens int32
    ``[n_seqs + 1]`` (CUDA or CPU tensor) or None for one sequence.
    ``max_split`` / ``max_helpers`` cap the schedule (``kda_chunk_fwd_sched``;
    None: the library's choice, 0: off).
    Returns ``(out, final_state)`` (final_state None if not requested)."""
    _need_cuda("q", q)
    N, H, dk = q.shape
    dt = q.dtype
    _need_cuda("k", k, dt, (N, H, dk))
    _need_cuda("v", v, dt)
    if v.shape[:2] != (N, H):
        raise ValueError("v must be [N, H, dv]")
    dv = v.shape[2]
    _need_cuda("log_alpha", log_alpha, torch.float32, (N, H, dk))
    _need_cuda("beta", beta, torch.float32, (N, H))
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32, device=q.device)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise TypeError("cu_seqlens must be a contiguous 1-D int32 tensor")
    n_seqs = cu_seqlens.shape[0] - 1
    if init_state is not None:
        _need_cuda("init_state", init_state, torch.float32, (n_seqs, H, dk, dv))
    if out is None:
        out = torch.empty(N, H, dv, dtype=dt, device=q.device)
    _need_cuda("out", out, dt, (N, H, dv))
    if final_state is None and output_final_state:
        final_state = torch.empty(n_seqs, H, dk, dv, dtype=torch.float32, device=q.device)
    if final_state is not None:
        _need_cuda("final_state", final_state, torch.float32, (n_seqs, H, dk, dv))
    code = _dtype_code(q)
    ws_bytes = kda_chunk_fwd_workspace_size(n_seqs, N, H, dk, dv, code)
    if workspace is None:
        # the library clears what it reads (status block, helper header) itself
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _need_cuda("workspace", workspace)
    ws_args = (_ptr(workspace), workspace.numel() * workspace.element_size(),
               _stream_handle(stream))
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(init_state),
            _ptr(cu_seqlens), n_seqs, N, H, dk, dv, code, _ptr(out), _ptr(final_state))
    if max_split is None and max_helpers is None:
        _check(library().kda_chunk_fwd(*args, *ws_args), "kda_chunk_fwd")
    else:
        caps = (-1 if max_split is None else int(max_split),
                -1 if max_helpers is None else int(max_helpers))
        _check(library().kda_chunk_fwd_sched(*args, *caps, *ws_args), "kda_chunk_fwd_sched")
    return out, final_state


def kda_chunk_bwd_workspace_size(n_seqs: int, n_tokens: int, H: int, dk: int = HEAD_DIM,
                                 dv: int = HEAD_DIM, dtype: int = KDA_BF16,
                                 ckpt_every: int = 0) -> int:
    """Workspace bytes of the backward pass (``ckpt_every`` 0: the library's
    checkpoint interval)."""
    out = ctypes.c_size_t(0)
    _check(library().kda_chunk_bwd_workspace_size_sched(n_seqs, n_tokens, H, dk, dv, dtype,
                                                        int(ckpt_every), ctypes.byref(out)),
           "kda_chunk_bwd_workspace_size_sched")
    return out.value


def kda_chunk_bwd(q, k, v, log_alpha, beta, init_state, cu_seqlens, d_out, d_final_state=None,
                  *, workspace=None, want_d_init=True, ckpt_every=None, stream=None):
    """Gradients of ``kda_chunk_fwd`` for output gradients ``d_out`` ``[N, H, 128]``
    (dtype of q) and final-state gradients ``d_final_state`` (or None).  Returns
    ``(dq, dk, dv, d_log_alpha, d_beta, d_init_state)`` in the layouts of the
    inputs (d_init_state None unless requested).  ``ckpt_every`` (a power of two
    in [4, 1024]) picks the interval of stored states through
    ``kda_chunk_bwd_sched``; None leaves it to the library."""
    _need_cuda("q", q)
    N, H, dk = q.shape
    dt = q.dtype
    _need_cuda("k", k, dt, (N, H, dk))
    _need_cuda("v", v, dt)
    dv = v.shape[2]
    _need_cuda("log_alpha", log_alpha, torch.float32, (N, H, dk))
    _need_cuda("beta", beta, torch.float32, (N, H))
    _need_cuda("d_out", d_out, dt, (N, H, dv))
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32, device=q.device)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise TypeError("cu_seqlens must be a contiguous 1-D int32 tensor")
    n_seqs = cu_seqlens.shape[0] - 1
    if init_state is not None:
        _need_cuda("init_state", init_state, torch.float32, (n_seqs, H, dk, dv))
    if d_final_state is not None:
        _need_cuda("d_final_state", d_final_state, torch.float32, (n_seqs, H, dk, dv))
    dq, dkk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dla = torch.empty_like(log_alpha)
    db = torch.empty_like(beta)
    ds0 = (torch.empty(n_seqs, H, dk, dv, dtype=torch.float32, device=q.device)
           if want_d_init else None)
    code = _dtype_code(q)
    every = 0 if ckpt_every is None else int(ckpt_every)
    if workspace is None:
        workspace = torch.empty(kda_chunk_bwd_workspace_size(n_seqs, N, H, dk, dv, code, every),
                                dtype=torch.uint8, device=q.device)
    _need_cuda("workspace", workspace)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(init_state),
            _ptr(cu_seqlens), n_seqs, N, H, dk, dv, code, _ptr(d_out), _ptr(d_final_state),
            _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dla), _ptr(db), _ptr(ds0))
    ws_args = (_ptr(workspace), workspace.numel() * workspace.element_size(),
               _stream_handle(stream))
    if ckpt_every is None:
        _check(library().kda_chunk_bwd(*args, *ws_args), "kda_chunk_bwd")
    else:
        _check(library().kda_chunk_bwd_sched(*args, every, *ws_args), "kda_chunk_bwd_sched")
    return dq, dkk, dvv, dla, db, ds0


def kda_chunk_fwd_transitions(q, k, v, log_alpha, beta, cu_seqlens=None, *, workspace=None,
                              stream=None):
    """The affine state map of every packed sequence (bf16): returns
    ``(state_b, state_m)``, each ``[n_seqs, H, 128, 128]`` fp32, with the
    sequence mapping a start state S to ``state_m @ S + state_b``."""
    _need_cuda("q", q)
    N, H, dk = q.shape
    dt = q.dtype
    _need_cuda("k", k, dt, (N, H, dk))
    _need_cuda("v", v, dt, (N, H, dk))
    _need_cuda("log_alpha", log_alpha, torch.float32, (N, H, dk))
    _need_cuda("beta", beta, torch.float32, (N, H))
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32, device=q.device)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise TypeError("cu_seqlens must be a contiguous 1-D int32 tensor")
    n_seqs = cu_seqlens.shape[0] - 1
    b = torch.empty(n_seqs, H, dk, dk, dtype=torch.float32, device=q.device)
    m = torch.empty_like(b)
    code = _dtype_code(q)
    if workspace is None:
        workspace = torch.empty(kda_chunk_fwd_workspace_size(n_seqs, N, H, dk, dk, code),
                                dtype=torch.uint8, device=q.device)
    _need_cuda("workspace", workspace)
    rc = library().kda_chunk_fwd_transitions(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(cu_seqlens), n_seqs, N, H,
        dk, dk, code, _ptr(b), _ptr(m), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "kda_chunk_fwd_transitions")
    return b, m


def kda_state_combine(state_b, state_m, n_segments: int, init_state=None, *, starts=True,
                      end=True, stream=None):
    """Composes per-segment affine state maps: ``state_b``, ``state_m`` are
    ``[n_seqs * n_segments, H, 128, 128]`` (segment j of sequence s at index
    ``s * n_segments + j``).  Returns ``(start_states, end_state)``: the state
    each segment starts from, and each sequence's composed final state (either
    None if not requested)."""
    _need_cuda("state_b", state_b, torch.float32)
    n_tot, H, dk, dv = state_b.shape
    _need_cuda("state_m", state_m, torch.float32, (n_tot, H, dk, dv))
    if n_segments < 1 or n_tot % n_segments:
        raise ValueError("the number of pairs must be a multiple of n_segments")
    n_seqs = n_tot // n_segments
    if init_state is not None:
        _need_cuda("init_state", init_state, torch.float32, (n_seqs, H, dk, dv))
    st = torch.empty_like(state_b) if starts else None
    en = torch.empty(n_seqs, H, dk, dv, dtype=torch.float32, device=state_b.device) if end else None
    _check(library().kda_state_combine(_ptr(init_state), _ptr(state_b), _ptr(state_m), n_seqs,
                                       n_segments, H, dk, dv, _ptr(st), _ptr(en),
                                       _stream_handle(stream)),
           "kda_state_combine")
    return st, en


def _piece_bounds(n_tokens: int, piece_tokens: int, min_tail: int = 1024) -> list:
    """Token bounds of the pieces: ``piece_tokens`` each, except that the last
    full piece is cut in halves down to ``min_tail`` tokens (multiples of the
    64-token chunk), so that the prefill and output copy left after the last
    input copy are short."""
    bounds, p0 = [0], 0
    while n_tokens - p0 > piece_tokens:
        p0 += piece_tokens
        bounds.append(p0)
    rest = n_tokens - p0
    while rest > max(min_tail, 64) and rest // 2 >= 64:
        half = (rest // 2 + 63) // 64 * 64
        p0 += half
        bounds.append(p0)
        rest -= half
    if bounds[-1] != n_tokens:
        bounds.append(n_tokens)
    return bounds


def kda_chunk_fwd_host(q, k, v, log_alpha, beta, init_state=None, *, out=None,
                       final_state=None, piece_tokens: int = 4096, device=None,
                       max_split=None, max_helpers=None):
    """Prefill of ONE sequence whose inputs are in host memory (pinned for the
    copies to overlap): the tokens go through in pieces of ``piece_tokens`` (a
    multiple of the 64-token chunk; the last one cut in halves down to 1024
    tokens), each piece's host-to-device copy overlapping the previous piece's
    prefill and the device-to-host copy of its outputs.
    Piece i starts from piece i-1's final state (fp32, exact), so the results
    are those of one kda_chunk_fwd call (with the same schedule caps, which
    every piece gets).  Returns host ``(out, final_state)``."""
    if piece_tokens <= 0 or piece_tokens % 64:
        raise ValueError("piece_tokens must be a positive multiple of 64")
    device = torch.device(device or "cuda")
    N, H, dk = q.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty(N, H, dv, dtype=q.dtype).pin_memory()
    if final_state is None:
        final_state = torch.empty(1, H, dk, dv, dtype=torch.float32).pin_memory()
    if N == 0:
        final_state.copy_(init_state if init_state is not None else torch.zeros_like(final_state))
        return out, final_state
    names = ("q", "k", "v", "log_alpha", "beta")
    host = dict(zip(names, (q, k, v, log_alpha, beta)))
    dev = {n: torch.empty(t.shape, dtype=t.dtype, device=device) for n, t in host.items()}
    d_out = torch.empty(N, H, dv, dtype=q.dtype, device=device)
    states = [torch.empty(1, H, dk, dv, dtype=torch.float32, device=device) for _ in range(2)]
    s0 = init_state.to(device, non_blocking=True) if init_state is not None else None
    compute = torch.cuda.current_stream(device)
    copy_in, copy_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ws = torch.empty(kda_chunk_fwd_workspace_size(1, piece_tokens, H, dk, dv, _dtype_code(q)),
                     dtype=torch.uint8, device=device)
    cu = {}
    bounds = _piece_bounds(N, piece_tokens)
    copied = []
    copy_in.wait_stream(compute)  # the device buffers are free
    for p0, p1 in zip(bounds[:-1], bounds[1:]):
        with torch.cuda.stream(copy_in):
            for n in names:
                dev[n][p0:p1].copy_(host[n][p0:p1], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(copy_in)
        copied.append(ev)
    done = []
    for i, (p0, p1) in enumerate(zip(bounds[:-1], bounds[1:])):
        compute.wait_event(copied[i])
        n_tok = p1 - p0
        if n_tok not in cu:
            cu[n_tok] = torch.tensor([0, n_tok], dtype=torch.int32, device=device)
        last = p1 == N
        kda_chunk_fwd(dev["q"][p0:p1], dev["k"][p0:p1], dev["v"][p0:p1],
                      dev["log_alpha"][p0:p1], dev["beta"][p0:p1],
                      s0 if i == 0 else states[(i - 1) & 1], cu[n_tok], out=d_out[p0:p1],
                      final_state=states[i & 1], workspace=ws, max_split=max_split,
                      max_helpers=max_helpers)
        ev = torch.cuda.Event()
        ev.record(compute)
        done.append(ev)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(ev)
            out[p0:p1].copy_(d_out[p0:p1], non_blocking=True)
            if last:
                final_state.copy_(states[i & 1], non_blocking=True)
    compute.wait_stream(copy_out)
    return out, final_state


def kda_chunk_fwd_noalloc(q, k, v, log_alpha, beta, init_state=None, cu_seqlens=None, *,
                          out=None, final_state=None, output_final_state=True, stream=None):
    """kda_chunk_fwd without a workspace: the library's fixed device scratch is
    used instead (at most 4095 sequences; concurrent calls on different streams
    race on that scratch).  Same arguments and results as ``kda_chunk_fwd``."""
    _need_cuda("q", q)
    N, H, dk = q.shape
    dt = q.dtype
    _need_cuda("k", k, dt, (N, H, dk))
    _need_cuda("v", v, dt)
    dv = v.shape[2]
    _need_cuda("log_alpha", log_alpha, torch.float32, (N, H, dk))
    _need_cuda("beta", beta, torch.float32, (N, H))
    if cu_seqlens is None:
        # host memory: the library copies it into its own array (no device allocation)
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32)
    n_seqs = cu_seqlens.shape[0] - 1
    if init_state is not None:
        _need_cuda("init_state", init_state, torch.float32, (n_seqs, H, dk, dv))
    if out is None:
        out = torch.empty(N, H, dv, dtype=dt, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(n_seqs, H, dk, dv, dtype=torch.float32, device=q.device)
    rc = library().kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                         _ptr(init_state), _ptr(cu_seqlens), n_seqs, N, H, dk, dv,
                                         _dtype_code(q), _ptr(out), _ptr(final_state),
                                         _stream_handle(stream))
    _check(rc, "kda_chunk_fwd_noalloc")
    return out, final_state


def kda_read_chunk_stats(workspace, stream=None):
    """Synchronise the stream and return (packages published by helper CTAs,
    packages chain CTAs used) of the last kda_chunk_fwd on this workspace."""
    _need_cuda("workspace", workspace)
    pub, con = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(library().kda_read_chunk_stats(_ptr(workspace), _stream_handle(stream),
                                          ctypes.byref(pub), ctypes.byref(con)),
           "kda_read_chunk_stats")
    return pub.value, con.value


def kda_read_device_status(workspace, stream=None, clear: bool = True) -> int:
    """Synchronise the stream and return the device status a kda_chunk_fwd or
    kda_chunk_bwd workspace recorded (KDA_OK or a kda_status code)."""
    _need_cuda("workspace", workspace)
    st = ctypes.c_int32(0)
    _check(library().kda_read_device_status(_ptr(workspace), _stream_handle(stream),
                                            1 if clear else 0, ctypes.byref(st)),
           "kda_read_device_status")
    return st.value


def kda_read_device_status_detail(workspace, stream=None, clear: bool = True):
    """As ``kda_read_device_status``, returning ``(code, detail, chain, chunk)``."""
    _need_cuda("workspace", workspace)
    d = (ctypes.c_int32 * 4)()
    _check(library().kda_read_device_status_detail(_ptr(workspace), _stream_handle(stream),
                                                   1 if clear else 0, d),
           "kda_read_device_status_detail")
    return tuple(int(x) for x in d)


def kda_noalloc_read_status(stream=None, clear: bool = True) -> int:
    """Device status recorded by the last ``kda_chunk_fwd_noalloc`` calls on the
    current device (the library's fixed array; allocates nothing)."""
    st = ctypes.c_int32(0)
    _check(library().kda_noalloc_read_status(_stream_handle(stream), 1 if clear else 0,
                                             ctypes.byref(st)),
           "kda_noalloc_read_status")
    return st.value


def kda_test_arm_timeout(workspace, chain: int, chunk: int, wait_us: int = 1000, stream=None):
    """Test control of the bounded waits (see include/kda.h): the next bf16
    plain-schedule ``kda_chunk_fwd`` on ``workspace`` times out in chain
    ``chain`` at chunk ``chunk``; ``chain < 0`` disarms."""
    _need_cuda("workspace", workspace)
    _check(library().kda_test_arm_timeout(_ptr(workspace), int(chain), int(chunk), int(wait_us),
                                          _stream_handle(stream)),
           "kda_test_arm_timeout")


def kda_decode_step(state, q, k, v, log_alpha, beta, *, out=None, stream=None):
    """One in-place decode step.  state ``[B, H, 128, 128]`` fp32 (updated in
    place); q, k ``[B, H, 128]``, v ``[B, H, 128]`` (bf16 or fp32); log_alpha
    ``[B, H, 128]`` fp32; beta ``[B, H]`` fp32.  Returns out ``[B, H, 128]``."""
    _need_cuda("state", state, torch.float32)
    B, H, dk, dv = state.shape
    _need_cuda("q", q, None, (B, H, dk))
    dt = q.dtype
    _need_cuda("k", k, dt, (B, H, dk))
    _need_cuda("v", v, dt, (B, H, dv))
    _need_cuda("log_alpha", log_alpha, torch.float32, (B, H, dk))
    _need_cuda("beta", beta, torch.float32, (B, H))
    if out is None:
        out = torch.empty(B, H, dv, dtype=dt, device=q.device)
    _need_cuda("out", out, dt, (B, H, dv))
    rc = library().kda_decode_step(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                   _ptr(beta), B, H, dk, dv, _dtype_code(q), _ptr(out),
                                   _stream_handle(stream))
    _check(rc, "kda_decode_step")
    return out


def kda_decode_replay(state, q, k, v, log_alpha, beta, n_accept, *, out=None,
                      output=True, stream=None):
    """Replays the accepted draft tokens of a speculative decode step in place.
    state ``[B, H, 128, 128]`` fp32 (updated in place); q, k, v ``[B, T, H, 128]``
    (bf16 or fp32); log_alpha ``[B, T, H, 128]`` fp32; beta ``[B, T, H]`` fp32;
    n_accept int32 CUDA tensor ``[B]`` (clamped to [0, T] on the device).
    Returns out ``[B, T, H, 128]`` (rows t >= n_accept[b] untouched) or None
    when ``output`` is false."""
    _need_cuda("state", state, torch.float32)
    B, H, dk, dv = state.shape
    _need_cuda("q", q)
    if q.dim() != 4 or q.shape[0] != B or q.shape[2] != H or q.shape[3] != dk:
        raise ValueError("q must be [B, T, H, dk]")
    T = q.shape[1]
    dt = q.dtype
    _need_cuda("k", k, dt, (B, T, H, dk))
    _need_cuda("v", v, dt, (B, T, H, dv))
    _need_cuda("log_alpha", log_alpha, torch.float32, (B, T, H, dk))
    _need_cuda("beta", beta, torch.float32, (B, T, H))
    _need_cuda("n_accept", n_accept, torch.int32, (B,))
    if out is None and output:
        out = torch.empty(B, T, H, dv, dtype=dt, device=q.device)
    if out is not None:
        _need_cuda("out", out, dt, (B, T, H, dv))
    rc = library().kda_decode_replay(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                     _ptr(beta), _ptr(n_accept), B, T, H, dk, dv,
                                     _dtype_code(q), _ptr(out), _stream_handle(stream))
    _check(rc, "kda_decode_replay")
    return out


def kda_prep_fwd(q_raw, k_raw, v_raw, conv_w, a_logit, b_logit, cu_seqlens, *, stream=None):
    """Short convolution + Swish (+ L2Norm for q, k) and the beta / decay gates
    before the recurrence.  q_raw, k_raw, v_raw ``[N, H, 128]`` (bf16 or fp32);
    conv_w ``[3, H, 128, 4]`` fp32; a_logit ``[N, H, 128]`` and b_logit ``[N, H]``
    fp32; cu_seqlens int32 CUDA tensor ``[n_seqs + 1]``.
    Returns ``(q, k, v, log_alpha, beta)`` ready for ``kda_chunk_fwd``."""
    _need_cuda("q_raw", q_raw)
    N, H, dk = q_raw.shape
    dt = q_raw.dtype
    _need_cuda("k_raw", k_raw, dt, (N, H, dk))
    _need_cuda("v_raw", v_raw, dt, (N, H, dk))
    _need_cuda("conv_w", conv_w, torch.float32, (3, H, dk, 4))
    _need_cuda("a_logit", a_logit, torch.float32, (N, H, dk))
    _need_cuda("b_logit", b_logit, torch.float32, (N, H))
    _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    n_seqs = cu_seqlens.shape[0] - 1
    q, k, v = (torch.empty_like(q_raw) for _ in range(3))
    log_alpha = torch.empty_like(a_logit)
    beta = torch.empty_like(b_logit)
    rc = library().kda_prep_fwd(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(conv_w),
                                _ptr(a_logit), _ptr(b_logit), _ptr(cu_seqlens), n_seqs, N, H,
                                dk, dk, _dtype_code(q_raw), _ptr(q), _ptr(k), _ptr(v),
                                _ptr(log_alpha), _ptr(beta), _stream_handle(stream))
    _check(rc, "kda_prep_fwd")
    return q, k, v, log_alpha, beta


def kda_prep_fwd_state(q_raw, k_raw, v_raw, conv_w, a_logit, b_logit, cu_seqlens,
                       conv_state_in=None, conv_state_out=None, *, stream=None):
    """``kda_prep_fwd`` continuing each packed sequence from a carried
    convolution window: ``conv_state_in`` / ``conv_state_out``
    ``[n_seqs, 3, 3, H, 128]`` in the dtype of the raw inputs ((q, k, v) x the
    three raw rows before the sequence's next token, oldest first), either None
    (zeros / not written), possibly the same tensor (updated in place).
    Returns ``(q, k, v, log_alpha, beta)``."""
    _need_cuda("q_raw", q_raw)
    N, H, dk = q_raw.shape
    dt = q_raw.dtype
    _need_cuda("k_raw", k_raw, dt, (N, H, dk))
    _need_cuda("v_raw", v_raw, dt, (N, H, dk))
    _need_cuda("conv_w", conv_w, torch.float32, (3, H, dk, 4))
    _need_cuda("a_logit", a_logit, torch.float32, (N, H, dk))
    _need_cuda("b_logit", b_logit, torch.float32, (N, H))
    _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    n_seqs = cu_seqlens.shape[0] - 1
    for name, w in (("conv_state_in", conv_state_in), ("conv_state_out", conv_state_out)):
        if w is not None:
            _need_cuda(name, w, dt, (n_seqs, 3, 3, H, dk))
    q, k, v = (torch.empty_like(q_raw) for _ in range(3))
    log_alpha = torch.empty_like(a_logit)
    beta = torch.empty_like(b_logit)
    rc = library().kda_prep_fwd_state(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(conv_w),
                                      _ptr(a_logit), _ptr(b_logit), _ptr(cu_seqlens), n_seqs, N,
                                      H, dk, dk, _dtype_code(q_raw), _ptr(conv_state_in),
                                      _ptr(conv_state_out), _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(log_alpha), _ptr(beta), _stream_handle(stream))
    _check(rc, "kda_prep_fwd_state")
    return q, k, v, log_alpha, beta


def kda_layer_replay(state, conv_state, q_raw, k_raw, v_raw, a_logit, b_logit, g, conv_w, gamma,
                     n_accept, *, out=None, output=True, stream=None):
    """The layer between its projections replayed over the accepted draft
    tokens, in one kernel: state ``[B, H, 128, 128]`` fp32 and conv_state
    ``[B, 3, 3, H, 128]`` (the raw inputs' dtype) are updated in place; q_raw,
    k_raw, v_raw, g ``[B, T, H, 128]``; a_logit ``[B, T, H, 128]`` and b_logit
    ``[B, T, H]`` fp32; conv_w ``[3, H, 128, 4]`` and gamma ``[128]`` fp32;
    n_accept int32 CUDA ``[B]``.  Returns the gated, normalised layer output
    ``[B, T, H, 128]`` (rows t >= n_accept[b] untouched) or None."""
    _need_cuda("state", state, torch.float32)
    B, H, dk, dv = state.shape
    _need_cuda("q_raw", q_raw)
    if q_raw.dim() != 4 or q_raw.shape[0] != B or q_raw.shape[2] != H or q_raw.shape[3] != dk:
        raise ValueError("q_raw must be [B, T, H, 128]")
    T = q_raw.shape[1]
    dt = q_raw.dtype
    for name, t in (("k_raw", k_raw), ("v_raw", v_raw), ("g", g)):
        _need_cuda(name, t, dt, (B, T, H, dk))
    _need_cuda("a_logit", a_logit, torch.float32, (B, T, H, dk))
    _need_cuda("b_logit", b_logit, torch.float32, (B, T, H))
    _need_cuda("conv_state", conv_state, dt, (B, 3, 3, H, dk))
    _need_cuda("conv_w", conv_w, torch.float32, (3, H, dk, 4))
    _need_cuda("gamma", gamma, torch.float32, (dk,))
    _need_cuda("n_accept", n_accept, torch.int32, (B,))
    if out is None and output:
        out = torch.empty(B, T, H, dv, dtype=dt, device=q_raw.device)
    if out is not None:
        _need_cuda("out", out, dt, (B, T, H, dv))
    rc = library().kda_layer_replay(_ptr(state), _ptr(conv_state), _ptr(q_raw), _ptr(k_raw),
                                    _ptr(v_raw), _ptr(a_logit), _ptr(b_logit), _ptr(g),
                                    _ptr(conv_w), _ptr(gamma), _ptr(n_accept), B, T, H, dk, dv,
                                    _dtype_code(q_raw), _ptr(out), _stream_handle(stream))
    _check(rc, "kda_layer_replay")
    return out


def kda_post_fwd(o, g, gamma, *, out=None, stream=None):
    """Head-wise RMSNorm of the recurrent output times the sigmoid output gate.
    o, g ``[N, H, 128]`` (same dtype); gamma ``[128]`` fp32.  Returns out (may be o)."""
    _need_cuda("o", o)
    N, H, dv = o.shape
    _need_cuda("g", g, o.dtype, (N, H, dv))
    _need_cuda("gamma", gamma, torch.float32, (dv,))
    if out is None:
        out = torch.empty_like(o)
    _need_cuda("out", out, o.dtype, (N, H, dv))
    rc = library().kda_post_fwd(_ptr(o), _ptr(g), _ptr(gamma), N, H, dv, _dtype_code(o), _ptr(out),
                                _stream_handle(stream))
    _check(rc, "kda_post_fwd")
    return out
