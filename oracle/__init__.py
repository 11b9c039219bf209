"""KDA oracle: plain fp64 CPU implementation of the KDA recurrence.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA product path never imports it, and the two share no code.

``kda_oracle.c`` holds the token-by-token recurrence (update and read-out of
the "Kimi K3" study notes, section 3-2 "2) Kimi Delta Attention");
``kda_oracle_bwd.c`` its gradient, the chain rule through the same token loop
in reverse; ``affine.py``
holds an independent brute-force form built from explicit transition matrices
(the affine-pair view of "Kimi K3: 架构、训练与系统全景解析" section 7.1, KCP).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_SRC_BWD = os.path.join(_HERE, "kda_oracle_bwd.c")
_LIB_BWD_PATH = os.path.join(_BUILD_DIR, "libkda_oracle_bwd.so")
# Same flags on x86_64 and aarch64: no FMA contraction, IEEE fp64 throughout.
CFLAGS = ["-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None
_lib_bwd = None


def compile_source(src: str, out_path: str) -> str:
    """Compile a C oracle source file into a shared library (used for mutants too)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    cmd = ["gcc", *CFLAGS, src, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``oracle/_build/libkda_oracle.so`` (and the
    gradient, ``kda_oracle_bwd.c``, into ``libkda_oracle_bwd.so``)."""
    with _lock:
        for src, lib in ((_SRC, _LIB_PATH), (_SRC_BWD, _LIB_BWD_PATH)):
            stale = (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)
            if force or stale:
                compile_source(src, lib)
    return _LIB_PATH


def load_bwd_library(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.kda_oracle_chunk_bwd.restype = ctypes.c_int
    lib.kda_oracle_chunk_bwd.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64),
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int64, dp, dp, dp, dp, dp, dp, dp, dp,
                                         ctypes.c_int]
    return lib


def _default_bwd_lib() -> ctypes.CDLL:
    global _lib_bwd
    if _lib_bwd is None:
        build()
        _lib_bwd = load_bwd_library(_LIB_BWD_PATH)
    return _lib_bwd


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    dp = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.kda_oracle_chunk_fwd.restype = ctypes.c_int
    lib.kda_oracle_chunk_fwd.argtypes = [dp, dp, dp, dp, dp, dp, i64p,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int64, dp, dp, ctypes.c_int]
    lib.kda_oracle_decode_step.restype = ctypes.c_int
    lib.kda_oracle_decode_step.argtypes = [dp, dp, dp, dp, dp, dp,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, dp]
    return lib


def load_library(path: str) -> ctypes.CDLL:
    return _bind(ctypes.CDLL(path))


def _default_lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> exact fp64 copy on the host
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def chunk_fwd(q, k, v, log_alpha, beta, init_state=None, cu_seqlens=None,
              n_threads: int | None = None, lib: ctypes.CDLL | None = None):
    """Run the recurrence over packed varlen sequences.

    Shapes: q, k, log_alpha ``[N, H, dk]``; v ``[N, H, dv]``; beta ``[N, H]``;
    init_state ``[n_seqs, H, dk, dv]`` or None; cu_seqlens ``[n_seqs + 1]`` or
    None (one sequence of length N).  Returns ``(out [N, H, dv], final_state
    [n_seqs, H, dk, dv])`` as fp64 numpy arrays.
    """
    lib = lib or _default_lib()
    q, k, v, la, b = (_f64(t) for t in (q, k, v, log_alpha, beta))
    s0 = _f64(init_state)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        cu = np.array([0, N], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    n_seqs = cu.shape[0] - 1
    out = np.zeros((N, H, dv), dtype=np.float64)
    fin = np.zeros((n_seqs, H, dk, dv), dtype=np.float64)
    rc = lib.kda_oracle_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(s0),
                                  _ptr(cu, ctypes.c_int64), n_seqs, H, dk, dv,
                                  _ptr(out), _ptr(fin), int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_chunk_fwd failed with code {rc}")
    return out, fin


def chunk_bwd(q, k, v, log_alpha, beta, init_state, cu_seqlens, d_out, d_final=None,
              n_threads: int | None = None, lib: ctypes.CDLL | None = None):
    """Gradient of ``chunk_fwd`` for a loss with gradients ``d_out`` ``[N, H, dv]``
    (every output) and ``d_final`` ``[n_seqs, H, dk, dv]`` or None (the final
    states).  Returns ``(dq, dk, dv, d_log_alpha, d_beta, d_init_state)`` as fp64
    numpy arrays in the layouts of q, k, v, log_alpha, beta and init_state."""
    lib = lib or _default_bwd_lib()
    q, k, v, la, b, do = (_f64(t) for t in (q, k, v, log_alpha, beta, d_out))
    s0, df = _f64(init_state), _f64(d_final)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        cu = np.array([0, N], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    n_seqs = cu.shape[0] - 1
    dq, dkk = np.zeros((N, H, dk)), np.zeros((N, H, dk))
    dvv, dla, db = np.zeros((N, H, dv)), np.zeros((N, H, dk)), np.zeros((N, H))
    ds0 = np.zeros((n_seqs, H, dk, dv))
    rc = lib.kda_oracle_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(s0),
                                  _ptr(cu, ctypes.c_int64), n_seqs, H, dk, dv, _ptr(do), _ptr(df),
                                  _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dla), _ptr(db), _ptr(ds0),
                                  int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_chunk_bwd failed with code {rc}")
    return dq, dkk, dvv, dla, db, ds0


def decode_step(state, q, k, v, log_alpha, beta, lib: ctypes.CDLL | None = None):
    """One in-place decode step.  ``state`` must be a C-contiguous fp64 numpy
    array ``[B, H, dk, dv]``; it is updated in place.  Returns out ``[B, H, dv]``."""
    lib = lib or _default_lib()
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64
            and state.flags["C_CONTIGUOUS"]):
        raise TypeError("state must be a C-contiguous float64 numpy array")
    q, k, v, la, b = (_f64(t) for t in (q, k, v, log_alpha, beta))
    B, H, dk, dv = state.shape
    out = np.zeros((B, H, dv), dtype=np.float64)
    rc = lib.kda_oracle_decode_step(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b),
                                    B, H, dk, dv, _ptr(out))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_decode_step failed with code {rc}")
    return out


def decode_replay(state, q, k, v, log_alpha, beta, n_accept, lib: ctypes.CDLL | None = None):
    """Replay of accepted draft tokens after speculative-decode verification
    ("Kimi K3: 架构、训练与系统全景解析", KDA state replay under speculative
    decoding: only the accepted prefix of the cached per-token inputs is replayed
    and only the final state is kept).  For every sequence b, the decode step is
    applied to tokens t = 0 .. n_b - 1 in order, n_b = n_accept[b] clamped to
    [0, T].  ``state`` (C-contiguous fp64 ``[B, H, dk, dv]``) is updated in place;
    q, k ``[B, T, H, dk]``, v ``[B, T, H, dv]``, log_alpha ``[B, T, H, dk]``,
    beta ``[B, T, H]``.  Returns out ``[B, T, H, dv]``, zero where t >= n_b."""
    q, k, v, la, b = (_f64(t) for t in (q, k, v, log_alpha, beta))
    B, T, H, _ = q.shape
    dv = v.shape[3]
    n = np.clip(np.asarray(n_accept, dtype=np.int64).reshape(B), 0, T)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    for t in range(T):
        sel = np.nonzero(n > t)[0]
        if sel.size == 0:
            break
        sub = np.ascontiguousarray(state[sel])
        out[sel, t] = decode_step(sub, q[sel, t], k[sel, t], v[sel, t], la[sel, t], b[sel, t],
                                  lib=lib)
        state[sel] = sub
    return out
