"""Per-phase cycle breakdown of the tensor-core prefill kernel.

Builds a separate copy of libkda with ``-DKDA_PHASE_PROFILE`` (the kernel then
stamps ``clock64()`` at its phase boundaries for chain 0) into
``gated_delta_rule_13_gb300/_build/prof/``, runs one workload twice and prints
the median cycles of every phase over the chunks of chain 0.  The normal library
is not touched.

    python -m gated_delta_rule_13_gb300.phase_profile [workload]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

from . import _build

# Phase boundaries stamped by thread 0 (PHASE_MARK indices 0..8); the last
# interval runs to the next chunk's first stamp.
PHASES = ["wait m2(prev) + sync", "S pass", "wait Gram MMAs", "A/P epilogue + sync",
          "solve (warps 0-3)", "wait Delta MMAs", "Delta pass", "scan + build (next)",
          "loop"]
# Extra stamps, printed as offsets from the chunk's first stamp.  Slots 9, 14
# and 15 belong to the build of this chunk, which runs in the previous iteration.
EXTRA = {9: "t0: build of this chunk: decay prefix done", 14: "t0: build: q/k tile arrived",
         15: "t0: build done (before arrive)", 10: "t0: A/P done (before sync)",
         11: "t0: diagonal blocks done", 12: "t0: level 16->32 done", 13: "t0: level 32->64 X stored",
         16: "w4: flush start", 17: "w4: flush done", 18: "w4: O+Y MMAs done",
         19: "w4: -Y pass done", 24: "mma: operands built, Gram issue",
         25: "mma: O+Y issue", 26: "mma: T' ready", 27: "mma: -Y ready",
         28: "mma: Delta ready, M2 issue", 29: "mma: Gram committed", 30: "mma: O+Y committed",
         31: "mma: M2 committed", 32: "w3: Gram waited", 33: "w3: A/P done (before sync)",
         34: "w3: solve done", 35: "w3: A/P TMEM load returned", 36: "w3: A/P first block done",
         37: "w3: S pass first TMEM load returned", 48: "w12: flush start",
         49: "w12: flush done", 40: "w7: A/P done (before sync)", 41: "w7: -Y pass done",
         42: "w7: build done (before arrive)", 51: "mma: next chunk planned",
         52: "t0: plan seen"}
SLOTS = 64


def build_profiling_library() -> str:
    out = os.path.join(_build.OBJ_DIR, "prof")
    os.makedirs(out, exist_ok=True)
    objs = []
    for src in _build.sources():
        obj = os.path.join(out, os.path.basename(src)[:-3] + ".o")
        subprocess.run([_build.nvcc(), *_build.ARCH, *_build.NVCC_FLAGS, "-DKDA_PHASE_PROFILE",
                        "-c", src, "-o", obj], check=True)
        objs.append(obj)
    lib = os.path.join(out, "libkda_prof.so")
    subprocess.run([_build.nvcc(), *_build.ARCH, "-shared", "-o", lib, *objs, "-cudart",
                    "static"], check=True)
    return lib


def main(workload: str = "k3_h96_t32768") -> None:
    import numpy as np
    import torch

    from . import inputs, kda

    _build.LIB_PATH = build_profiling_library()
    x = inputs.workload_inputs(workload, device="cuda")
    for _ in range(2):
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                          x["cu_seqlens"])
    torch.cuda.synchronize()
    n_chunks = min(4096, (int(x["lengths"][0]) + 63) // 64)
    buf = (ctypes.c_longlong * (4096 * SLOTS))()
    kda.library().kda_debug_phase_clock(buf, 4096 * SLOTS)
    raw = np.array(buf[:], dtype=np.int64).reshape(4096, SLOTS)[:n_chunks]
    stamps = raw[:, :len(PHASES)]
    # interval k = stamp k+1 - stamp k; the last one runs to the next chunk's stamp 0
    nxt = np.concatenate([stamps[1:, :1], stamps[-1:, :1]])
    d = np.diff(np.concatenate([stamps, nxt], axis=1), axis=1)[1:-1]
    med = np.median(d, axis=0)
    total = med.sum()
    print(f"{workload}: median cycles per chunk of chain 0 over {d.shape[0]} chunks")
    for name, v in zip(PHASES, med):
        print(f"  {name:28s} {v:8.0f}  {100 * v / total:5.1f}%")
    print(f"  {'total per chunk':28s} {total:8.0f}")
    # chunks whose state-independent half came from a helper CTA (slot 50)
    helped = raw[1:-1, 50] == 1
    for label, sel in (("helped", helped), ("computed", ~helped)):
        if sel.sum() == 0:
            continue
        m = np.median(d[sel], axis=0)
        print(f"  {label} chunks ({int(sel.sum())}): " +
              ", ".join(f"{n.split(' ')[0]} {v:.0f}" for n, v in zip(PHASES, m)) +
              f"; total {m.sum():.0f}")
    print("stamps as offsets from the chunk's first stamp (median):")
    marks = sorted([(np.median(raw[1:-1, i] - raw[1:-1, 0]), EXTRA[i]) for i in EXTRA
                    if raw[1:-1, i].any()] +
                   [(np.median(raw[1:-1, i] - raw[1:-1, 0]), "t0: end of " + PHASES[i - 1])
                    for i in range(1, len(PHASES))])
    for off, name in marks:
        print(f"  {off:8.0f}  {name}")

if __name__ == "__main__":
    main(*sys.argv[1:2])
