"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU.

Nothing here launches a kernel or needs a GPU: every call below fails host-side
validation, which runs before any CUDA call.  Pointers are fake, 16-byte
aligned addresses that are never dereferenced.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_13_gb300 import _build, kda
    _build.build_library()
    return kda.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("kda_chunk_fwd", "kda_chunk_fwd_sched", "kda_decode_step", "kda_decode_replay",
              "kda_prep_fwd", "kda_post_fwd", "kda_chunk_fwd_workspace_size",
              "kda_status_string", "kda_read_device_status", "kda_read_device_status_detail",
              "kda_read_chunk_stats", "kda_chunk_fwd_transitions", "kda_state_combine",
              "kda_version", "kda_test_arm_timeout", "kda_chunk_fwd_noalloc",
              "kda_noalloc_read_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libkda.so does not export {name}"
    from gated_delta_rule_13_gb300 import kda
    assert set(kda.EXPORTED) == set(declared_functions())


def test_status_strings(lib):
    from gated_delta_rule_13_gb300 import kda
    for code in range(6):
        s = kda.status_string(code)
        assert s.startswith("KDA_")
    assert "unknown" in kda.status_string(99)
    assert kda.kda_version() >= 10000


A = 0x10000  # fake aligned addresses, never dereferenced


def _fwd(lib, **over):
    args = dict(q=A, k=A + 0x1000, v=A + 0x2000, la=A + 0x3000, beta=A + 0x4000, s0=None,
                cu=A + 0x5000, n_seqs=2, n_tokens=100, H=4, dk=128, dv=128, dtype=1,
                out=A + 0x6000, fin=None, ws=A + 0x7000, ws_bytes=1 << 20, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_chunk_fwd(vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["la"]),
                             vp(args["beta"]), vp(args["s0"]), vp(args["cu"]), args["n_seqs"],
                             args["n_tokens"], args["H"], args["dk"], args["dv"], args["dtype"],
                             vp(args["out"]), vp(args["fin"]), vp(args["ws"]), args["ws_bytes"],
                             vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(la=None), 1),
    (dict(beta=None), 1), (dict(out=None), 1), (dict(cu=None), 1),
    (dict(H=0), 1), (dict(H=-3), 1), (dict(n_seqs=-1), 1), (dict(n_tokens=-5), 1),
    (dict(dk=0), 1), (dict(dk=64), 2), (dict(dv=256), 2), (dict(dtype=7), 2),
    (dict(q=A + 8), 1), (dict(out=A + 0x6004), 1), (dict(la=A + 0x3002), 1),
    (dict(s0=A + 0x100000, fin=A + 0x100000 + 4096), 1),   # init/final overlap
    (dict(ws=None), 3), (dict(ws_bytes=16), 3), (dict(ws=A + 0x7008), 3),
])
def test_chunk_fwd_rejects_before_launch(lib, over, code):
    assert _fwd(lib, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(H=0), 1), (dict(dk=64), 2), (dict(dtype=7), 2),
    (dict(la=A + 0x3002), 1), (dict(ws=None), 3), (dict(ws_bytes=16), 3),
])
@pytest.mark.parametrize("caps", [(-1, -1), (0, 0), (4, 7)])
def test_chunk_fwd_sched_rejects_before_launch(lib, over, code, caps):
    """The schedule caps change nothing about argument checking."""
    args = dict(q=A, k=A + 0x1000, v=A + 0x2000, la=A + 0x3000, beta=A + 0x4000, s0=None,
                cu=A + 0x5000, n_seqs=2, n_tokens=100, H=4, dk=128, dv=128, dtype=1,
                out=A + 0x6000, fin=None, ws=A + 0x7000, ws_bytes=1 << 20, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    rc = lib.kda_chunk_fwd_sched(
        vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["la"]), vp(args["beta"]),
        vp(args["s0"]), vp(args["cu"]), args["n_seqs"], args["n_tokens"], args["H"], args["dk"],
        args["dv"], args["dtype"], vp(args["out"]), vp(args["fin"]), caps[0], caps[1],
        vp(args["ws"]), args["ws_bytes"], vp(args["stream"]))
    assert rc == code


def test_no_environment_reads():
    """The schedule is an argument: the library source reads no environment."""
    csrc = os.path.join(ROOT, "gated_delta_rule_13_gb300", "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f), encoding="utf-8").read()
        assert "getenv" not in text, f


def test_test_control_and_status_readers_reject_bad_arguments(lib):
    vp = ctypes.c_void_p
    assert lib.kda_test_arm_timeout(None, 0, 0, 1000, None) == 1
    assert lib.kda_test_arm_timeout(vp(A + 8), 0, 0, 1000, None) == 1       # misaligned
    assert lib.kda_test_arm_timeout(vp(A), 0, -1, 1000, None) == 1          # chunk < 0
    assert lib.kda_test_arm_timeout(vp(A), 0, 0, 0, None) == 1              # no wait
    assert lib.kda_test_arm_timeout(vp(A), 0, 0, 2000001, None) == 1        # beyond 2 s
    d = (ctypes.c_int32 * 4)()
    assert lib.kda_read_device_status_detail(None, None, 0, d) == 1
    assert lib.kda_read_device_status_detail(vp(A), None, 0, None) == 1
    assert lib.kda_noalloc_read_status(None, 0, None) == 1


def test_workspace_size(lib):
    from gated_delta_rule_13_gb300 import kda
    a = kda.kda_chunk_fwd_workspace_size(1, 512, 1)
    b = kda.kda_chunk_fwd_workspace_size(1000, 512, 1)
    assert a >= 256 + 8 and b >= 256 + 4 * 1001 and a % 256 == 0 and b % 256 == 0
    with pytest.raises(kda.KDAError) as e:
        kda.kda_chunk_fwd_workspace_size(1, 512, 1, dk=64)
    assert e.value.code == kda.KDA_ERR_UNSUPPORTED
    with pytest.raises(kda.KDAError) as e:
        kda.kda_chunk_fwd_workspace_size(-1, 512, 1)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_chunk_fwd_workspace_size(1, 1, 1, 128, 128, 1, None) == 1


def _dec(lib, **over):
    args = dict(state=A, q=A + 0x1000, k=A + 0x2000, v=A + 0x3000, la=A + 0x4000,
                beta=A + 0x5000, B=4, H=2, dk=128, dv=128, dtype=1, out=A + 0x40000000,
                stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_decode_step(vp(args["state"]), vp(args["q"]), vp(args["k"]), vp(args["v"]),
                               vp(args["la"]), vp(args["beta"]), args["B"], args["H"],
                               args["dk"], args["dv"], args["dtype"], vp(args["out"]),
                               vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(state=None), 1), (dict(q=None), 1), (dict(out=None), 1), (dict(beta=None), 1),
    (dict(B=-1), 1), (dict(H=0), 1), (dict(dk=32), 2), (dict(dv=64), 2), (dict(dtype=3), 2),
    (dict(k=A + 0x2001), 1), (dict(v=A + 0x3004), 1), (dict(beta=A + 0x5002), 1),
    (dict(out=A + 0x800), 1),                               # out inside the state
])
def test_decode_rejects_before_launch(lib, over, code):
    assert _dec(lib, **over) == code


def _replay(lib, **over):
    args = dict(state=A, q=A + 0x1000, k=A + 0x2000, v=A + 0x3000, la=A + 0x4000,
                beta=A + 0x5000, n=A + 0x6000, B=4, T=3, H=2, dk=128, dv=128, dtype=1,
                out=A + 0x40000000, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_decode_replay(vp(args["state"]), vp(args["q"]), vp(args["k"]), vp(args["v"]),
                                 vp(args["la"]), vp(args["beta"]), vp(args["n"]), args["B"],
                                 args["T"], args["H"], args["dk"], args["dv"], args["dtype"],
                                 vp(args["out"]), vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(state=None), 1), (dict(q=None), 1), (dict(n=None), 1), (dict(beta=None), 1),
    (dict(B=-1), 1), (dict(T=0), 1), (dict(H=0), 1), (dict(dk=32), 2), (dict(dtype=3), 2),
    (dict(k=A + 0x2001), 1), (dict(v=A + 0x3004), 1), (dict(n=A + 0x6002), 1),
    # element-aligned but not 16-byte aligned: rows are fetched by bulk copies
    (dict(q=A + 0x1002), 1), (dict(k=A + 0x2008), 1), (dict(la=A + 0x4004), 1),
    (dict(out=A + 0x800), 1),                               # out inside the state
])
def test_replay_rejects_before_launch(lib, over, code):
    assert _replay(lib, **over) == code


def test_replay_empty_batch_launches_nothing(lib):
    assert _replay(lib, B=0) == 0


def _prep(lib, **over):
    n = 0x100000
    args = dict(qr=A, kr=A + n, vr=A + 2 * n, w=A + 3 * n, a=A + 4 * n, b=A + 5 * n,
                cu=A + 6 * n, n_seqs=1, N=64, H=2, dk=128, dv=128, dtype=1, q=A + 7 * n,
                k=A + 8 * n, v=A + 9 * n, la=A + 10 * n, beta=A + 11 * n, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_prep_fwd(*(vp(args[x]) for x in ("qr", "kr", "vr", "w", "a", "b", "cu")),
                            args["n_seqs"], args["N"], args["H"], args["dk"], args["dv"],
                            args["dtype"],
                            *(vp(args[x]) for x in ("q", "k", "v", "la", "beta", "stream")))


@pytest.mark.parametrize("over,code", [
    (dict(qr=None), 1), (dict(cu=None), 1), (dict(beta=None), 1), (dict(n_seqs=0), 1),
    (dict(N=-1), 1), (dict(H=0), 1), (dict(dk=64), 2), (dict(dtype=3), 2),
    (dict(qr=A + 4), 1), (dict(w=A + 0x300008), 1), (dict(b=A + 0x500002), 1),
    (dict(q=A + 0x40), 1),                                 # q overlaps q_raw
])
def test_prep_rejects_before_launch(lib, over, code):
    assert _prep(lib, **over) == code


def _post(lib, **over):
    args = dict(o=A, g=A + 0x100000, gamma=A + 0x200000, N=64, H=2, dv=128, dtype=1,
                out=A + 0x300000, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_post_fwd(vp(args["o"]), vp(args["g"]), vp(args["gamma"]), args["N"],
                            args["H"], args["dv"], args["dtype"], vp(args["out"]),
                            vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(o=None), 1), (dict(gamma=None), 1), (dict(N=-1), 1), (dict(H=0), 1),
    (dict(dv=64), 2), (dict(dtype=7), 2), (dict(gamma=A + 0x200004), 1), (dict(g=A + 2), 1),
])
def test_post_rejects_before_launch(lib, over, code):
    assert _post(lib, **over) == code


def test_empty_layer_ops_launch_nothing(lib):
    assert _prep(lib, N=0) == 0 and _post(lib, N=0) == 0


def test_read_device_status_null(lib):
    st = ctypes.c_int32(0)
    assert lib.kda_read_device_status(None, None, 0, ctypes.byref(st)) == 1
    assert lib.kda_read_device_status(ctypes.c_void_p(A), None, 0, None) == 1


def _transitions(lib, **over):
    args = dict(q=A, k=A + 0x1000, v=A + 0x2000, la=A + 0x3000, beta=A + 0x4000, cu=A + 0x5000,
                n_seqs=2, n_tokens=100, H=4, dk=128, dv=128, dtype=1, b=A + 0x100000,
                m=A + 0x300000, ws=A + 0x7000, ws_bytes=1 << 20, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_chunk_fwd_transitions(
        vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["la"]), vp(args["beta"]),
        vp(args["cu"]), args["n_seqs"], args["n_tokens"], args["H"], args["dk"], args["dv"],
        args["dtype"], vp(args["b"]), vp(args["m"]), vp(args["ws"]), args["ws_bytes"],
        vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(dtype=0), 2),              # fp32 inputs: bf16 only
    (dict(dk=64), 2),
    (dict(b=None), 1), (dict(m=None), 1), (dict(cu=None), 1),
    (dict(H=0), 1), (dict(n_seqs=-1), 1),
    (dict(b=A + 0x100008), 1),       # misaligned state
    (dict(m=A + 0x100000), 1),       # B and M overlap
    (dict(ws=None), 3), (dict(ws_bytes=16), 3),
])
def test_transitions_reject_before_launch(lib, over, code):
    assert _transitions(lib, **over) == code


def _combine(lib, **over):
    one = 4 * 128 * 128 * 4  # H = 4 states of one sequence
    args = dict(init=A, b=A + 0x1000000, m=A + 0x2000000, n_seqs=2, K=3, H=4, dk=128, dv=128,
                starts=A + 0x3000000, end=A + 0x4000000, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_state_combine(vp(args["init"]), vp(args["b"]), vp(args["m"]), args["n_seqs"],
                                 args["K"], args["H"], args["dk"], args["dv"],
                                 vp(args["starts"]), vp(args["end"]), vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(K=0), 1), (dict(H=0), 1), (dict(n_seqs=-1), 1),
    (dict(b=None), 1), (dict(m=None), 1), (dict(dk=64), 2),
    (dict(end=A + 0x4000004), 1),               # misaligned
    (dict(starts=A + 0x1000000), 1),            # starts overlap B
    (dict(end=A + 0x2000000 + 65536), 1),       # end overlaps M
    (dict(end=A + 0x3000000), 1),               # end overlaps starts
    (dict(init=A + 0x4000000), 1),              # end overlaps init
])
def test_state_combine_rejects_before_launch(lib, over, code):
    assert _combine(lib, **over) == code


def test_empty_combine_launches_nothing(lib):
    assert _combine(lib, n_seqs=0) == 0


def test_read_chunk_stats_null(lib):
    a, b = ctypes.c_int32(0), ctypes.c_int32(0)
    assert lib.kda_read_chunk_stats(None, None, ctypes.byref(a), ctypes.byref(b)) == 1
    assert lib.kda_read_chunk_stats(ctypes.c_void_p(A), None, None, ctypes.byref(b)) == 1
    assert lib.kda_read_chunk_stats(ctypes.c_void_p(A), None, ctypes.byref(a), None) == 1


def test_product_path_does_not_import_oracle():
    """The CUDA path never reaches the oracle (it is test infrastructure)."""
    pkg = os.path.join(ROOT, "gated_delta_rule_13_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "kda_oracle" not in text, f


def test_host_pipeline_piece_bounds():
    """Pieces of kda_chunk_fwd_host: whole chunks except the sequence's end, the
    last full piece cut in halves down to 1024 tokens, bounds increasing."""
    from gated_delta_rule_13_gb300.kda import _piece_bounds
    assert _piece_bounds(32768, 4096) == [0, 4096, 8192, 12288, 16384, 20480, 24576, 28672,
                                          30720, 31744, 32768]
    assert _piece_bounds(5000, 4096) == [0, 4096, 5000]
    assert _piece_bounds(100, 4096) == [0, 100]
    for n in (1, 63, 64, 65, 1000, 2048, 4097, 9999, 70000):
        for piece in (64, 256, 4096):
            b = _piece_bounds(n, piece)
            assert b[0] == 0 and b[-1] == n
            assert all(x % 64 == 0 for x in b[:-1])
            assert all(b1 - b0 <= piece for b0, b1 in zip(b, b[1:]))
            assert all(b0 < b1 for b0, b1 in zip(b, b[1:]))


def _prep_state(lib, **over):
    n = 0x100000
    args = dict(qr=A, kr=A + n, vr=A + 2 * n, w=A + 3 * n, a=A + 4 * n, b=A + 5 * n,
                cu=A + 6 * n, n_seqs=1, N=64, H=2, dk=128, dv=128, dtype=1, wi=A + 12 * n,
                wo=A + 13 * n, q=A + 7 * n, k=A + 8 * n, v=A + 9 * n, la=A + 10 * n,
                beta=A + 11 * n, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_prep_fwd_state(*(vp(args[x]) for x in ("qr", "kr", "vr", "w", "a", "b", "cu")),
                                  args["n_seqs"], args["N"], args["H"], args["dk"], args["dv"],
                                  args["dtype"], vp(args["wi"]), vp(args["wo"]),
                                  *(vp(args[x]) for x in ("q", "k", "v", "la", "beta", "stream")))


@pytest.mark.parametrize("over,code", [
    (dict(qr=None), 1), (dict(cu=None), 1), (dict(n_seqs=0), 1), (dict(H=0), 1),
    (dict(dk=64), 2), (dict(dtype=3), 2), (dict(wi=A + 0xC00004), 1), (dict(wo=A + 0xD00002), 1),
    (dict(wo=A + 0xC00100), 1),                 # windows overlap without being the same array
    (dict(wo=A + 0x700000), 1),                 # window over the q output
    (dict(wi=A), 1),                            # window over q_raw
])
def test_prep_state_rejects_before_launch(lib, over, code):
    assert _prep_state(lib, **over) == code


def _layer_replay(lib, **over):
    n = 0x1000000
    args = dict(state=A, win=A + n, qr=A + 2 * n, kr=A + 3 * n, vr=A + 4 * n, a=A + 5 * n,
                b=A + 6 * n, g=A + 7 * n, w=A + 8 * n, gamma=A + 9 * n, na=A + 10 * n, B=4, T=3,
                H=2, dk=128, dv=128, dtype=1, out=A + 11 * n, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_layer_replay(*(vp(args[x]) for x in ("state", "win", "qr", "kr", "vr", "a", "b",
                                                         "g", "w", "gamma", "na")),
                                args["B"], args["T"], args["H"], args["dk"], args["dv"],
                                args["dtype"], vp(args["out"]), vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(state=None), 1), (dict(win=None), 1), (dict(g=None), 1), (dict(na=None), 1),
    (dict(B=-1), 1), (dict(T=0), 1), (dict(H=0), 1), (dict(dk=64), 2), (dict(dtype=5), 2),
    (dict(state=A + 8), 1), (dict(w=A + 0x8000004), 1), (dict(out=A + 0xB000002), 1),
    # element-aligned but not 16-byte aligned: rows are fetched by bulk copies
    (dict(win=A + 0x1000002), 1), (dict(qr=A + 0x2000002), 1), (dict(g=A + 0x7000008), 1),
    (dict(a=A + 0x5000004), 1),
    (dict(win=A + 0x100), 1),                   # window inside the state
    (dict(out=A + 0x1000000), 1),               # output over the window
])
def test_layer_replay_rejects_before_launch(lib, over, code):
    assert _layer_replay(lib, **over) == code


def test_layer_replay_empty_batch_launches_nothing(lib):
    assert _layer_replay(lib, B=0) == 0


def _bwd(lib, **over):
    n = 0x1000000
    args = dict(q=A, k=A + n, v=A + 2 * n, la=A + 3 * n, beta=A + 4 * n, init=None, cu=A + 5 * n,
                n_seqs=1, N=64, H=2, dk=128, dv=128, dtype=1, do=A + 6 * n, df=None, dq=A + 7 * n,
                dkk=A + 8 * n, dvv=A + 9 * n, dla=A + 10 * n, db=A + 11 * n, dinit=None, every=0,
                ws=None, ws_bytes=0, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.kda_chunk_bwd_sched(
        *(vp(args[x]) for x in ("q", "k", "v", "la", "beta", "init", "cu")), args["n_seqs"],
        args["N"], args["H"], args["dk"], args["dv"], args["dtype"],
        *(vp(args[x]) for x in ("do", "df", "dq", "dkk", "dvv", "dla", "db", "dinit")),
        args["every"], vp(args["ws"]), args["ws_bytes"], vp(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(), 3),                                      # everything valid but the workspace
    (dict(every=16), 3), (dict(every=1024), 3),
    (dict(every=3), 1), (dict(every=2), 1), (dict(every=6), 1), (dict(every=2048), 1),
    (dict(every=-1), 1),
    (dict(q=None), 1), (dict(cu=None), 1), (dict(dk=64), 2), (dict(dtype=4), 2),
    (dict(q=A + 1), 1), (dict(la=A + 0x3000002), 1),
    # element-aligned but not 16-byte aligned: rows are fetched by 16-byte copies
    (dict(q=A + 2), 1), (dict(v=A + 0x2000008), 1), (dict(do=A + 0x6000004), 1),
    (dict(dq=A + 0x7000002), 3),                      # outputs need element alignment only
    (dict(dq=A), 1),                                  # dq over q
    (dict(db=A + 0xA000000), 1),                      # d_beta over d_log_alpha
])
def test_bwd_rejects_before_launch(lib, over, code):
    assert _bwd(lib, **over) == code


def test_bwd_workspace_size_follows_the_checkpoint_interval(lib):
    from gated_delta_rule_13_gb300 import kda
    f32 = kda.KDA_F32
    small = kda.kda_chunk_bwd_workspace_size(4, 16384, 16, dtype=f32)
    assert small == kda.kda_chunk_bwd_workspace_size(4, 16384, 16, dtype=f32, ckpt_every=4)
    s16 = kda.kda_chunk_bwd_workspace_size(4, 16384, 16, dtype=f32, ckpt_every=16)
    state = 128 * 128 * 4
    assert small - s16 == (16384 // 4 - 16384 // 16) * 16 * state
    # bf16 by default: the chunked pass, bf16 states every 16 tokens and no fp32
    # accumulators of dq and dk; an explicit interval selects the token loop
    acc = 2 * 16384 * 16 * 128 * 4
    half_states = (16384 // 16 + 4 + 1) * 16 * 128 * 128 * 2
    chunked = kda.kda_chunk_bwd_workspace_size(4, 16384, 16)
    assert chunked == kda.kda_chunk_bwd_workspace_size(4, 16384, 16, ckpt_every=16) - acc - half_states
    assert kda.kda_chunk_bwd_workspace_size(4, 16384, 16, ckpt_every=4) == small
    # a long problem gets a wider default interval, its states within 16 GiB
    # (for bf16 too: states every 16 tokens would not fit)
    for dt in (kda.KDA_BF16, f32):
        big = kda.kda_chunk_bwd_workspace_size(8, 1 << 20, 96, dtype=dt)
        acc = 2 * (1 << 20) * 96 * 128 * 4
        assert big - acc <= (16 << 30) + (1 << 20)
    for bad in (3, 6, 2048, -4):
        with pytest.raises(RuntimeError):
            kda.kda_chunk_bwd_workspace_size(1, 64, 1, ckpt_every=bad)
