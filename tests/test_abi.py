"""The C ABI library builds, loads and exports every entry point the header
declares (no GPU needed: nothing here launches device work)."""
import os
import re
import subprocess

import pytest

import wfst_beam_search_gb300 as W
from wfst_beam_search_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wfst_gb300.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wfst_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return W.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["wfst_graph_upload", "wfst_decode", "wfst_lattice_export", "wfst_stream_create",
              "wfst_stream_advance", "wfst_stream_finalize", "wfst_stream_release"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (wfst_[a-z_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_binding_uses_the_c_names():
    for n in declared_functions():
        assert hasattr(W, n), n


def test_last_error_and_argument_checks_without_gpu(lib):
    # NULL arguments are rejected on the host before any CUDA call
    assert lib.wfst_graph_upload(None, 0, None) == -1
    assert b"NULL" in lib.wfst_last_error()
    assert lib.wfst_decode(None, None, 0, 0, 0, None, 0, 0, None, None, 0, None, None, None) == -1
    assert lib.wfst_decode_static(None, None, None, 0, 0, 0, None, 0, 0, None, None, 0, None, None,
                                  None) == -1
    import ctypes as C
    n = C.c_int64()
    ch = C.c_int32()
    for rc in (lib.wfst_lattice_export(None, 0, None, 0, C.byref(n)),
               lib.wfst_stream_create(None, C.byref(ch)),
               lib.wfst_stream_advance(None, None, 0, None, 0, 0, 0, None, 0, 0, None, None, 0, None,
                                       None, None),
               lib.wfst_stream_finalize(None, None, 0, None, None, 0, None, None, None),
               lib.wfst_stream_release(None, 0),
               lib.wfst_stats(None, None, 0),
               lib.wfst_mem_stats(None, None, 0),
               lib.wfst_test_barrier_timeout(None, 200_000_000),
               lib.wfst_probe_random_gather(None, 0, 16, 1, 4, 0, None, None),
               lib.wfst_decoder_create(None, None, 1, 1, None, None)):
        assert rc == -1
        assert lib.wfst_last_error()


def test_graph_validation_rejects_corrupt_graphs_on_host(lib):
    import ctypes as C
    import numpy as np
    import synth
    # epsilon cycle -> CORRUPT_GRAPH before any device allocation
    g = synth.graph_from_arcs(3, 2, np.array([0, 1, 2]), [1, 2, 0], [-1, -1, -1], [0, 0, 0],
                              [0.0, 0.0, 0.0], np.zeros(3, np.float32))
    for bad, msg in [(g, b"cycle")]:
        keep = [np.ascontiguousarray(bad[k]) for k in ("row_splits", "ilabel", "olabel",
                                                       "weight", "dst", "final")]
        desc = W.GraphDesc(3, 0, 2, 0, 3, *[k.ctypes.data_as(C.c_void_p) for k in keep])
        h = C.c_void_p()
        assert lib.wfst_graph_upload(C.byref(desc), 0, C.byref(h)) == -2
        assert msg in lib.wfst_last_error()
    # vocab too large for u16 labels
    keep = [np.ascontiguousarray(g[k]) for k in ("row_splits", "ilabel", "olabel", "weight",
                                                 "dst", "final")]
    desc = W.GraphDesc(3, 0, 70000, 0, 3, *[k.ctypes.data_as(C.c_void_p) for k in keep])
    h = C.c_void_p()
    assert lib.wfst_graph_upload(C.byref(desc), 0, C.byref(h)) == -2
    assert b"vocab" in lib.wfst_last_error()


def test_missing_library_fails_loudly():
    """Without the built library every entry of the binding raises: there is
    no CPU path to fall back on.  Checked in a child process that points the
    binding at a library file that does not exist."""
    import sys
    code = (
        "import numpy as np, synth, wfst_beam_search_gb300 as W\n"
        "from wfst_beam_search_gb300 import _build\n"
        "_build.LIB = '/nonexistent/libwfst_gb300.so'\n"
        "for f in (W.load, lambda: W.Graph(synth.make_graph(0), device=0)):\n"
        "    try:\n"
        "        f()\n"
        "    except ImportError as e:\n"
        "        assert 'no CPU fallback' in str(e), e\n"
        "    else:\n"
        "        raise SystemExit('no error')\n"
        "print('ok')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr[-2000:]


def test_log_prob_arguments_are_checked_on_the_host():
    import numpy as np
    with pytest.raises(ValueError, match=r"\[B, T, V\]"):
        W._lp_args(np.zeros((4, 5), np.float32))
    with pytest.raises(TypeError):
        W._lp_args(np.zeros((1, 4, 5), np.float64))
    with pytest.raises(ValueError, match="unit stride"):
        W._lp_args(np.zeros((1, 5, 4), np.float32).transpose(0, 2, 1))
    lp = np.zeros((2, 3, 5), np.float16)[:, ::2]
    _, dt, sb, st, B, T = W._lp_args(lp)
    assert (dt, sb, st, B, T) == (W.WFST_F16, 15, 10, 2, 2)
    # host arrays keep the caller's stream choice (None: the default stream)
    assert W._default_stream(lp, None) is None and W._default_stream(lp, 7) == 7


def test_graph_upload_checks_the_device_id(lib):
    """A negative device id is refused before anything else; an id past the
    visible devices is refused once the graph itself has validated (without
    any CUDA device the count itself fails: WFST_ERR_CUDA)."""
    import ctypes as C
    import numpy as np
    import synth
    g = synth.graph_from_arcs(2, 2, np.array([0]), [1], [1], [0], [0.0], np.zeros(2, np.float32))
    keep = [np.ascontiguousarray(g[k]) for k in ("row_splits", "ilabel", "olabel", "weight", "dst", "final")]
    desc = W.GraphDesc(2, 0, 2, 0, 1, *[k.ctypes.data_as(C.c_void_p) for k in keep])
    h = C.c_void_p()
    assert lib.wfst_graph_upload(C.byref(desc), -1, C.byref(h)) == -1
    assert b"device" in lib.wfst_last_error() and not h.value
    rc = lib.wfst_graph_upload(C.byref(desc), 1 << 20, C.byref(h))
    assert rc == (-1 if _has_cuda_device() else -3) and not h.value
    assert b"device" in lib.wfst_last_error()


def _has_cuda_device():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def test_binding_structs_match_the_header(tmp_path):
    """The ctypes mirrors of wfst_params, wfst_capacity and wfst_graph_desc
    have the header's sizes and field offsets (compiled with the host C
    compiler against include/wfst_gb300.h)."""
    import ctypes as C
    structs = {"wfst_params": W.Params, "wfst_capacity": W.Capacity, "wfst_graph_desc": W.GraphDesc}
    lines = ["#include <stdio.h>", "#include <stddef.h>", f'#include "{HEADER}"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'  printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, py in structs.items():
        assert got[(cname, "size")] == C.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_blank_skip_argument_checks_without_gpu(lib):
    """wfst_blank_skip validates its arguments on the host before any launch:
    NULL arrays, a blank id outside [0, V), a non-positive threshold, short
    strides and host (not device) arrays are refused with INVALID_ARG."""
    import ctypes as C
    import numpy as np
    lp = np.zeros((2, 3, 4), np.float32)
    lens = np.array([3, 3], np.int32)
    out = np.zeros_like(lp)
    out_lens = np.zeros(2, np.int32)
    fmap = np.zeros((2, 3), np.int32)
    P = lambda a: a.ctypes.data_as(C.c_void_p)  # noqa: E731
    f = lib.wfst_blank_skip
    base = dict(lp=P(lp), dt=0, sb=12, st=4, V=4, blank=0, thr=C.c_float(0.98), lens=P(lens), B=2, T=3,
                out=P(out), ol=P(out_lens), fm=P(fmap))

    def call(**kw):
        a = dict(base, **kw)
        return f(a["lp"], a["dt"], a["sb"], a["st"], a["V"], a["blank"], a["thr"], a["lens"], a["B"], a["T"],
                 a["out"], a["ol"], a["fm"], None)
    assert call(B=0) == 0                      # nothing to do
    assert call(lp=None) == -1 and b"NULL" in lib.wfst_last_error()
    assert call(blank=4) == -1 and b"blank_id" in lib.wfst_last_error()
    assert call(thr=C.c_float(0.0)) == -1 and b"threshold" in lib.wfst_last_error()
    assert call(st=3) == -1 and b"stride" in lib.wfst_last_error()
    assert call(dt=7) == -1 and b"dtype" in lib.wfst_last_error()
    assert call() == -1 and b"device memory" in lib.wfst_last_error()   # host arrays
