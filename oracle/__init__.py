"""CPU reference decoder (the oracle).  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It wraps ``wfst_oracle.c`` — a plain,
single-threaded C restatement of the decoding rules of the page "GPU WFST
Beam-Search Decoder" — through ctypes, and shares no code with the CUDA
decoder in ``wfst_beam_search_gb300``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "wfst_oracle.c")
_HDR = os.path.join(_HERE, "wfst_oracle.h")

REC_EPS, REC_FINAL, REC_REDIRECT = 1, 2, 4
ST_NAMES = ["frames", "arcs_expanded", "sum_n", "sum_D", "sum_a", "sum_m", "max_n",
            "max_D", "tokens", "records", "eps_relaxed", "finals", "records_dropped"]

LAT_DTYPE = np.dtype([("t", "<i4"), ("src_state", "<i4"), ("dst_state", "<i4"),
                      ("arc_id", "<i4"), ("flags", "<i4"), ("score", "<f4")])
STEP_DTYPE = np.dtype([("t", "<i4"), ("n", "<i4"), ("num_cands", "<i4"),
                       ("num_admitted", "<i4"), ("next_size", "<i4"), ("pad", "<i4"),
                       ("beam", "<f4"), ("max_end", "<f4"), ("cutoff", "<f4"),
                       ("pad2", "<f4")])

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with plain IEEE fp32 semantics (no contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _GraphDesc(C.Structure):
    _fields_ = [("num_states", C.c_int32), ("start_state", C.c_int32),
                ("vocab_size", C.c_int32), ("pad_", C.c_int32), ("num_arcs", C.c_int64),
                ("row_splits", C.c_void_p), ("ilabel", C.c_void_p), ("olabel", C.c_void_p),
                ("weight", C.c_void_p), ("dst", C.c_void_p), ("final_weight", C.c_void_p)]


class _Params(C.Structure):
    _fields_ = [("search_beam", C.c_float), ("output_beam", C.c_float),
                ("min_active", C.c_int32), ("max_active", C.c_int32),
                ("allow_partial", C.c_int32), ("lattice", C.c_int32),
                ("lat_prune_interval", C.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
            L.or_graph_new.restype = P
            L.or_graph_new.argtypes = [C.POINTER(_GraphDesc), C.c_char_p, i32]
            L.or_graph_free.argtypes = [P]
            L.or_graph_eps_rank.argtypes = [P, P]
            L.or_graph_eps_rank.restype = i32
            L.or_dec_new.restype = P
            L.or_dec_new.argtypes = [P, C.POINTER(_Params), i32]
            L.or_dec_free.argtypes = [P]
            L.or_dec_advance.argtypes = [P, P, i64, i32]
            L.or_dec_advance.restype = i32
            L.or_dec_partial.argtypes = [P, P, i32, P, P, P]
            L.or_dec_partial.restype = i32
            L.or_dec_finalize.argtypes = [P, P, i32, P, P, i32, P, P, P, P]
            L.or_dec_finalize.restype = i32
            L.or_dec_lattice.argtypes = [P, P, i64]
            L.or_dec_lattice.restype = i64
            L.or_dec_lattice_all.argtypes = [P, P, i64]
            L.or_dec_lattice_all.restype = i64
            L.or_dec_stats.argtypes = [P, P]
            L.or_dec_trace.argtypes = [P, P, i64]
            L.or_dec_trace.restype = i64
            _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(C.c_void_p)


class Graph:
    """An uploaded copy of a CSR graph dict (see ``synth``)."""

    def __init__(self, g: dict):
        L = lib()
        self._keep = dict(
            row_splits=np.ascontiguousarray(g["row_splits"], dtype=np.int64),
            ilabel=np.ascontiguousarray(g["ilabel"], dtype=np.int32),
            olabel=np.ascontiguousarray(g["olabel"], dtype=np.int32),
            weight=np.ascontiguousarray(g["weight"], dtype=np.float32),
            dst=np.ascontiguousarray(g["dst"], dtype=np.int32),
            final=np.ascontiguousarray(g["final"], dtype=np.float32),
        )
        k = self._keep
        self.num_states = int(g["num_states"])
        self.num_arcs = int(len(k["ilabel"]))
        desc = _GraphDesc(self.num_states, int(g["start_state"]), int(g["vocab_size"]), 0,
                          self.num_arcs, _ptr(k["row_splits"]), _ptr(k["ilabel"]),
                          _ptr(k["olabel"]), _ptr(k["weight"]), _ptr(k["dst"]),
                          _ptr(k["final"]))
        err = C.create_string_buffer(256)
        self._h = L.or_graph_new(C.byref(desc), err, 256)
        if not self._h:
            raise ValueError("oracle rejected graph: " + err.value.decode())
        self._keep = None   # the oracle holds its own copy

    def eps_rank(self):
        out = np.empty(self.num_states, dtype=np.int32)
        has = lib().or_graph_eps_rank(self._h, _ptr(out))
        return out, bool(has)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().or_graph_free(h)
            self._h = None


def params(search_beam=20.0, output_beam=8.0, min_active=30, max_active=10000,
           allow_partial=True, lattice=False, lat_prune_interval=0):
    return dict(search_beam=float(search_beam), output_beam=float(output_beam),
                min_active=int(min_active), max_active=int(max_active),
                allow_partial=bool(allow_partial), lattice=bool(lattice),
                lat_prune_interval=int(lat_prune_interval))


class Decoder:
    """One lane.  ``t_eff`` = the utterance length offline, None for streaming."""

    def __init__(self, graph: Graph, p: dict, t_eff: int | None):
        self.graph = graph
        self.p = p
        cp = _Params(p["search_beam"], p["output_beam"], p["min_active"], p["max_active"],
                     int(p["allow_partial"]), int(p["lattice"]), int(p.get("lat_prune_interval", 0)))
        self._h = lib().or_dec_new(graph._h, C.byref(cp), -1 if t_eff is None else int(t_eff))
        if not self._h:
            raise MemoryError("oracle decoder allocation failed")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().or_dec_free(h)
            self._h = None

    def advance(self, lp):
        lp = np.ascontiguousarray(lp, dtype=np.float32)   # fp16 widens exactly
        if lp.ndim != 2:
            raise ValueError("advance takes [frames, V]")
        rc = lib().or_dec_advance(self._h, _ptr(lp), lp.shape[1], lp.shape[0])
        if rc != 0:
            raise RuntimeError(f"oracle advance failed ({rc})")

    def partial(self, cap=1 << 16):
        words = np.zeros(cap, np.int32)
        nw, ok = C.c_int32(), C.c_int32()
        sc = C.c_float()
        rc = lib().or_dec_partial(self._h, _ptr(words), cap, C.byref(nw), C.byref(sc), C.byref(ok))
        if rc != 0:
            raise RuntimeError(f"oracle partial failed ({rc})")
        return dict(words=words[: min(nw.value, cap)].copy(), score=sc.value, ok=ok.value)

    def finalize(self, cap=1 << 16):
        words = np.zeros(cap, np.int32)
        arcs = np.zeros(cap, np.int32)
        nw, na, rf, ok = C.c_int32(), C.c_int32(), C.c_int32(), C.c_int32()
        sc = C.c_float()
        rc = lib().or_dec_finalize(self._h, _ptr(words), cap, C.byref(nw), _ptr(arcs), cap,
                                   C.byref(na), C.byref(sc), C.byref(rf), C.byref(ok))
        if rc != 0:
            raise RuntimeError(f"oracle finalize failed ({rc})")
        return dict(words=words[: min(nw.value, cap)].copy(),
                    arcs=arcs[: min(na.value, cap)].copy(), score=sc.value,
                    reached_final=rf.value, ok=ok.value, n_words=nw.value)

    def lattice(self, kept=True):
        f = lib().or_dec_lattice if kept else lib().or_dec_lattice_all
        n = f(self._h, None, 0)
        out = np.zeros(n, dtype=LAT_DTYPE)
        if n:
            f(self._h, _ptr(out), n)
        return out

    def stats(self):
        out = np.zeros(len(ST_NAMES), np.int64)
        lib().or_dec_stats(self._h, _ptr(out))
        return dict(zip(ST_NAMES, out.tolist()))

    def trace(self):
        n = lib().or_dec_trace(self._h, None, 0)
        out = np.zeros(n, dtype=STEP_DTYPE)
        if n:
            lib().or_dec_trace(self._h, _ptr(out), n)
        return out


def decode(graph: Graph, lp, length: int, p: dict, lattice_out=False, trace=False):
    """Offline decode of one utterance: ``lp`` [>=length, V] (fp32 or fp16)."""
    d = Decoder(graph, p, t_eff=int(length))
    if length > 0:
        d.advance(np.asarray(lp)[:length])
    r = d.finalize()
    r["stats"] = d.stats()
    if lattice_out and p["lattice"]:
        r["lattice"] = d.lattice()
    if trace:
        r["trace"] = d.trace()
    return r


def decode_batch(graph: Graph, lp, lens, p: dict, threads: int = 1, lattice_out=False):
    """Decode every lane; lanes run on ``threads`` host threads (the C call
    releases the GIL)."""
    lp = np.asarray(lp)
    lens = [int(x) for x in lens]
    if threads <= 1:
        return [decode(graph, lp[b], lens[b], p, lattice_out) for b in range(len(lens))]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(decode, graph, lp[b], lens[b], p, lattice_out) for b in range(len(lens))]
        return [f.result() for f in futs]


def blank_skip(lp, lens, threshold=0.98, blank=0):
    """Blank-skip frame pre-slicing, outside the decoder (page "GPU WFST
    Beam-Search Decoder", §3 Decoding Semantics: blank-dominated frames are
    removed before the search, in the WeNet manner, threshold 0.98 by
    default).

    Frame t < lens[b] of lane b is dropped when its blank posterior is above
    the threshold, tested in the log domain in fp32: lp[b, t, blank] (widened
    to fp32) > fp32(log(threshold)), the log taken in double.  Returns the
    kept rows of each lane in order (original dtype) and their frame indices.
    """
    lthr = np.float32(np.log(np.float64(threshold)))
    rows, frames = [], []
    for b in range(len(lens)):
        n = int(lens[b])
        lpb = np.asarray(lp[b][:n])
        keep = ~(lpb[:, blank].astype(np.float32) > lthr)
        idx = np.nonzero(keep)[0].astype(np.int32)
        rows.append(lpb[idx])
        frames.append(idx)
    return rows, frames

