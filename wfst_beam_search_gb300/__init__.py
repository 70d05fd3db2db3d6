"""Python binding of the GB300 WFST beam-search decoder's C ABI.

The functions below carry the C names (``wfst_graph_upload``, ``wfst_decode``,
...) and only marshal arguments: every step of the decode runs in the CUDA
library ``_build/libwfst_gb300.so`` (see ``include/wfst_gb300.h``).  There is
no CPU fallback; loading fails loudly when the library is missing.

``Graph`` and ``Decoder`` wrap the handles for convenience.  Device buffers
may be torch CUDA tensors (pointer + strides are passed through) or numpy
arrays (host input: the library copies them to the device inside the call).
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import numpy as np

from . import _build

WFST_OK = 0
WFST_F32, WFST_F16 = 0, 1
OVF_ARENA, OVF_KEPT, OVF_PATH = 4, 16, 32
REC_EPS, REC_FINAL, REC_REDIRECT = 1, 2, 4
STAT_NAMES = ["frames", "arcs_expanded", "sum_n", "sum_D", "sum_a", "sum_m", "eps",
              "steps", "barriers", "kernel_ns", "ns_init", "ns_max", "ns_expand", "ns_closure",
              "ns_prune", "ns_prologue", "ns_commit", "ns_clear", "ns_max_tiles", "ns_wait_x",
              "ns_expand_tiles", "ns_final", "ns_wait_y", "lattice_records_held", "eps_passes",
              "log_high_water"]
ERRORS = {-1: "INVALID_ARG", -2: "CORRUPT_GRAPH", -3: "CUDA", -4: "OOM", -5: "CAPACITY",
          -6: "TIMEOUT", -7: "STATE"}

LAT_DTYPE = np.dtype([("t", "<i4"), ("src_state", "<i4"), ("dst_state", "<i4"),
                      ("arc_id", "<i4"), ("flags", "<i4"), ("score", "<f4")])

EXPORTED = ["wfst_graph_upload", "wfst_graph_info", "wfst_graph_free", "wfst_decoder_create",
            "wfst_decoder_free", "wfst_decode", "wfst_lattice_export", "wfst_stream_create",
            "wfst_stream_advance", "wfst_stream_finalize", "wfst_stream_release", "wfst_stats",
            "wfst_decode_static", "wfst_mem_stats", "wfst_blank_skip", "wfst_test_barrier_timeout",
            "wfst_probe_random_gather", "wfst_last_error"]


class WfstError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class GraphDesc(C.Structure):
    _fields_ = [("num_states", C.c_int32), ("start_state", C.c_int32),
                ("vocab_size", C.c_int32), ("reserved", C.c_int32), ("num_arcs", C.c_int64),
                ("row_splits", C.c_void_p), ("ilabel", C.c_void_p), ("olabel", C.c_void_p),
                ("weight", C.c_void_p), ("dst", C.c_void_p), ("final_weight", C.c_void_p)]


class Params(C.Structure):
    _fields_ = [("search_beam", C.c_float), ("output_beam", C.c_float),
                ("min_active", C.c_int32), ("max_active", C.c_int32),
                ("allow_partial", C.c_int32), ("lattice", C.c_int32), ("streaming", C.c_int32),
                ("options", C.c_int32), ("gc_interval", C.c_int32), ("lat_prune_interval", C.c_int32)]


class Capacity(C.Structure):
    _fields_ = [("frontier_cap", C.c_int64), ("log_cap", C.c_int64),
                ("lattice_cap", C.c_int64), ("path_cap", C.c_int64), ("fin_cap", C.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load the CUDA library (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise ImportError("libwfst_gb300.so is not built; run __graft_entry__.build() "
                              "(the decoder has no CPU fallback)")
        L = C.CDLL(_build.LIB)
        P, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        L.wfst_last_error.restype = C.c_char_p
        L.wfst_graph_upload.argtypes = [C.POINTER(GraphDesc), i32, C.POINTER(P)]
        L.wfst_graph_info.argtypes = [P, P]
        L.wfst_graph_free.argtypes = [P]
        L.wfst_graph_free.restype = None
        L.wfst_decoder_create.argtypes = [P, C.POINTER(Params), i32, i32, C.POINTER(Capacity),
                                          C.POINTER(P)]
        L.wfst_decoder_free.argtypes = [P]
        L.wfst_decoder_free.restype = None
        L.wfst_decode.argtypes = [P, P, i32, i64, i64, P, i32, i32, P, P, i32, P, P, P]
        L.wfst_decode_static.argtypes = [P, C.POINTER(Params), P, i32, i64, i64, P, i32, i32, P, P,
                                         i32, P, P, P]
        L.wfst_lattice_export.argtypes = [P, i32, P, i64, C.POINTER(i64)]
        L.wfst_stream_create.argtypes = [P, C.POINTER(i32)]
        L.wfst_stream_advance.argtypes = [P, P, i32, P, i32, i64, i64, P, i32, i32, P, P, i32, P,
                                          P, P]
        L.wfst_stream_finalize.argtypes = [P, P, i32, P, P, i32, P, P, P]
        L.wfst_stream_release.argtypes = [P, i32]
        L.wfst_stats.argtypes = [P, P, i32]
        L.wfst_mem_stats.argtypes = [P, P, i32]
        L.wfst_test_barrier_timeout.argtypes = [P, i64]
        L.wfst_probe_random_gather.argtypes = [P, i64, i32, i32, i32, i32, P, P]
        L.wfst_blank_skip.argtypes = [P, i32, i64, i64, i32, i32, C.c_float, P, i32, i32, P, P, P, P]
        for name in EXPORTED:
            if name not in ("wfst_last_error", "wfst_graph_free", "wfst_decoder_free"):
                getattr(L, name).restype = C.c_int
        _lib = L
        return _lib


def _check(rc):
    if rc != WFST_OK:
        raise WfstError(rc, load().wfst_last_error().decode())


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.ctypes.data_as(C.c_void_p)
    return C.c_void_p(int(a.data_ptr()))   # torch tensor


# ------------------------------------------------------------ raw C entry points

def wfst_last_error() -> str:
    return load().wfst_last_error().decode()


def wfst_graph_upload(desc: GraphDesc, device: int):
    h = C.c_void_p()
    _check(load().wfst_graph_upload(C.byref(desc), device, C.byref(h)))
    return h


def wfst_graph_info(h):
    out = np.zeros(8, np.int64)
    _check(load().wfst_graph_info(h, _ptr(out)))
    return out


def wfst_graph_free(h):
    load().wfst_graph_free(h)


def wfst_decoder_create(graph_h, params: Params, max_lanes: int, max_frames: int, caps=None):
    h = C.c_void_p()
    _check(load().wfst_decoder_create(graph_h, C.byref(params), max_lanes, max_frames,
                                      C.byref(caps) if caps is not None else None, C.byref(h)))
    return h


def wfst_decoder_free(h):
    load().wfst_decoder_free(h)


def wfst_decode(h, lp_ptr, dtype, stride_b, stride_t, lens_ptr, B, T, stream, words_ptr,
                words_cap, word_lens_ptr, scores_ptr, meta_ptr):
    _check(load().wfst_decode(h, lp_ptr, dtype, stride_b, stride_t, lens_ptr, B, T, stream,
                              words_ptr, words_cap, word_lens_ptr, scores_ptr, meta_ptr))


def wfst_decode_static(graph_h, params, lp_ptr, dtype, stride_b, stride_t, lens_ptr, B, T, stream,
                       words_ptr, words_cap, word_lens_ptr, scores_ptr, meta_ptr):
    _check(load().wfst_decode_static(graph_h, C.byref(params), lp_ptr, dtype, stride_b, stride_t,
                                     lens_ptr, B, T, stream, words_ptr, words_cap, word_lens_ptr,
                                     scores_ptr, meta_ptr))


def decode_static(graph, params, lp, lens, stream=None, words_cap=4096):
    """Offline decode through ``wfst_decode_static`` (no allocation by the
    library; ``lp`` must be a CUDA tensor on the graph's device, B <= 8)."""
    ptr, dt, sb, st, B, T = _lp_args(lp)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    words = np.zeros((B, max(words_cap, 1)), np.int32)
    wl = np.zeros(B, np.int32)
    sc = np.zeros(B, np.float64)
    meta = np.zeros((B, 3), np.int32)
    wfst_decode_static(graph.h, params, ptr, dt, sb, st, _ptr(lens), B, T, _stream(stream),
                       _ptr(words), words_cap, _ptr(wl), _ptr(sc), _ptr(meta))
    return [dict(words=words[b, : min(wl[b], words_cap)].copy(), n_words=int(wl[b]),
                 score=float(sc[b]), ok=int(meta[b, 0]), reached_final=int(meta[b, 1]),
                 overflow=int(meta[b, 2])) for b in range(B)]


def wfst_lattice_export(h, lane, out_ptr, cap):
    n = C.c_int64()
    _check(load().wfst_lattice_export(h, lane, out_ptr, cap, C.byref(n)))
    return n.value


def wfst_stream_create(h):
    ch = C.c_int32()
    _check(load().wfst_stream_create(h, C.byref(ch)))
    return ch.value


def wfst_stream_advance(h, ch_ptr, n, lp_ptr, dtype, stride_b, stride_t, lens_ptr, chunk_T,
                        want_partial, stream, words_ptr, words_cap, word_lens_ptr, scores_ptr,
                        meta_ptr):
    _check(load().wfst_stream_advance(h, ch_ptr, n, lp_ptr, dtype, stride_b, stride_t, lens_ptr,
                                      chunk_T, want_partial, stream, words_ptr, words_cap,
                                      word_lens_ptr, scores_ptr, meta_ptr))


def wfst_stream_finalize(h, ch_ptr, n, stream, words_ptr, words_cap, word_lens_ptr, scores_ptr,
                         meta_ptr):
    _check(load().wfst_stream_finalize(h, ch_ptr, n, stream, words_ptr, words_cap, word_lens_ptr,
                                       scores_ptr, meta_ptr))


def wfst_stream_release(h, ch):
    _check(load().wfst_stream_release(h, ch))


def wfst_stats(h):
    out = np.zeros(len(STAT_NAMES), np.int64)
    _check(load().wfst_stats(h, _ptr(out), len(STAT_NAMES)))
    return dict(zip(STAT_NAMES, out.tolist()))


def wfst_test_barrier_timeout(h, timeout_ns):
    _check(load().wfst_test_barrier_timeout(h, int(timeout_ns)))


def wfst_probe_random_gather(table, table_bytes, seg_bytes, grid, loads_per_thread, seed, sink, stream):
    _check(load().wfst_probe_random_gather(table, table_bytes, seg_bytes, grid, loads_per_thread, seed, sink,
                                           stream))


def wfst_mem_stats(h):
    out = np.zeros(len(MEM_NAMES), np.int64)
    _check(load().wfst_mem_stats(h, _ptr(out), len(MEM_NAMES)))
    return dict(zip(MEM_NAMES, out.tolist()))


def wfst_blank_skip(lp_ptr, dtype, stride_b, stride_t, vocab_size, blank_id, threshold, lens_ptr, B, T,
                    out_ptr, out_lens_ptr, frame_map_ptr, stream):
    _check(load().wfst_blank_skip(lp_ptr, dtype, stride_b, stride_t, vocab_size, blank_id,
                                  float(threshold), lens_ptr, B, T, out_ptr, out_lens_ptr,
                                  frame_map_ptr, stream))


def blank_skip(lp, lens, threshold=0.98, blank_id=0, stream=None):
    """Blank-skip frame pre-slicing of a CUDA [B, T, V] log-prob tensor
    (a pre-pass outside the decoder).  Returns (out [B, T, V] packed kept
    rows, out_lens [B] int32, frame_map [B, T] int32), all CUDA tensors; the
    kernels run on `stream` (torch's current stream if None)."""
    import torch
    ptr, dt, sb, st, B, T = _lp_args(lp)
    V = int(lp.shape[2])
    dev = lp.device
    lens_d = torch.as_tensor(np.ascontiguousarray(lens, dtype=np.int32)).to(dev)
    out = torch.empty((B, T, V), dtype=lp.dtype, device=dev)
    out_lens = torch.empty(B, dtype=torch.int32, device=dev)
    fmap = torch.empty((B, T), dtype=torch.int32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    wfst_blank_skip(ptr, dt, sb, st, V, int(blank_id), threshold, _ptr(lens_d), B, T, _ptr(out),
                    _ptr(out_lens), _ptr(fmap), _stream(s))
    return out, out_lens, fmap


# ------------------------------------------------------------ convenience wrappers

class Graph:
    """Device graph uploaded from a CSR dict (keys as produced by ``synth``)."""

    def __init__(self, g: dict, device: int = 0):
        keep = dict(
            row_splits=np.ascontiguousarray(g["row_splits"], dtype=np.int64),
            ilabel=np.ascontiguousarray(g["ilabel"], dtype=np.int32),
            olabel=np.ascontiguousarray(g["olabel"], dtype=np.int32),
            weight=np.ascontiguousarray(g["weight"], dtype=np.float32),
            dst=np.ascontiguousarray(g["dst"], dtype=np.int32),
            final=np.ascontiguousarray(g["final"], dtype=np.float32),
        )
        desc = GraphDesc(int(g["num_states"]), int(g["start_state"]), int(g["vocab_size"]), 0,
                         int(len(keep["ilabel"])), _ptr(keep["row_splits"]), _ptr(keep["ilabel"]),
                         _ptr(keep["olabel"]), _ptr(keep["weight"]), _ptr(keep["dst"]),
                         _ptr(keep["final"]))
        self.h = wfst_graph_upload(desc, device)
        self.device = device
        info = wfst_graph_info(self.h)
        self.num_states, self.num_arcs, self.vocab_size = int(info[0]), int(info[1]), int(info[2])
        self.has_eps, self.eps_depth, self.device_bytes = bool(info[4]), int(info[5]), int(info[6])

    def close(self):
        if getattr(self, "h", None):
            wfst_graph_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


OPT_NO_UB_SKIP = 1
OPT_NO_GROW = 4
MEM_NAMES = ["bytes", "frontier_cap", "log_cap", "lattice_cap", "path_cap", "grows", "max_frames",
             "reserved", "lazy_committed"]


def make_params(search_beam=20.0, output_beam=8.0, min_active=30, max_active=10000,
                allow_partial=True, lattice=False, streaming=False, options=0,
                gc_interval=0, lat_prune_interval=0) -> Params:
    """gc_interval > 0 turns on the winners-log GC (a GC round every
    gc_interval frames per lane; lattice must be off); lat_prune_interval > 0
    (lattice on) prunes the lattice arena every that many frames."""
    return Params(float(search_beam), float(output_beam), int(min_active), int(max_active),
                  int(bool(allow_partial)), int(bool(lattice)), int(bool(streaming)), int(options),
                  int(gc_interval), int(lat_prune_interval))


def _lp_args(lp):
    """(pointer, dtype code, stride_b, stride_t, B, T) of a [B, T, V] tensor."""
    if len(lp.shape) != 3:
        raise ValueError(f"log_probs must be [B, T, V], got shape {tuple(lp.shape)}")
    if isinstance(lp, np.ndarray):
        if lp.dtype not in (np.float32, np.float16):
            raise TypeError("log_probs must be float32 or float16")
        dt = WFST_F16 if lp.dtype == np.float16 else WFST_F32
        es = lp.itemsize
        sb, st, sv = (s // es for s in lp.strides)
    else:  # torch tensor
        import torch
        if lp.dtype not in (torch.float32, torch.float16):
            raise TypeError("log_probs must be float32 or float16")
        dt = WFST_F16 if lp.dtype == torch.float16 else WFST_F32
        sb, st, sv = lp.stride()
    if sv != 1:
        raise ValueError("log_probs must have unit stride over the vocabulary")
    return _ptr(lp), dt, int(sb), int(st), int(lp.shape[0]), int(lp.shape[1])


class Decoder:
    def __init__(self, graph: Graph, params: Params, max_lanes: int, max_frames: int,
                 caps: Capacity | None = None):
        self.graph = graph
        self.params = params
        self.max_lanes = max_lanes
        self.max_frames = max_frames
        self.h = wfst_decoder_create(graph.h, params, max_lanes, max_frames, caps)

    def close(self):
        if getattr(self, "h", None):
            wfst_decoder_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def decode(self, lp, lens, stream=None, words_cap=4096):
        """Offline decode of [B, T, V] log-probs (torch CUDA tensor or numpy).
        The call runs on ``stream``; by default, for a CUDA tensor, on torch's
        current stream of its device (where its producer most likely ran)."""
        stream = _default_stream(lp, stream)
        ptr, dt, sb, st, B, T = _lp_args(lp)
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        words = np.zeros((B, max(words_cap, 1)), np.int32)
        wl = np.zeros(B, np.int32)
        sc = np.zeros(B, np.float64)
        meta = np.zeros((B, 3), np.int32)
        wfst_decode(self.h, ptr, dt, sb, st, _ptr(lens), B, T, _stream(stream), _ptr(words),
                    words_cap, _ptr(wl), _ptr(sc), _ptr(meta))
        return [dict(words=words[b, : min(wl[b], words_cap)].copy(), n_words=int(wl[b]),
                     score=float(sc[b]), ok=int(meta[b, 0]), reached_final=int(meta[b, 1]),
                     overflow=int(meta[b, 2])) for b in range(B)]

    def lattice(self, lane: int):
        n = wfst_lattice_export(self.h, lane, None, 0)
        out = np.zeros(n, LAT_DTYPE)
        if n:
            wfst_lattice_export(self.h, lane, _ptr(out), n)
        return out

    def stats(self):
        return wfst_stats(self.h)

    def arm_barrier_timeout(self, timeout_ns=200_000_000):
        """Test hook: the next call's grid barriers cannot complete and give
        up after ``timeout_ns``; that call raises WfstError (TIMEOUT)."""
        wfst_test_barrier_timeout(self.h, timeout_ns)

    def mem_stats(self):
        return wfst_mem_stats(self.h)

    # streaming
    def stream_create(self) -> int:
        return wfst_stream_create(self.h)

    def stream_advance(self, channels, lp, chunk_lens, want_partial=True, stream=None,
                       words_cap=4096):
        ch = np.ascontiguousarray(channels, dtype=np.int32)
        n = len(ch)
        stream = _default_stream(lp, stream)
        ptr, dt, sb, st, B, T = _lp_args(lp)
        if B != n:
            raise ValueError("one log-prob row per channel")
        cl = np.ascontiguousarray(chunk_lens, dtype=np.int32)
        words = np.zeros((n, max(words_cap, 1)), np.int32)
        wl = np.zeros(n, np.int32)
        sc = np.zeros(n, np.float64)
        meta = np.zeros((n, 3), np.int32)
        wfst_stream_advance(self.h, _ptr(ch), n, ptr, dt, sb, st, _ptr(cl), T, int(want_partial),
                            _stream(stream), _ptr(words), words_cap, _ptr(wl), _ptr(sc),
                            _ptr(meta))
        if not want_partial:
            return None
        return [dict(words=words[i, : min(wl[i], words_cap)].copy(), n_words=int(wl[i]),
                     score=float(sc[i]), ok=int(meta[i, 0]), overflow=int(meta[i, 2]))
                for i in range(n)]

    def stream_finalize(self, channels, stream=None, words_cap=4096):
        ch = np.ascontiguousarray(channels, dtype=np.int32)
        n = len(ch)
        words = np.zeros((n, max(words_cap, 1)), np.int32)
        wl = np.zeros(n, np.int32)
        sc = np.zeros(n, np.float64)
        meta = np.zeros((n, 3), np.int32)
        wfst_stream_finalize(self.h, _ptr(ch), n, _stream(stream), _ptr(words), words_cap,
                             _ptr(wl), _ptr(sc), _ptr(meta))
        return [dict(words=words[i, : min(wl[i], words_cap)].copy(), n_words=int(wl[i]),
                     score=float(sc[i]), ok=int(meta[i, 0]), reached_final=int(meta[i, 1]),
                     overflow=int(meta[i, 2])) for i in range(n)]

    def stream_release(self, channel: int):
        wfst_stream_release(self.h, int(channel))


def _default_stream(lp, stream):
    """The stream a call on ``lp`` runs on when the caller names none: torch's
    current stream of a CUDA tensor's device, else the default stream."""
    if stream is not None or isinstance(lp, np.ndarray) or not getattr(lp, "is_cuda", False):
        return stream
    import torch
    return torch.cuda.current_stream(lp.device)


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return C.c_void_p(s)
    return C.c_void_p(int(s.cuda_stream))   # torch.cuda.Stream


class StreamingSearch:
    """One stream decoded through a channel of a streaming ``Decoder``, with
    the caller-side overflow policy of the page "GPU WFST Beam-Search
    Decoder" (§7 overflow handling, §8.1): a channel whose chunk comes back
    with a capacity overflow bit set (winners log or frontier: the channel's
    search state is incomplete) cannot be trusted from then on, so it is
    abandoned, the hypothesis it gave before that chunk is kept as a finished
    prefix, and the chunk runs once more on a newly opened channel.  The new
    channel starts its search from scratch, so hypotheses that spanned the
    overflow are gone, but no frame after it is skipped.

    ``feed`` returns the words so far (prefix + the channel's partial
    hypothesis); ``finish`` runs the final step and releases the channel.
    Scores are the current channel's (they do not include the prefix)."""

    def __init__(self, decoder, words_cap=4096):
        self.d = decoder
        self.words_cap = words_cap
        self.prefix = []
        self.last_words = []
        self.restarts = 0
        self.ch = self._open()

    def _open(self):
        ch = self.d.stream_create()
        if ch < 0:
            raise RuntimeError("StreamingSearch: every channel of the decoder is busy")
        return ch

    def _advance(self, lp_chunk, length):
        return self.d.stream_advance([self.ch], lp_chunk[None], [int(length)], want_partial=True,
                                     words_cap=self.words_cap)[0]

    def feed(self, lp_chunk, length=None):
        """Decode one chunk ([T_c, V] log-probs; ``length`` frames of it, all
        by default) and return the words so far."""
        length = int(lp_chunk.shape[0]) if length is None else int(length)
        r = self._advance(lp_chunk, length)
        if r["overflow"] & (OVF_ARENA | OVF_KEPT):
            self.d.stream_release(self.ch)
            self.prefix += list(self.last_words)
            self.last_words = []
            self.restarts += 1
            self.ch = self._open()
            r = self._advance(lp_chunk, length)
        # only a result whose search state is complete may later become the
        # finished prefix (a retried chunk can overflow again: it is reported)
        if r["ok"] and not (r["overflow"] & (OVF_ARENA | OVF_KEPT)):
            self.last_words = list(r["words"])
        return dict(words=self.prefix + list(r["words"]), score=r["score"], ok=r["ok"],
                    overflow=r["overflow"], restarts=self.restarts)

    def finish(self):
        """Final step of the stream; the channel returns to the decoder."""
        f = self.d.stream_finalize([self.ch], words_cap=self.words_cap)[0]
        self.d.stream_release(self.ch)
        self.ch = -1
        words = self.prefix + (list(f["words"]) if f["ok"] else list(self.last_words))
        return dict(words=words, score=f["score"], ok=f["ok"], reached_final=f["reached_final"],
                    overflow=f["overflow"], restarts=self.restarts)
