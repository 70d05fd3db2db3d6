"""Seeded synthetic inputs shared by the CPU oracle and the CUDA decoder.

This module only draws random graphs and log-posteriors; it holds none of the
decoder's arithmetic.  Both sides of every parity test consume the exact same
arrays produced here.

Workloads (one per decoding regime the GPU WFST decoder page covers):

  0 tiny      B=1,   T=50,  V=32,   200 states, fp32, lattice on
  1 mid       B=16,  T=200, V=500,  50k states / ~300k arcs, fp32
  2 hlg       B=64,  T=500, V=5000, 2M states / 10M arcs, power-law degree, fp16
  3 tlg       B=32,  T=300, V=5000, 1M states / 6M arcs, 20% epsilon arcs, fp32
  4 stream    128 lanes, T<=800 in 16-frame chunks, workload 2's graph, fp16,
              lattice on
  5 hlg_zipf15  workload 2 with the degree law taken literally: non-blank
              out-degree Zipf(s = 1.5) capped at 2000 (mean 34.3, ~70M arcs
              on 2M states), reported beside workload 2 as a stress case

Graph conventions (the decoder's C ABI):
  * CSR by source state: ``row_splits`` int64 [N+1], per-arc ``ilabel`` int32
    (-1 = epsilon, 0 = blank, 1..V-1 = tokens), ``olabel`` int32 (0 = no word),
    ``weight`` float32 (log-semiring score, higher is better), ``dst`` int32;
    per-state ``final`` float32 (-inf = not final); start state 0.
  * Within a state: the blank self-loop (ilabel 0, olabel 0, weight 0) first,
    then the non-blank emitting arcs in draw order, then epsilon arcs.

Random streams: the graph of workload ``i`` draws from
``default_rng([seed_i, 0])`` in the order degrees/sources, destinations,
ilabels, word mask, words, weights, finals; lane ``b``'s log-posteriors draw
from ``default_rng([seed_i, 1, b])`` (logits, then the blank-boost mask), so
any lane can be regenerated alone; lengths draw from ``default_rng([seed_i,
2])``.  Log-posteriors are log_softmax of N(0, 2^2) logits in float64 with +3
added to the blank logit in 70% of frames, then cast to float32 or float16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "make_graph", "make_log_probs",
    "make_lane_log_probs", "make_lens", "graph_from_arcs", "zipf_exponent",
]


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    T: int
    V: int
    dtype: str                 # "f32" | "f16"
    seed: int
    search_beam: float
    output_beam: float
    min_active: int
    max_active: int
    lattice: bool
    streaming: bool = False
    chunk: int = 0
    graph: dict = field(default_factory=dict)


WORKLOADS = {
    0: Workload(0, "tiny", B=1, T=50, V=32, dtype="f32", seed=0,
                search_beam=20.0, output_beam=8.0, min_active=30, max_active=1000,
                lattice=True,
                graph=dict(kind="uniform", N=200, deg=4, word_max=100, p_word=0.2,
                           w_kind="uniform", w_scale=3.0)),
    1: Workload(1, "mid", B=16, T=200, V=500, dtype="f32", seed=1,
                search_beam=20.0, output_beam=8.0, min_active=30, max_active=7000,
                lattice=False,
                graph=dict(kind="poisson", N=50_000, lam=5.0, word_max=20_000, p_word=0.15,
                           w_kind="uniform", w_scale=5.0)),
    2: Workload(2, "hlg", B=64, T=500, V=5000, dtype="f16", seed=2,
                search_beam=20.0, output_beam=8.0, min_active=200, max_active=10_000,
                lattice=False,
                graph=dict(kind="zipf", N=2_000_000, A=10_000_000, cap=2000, mean_nb=4.0,
                           word_max=200_000, p_word=0.1, w_kind="exp")),
    3: Workload(3, "tlg", B=32, T=300, V=5000, dtype="f32", seed=3,
                search_beam=16.0, output_beam=8.0, min_active=30, max_active=7000,
                lattice=False,
                graph=dict(kind="tlg", N=1_000_000, n_emit=3_800_000, n_eps=1_200_000,
                           word_max=100_000, p_word=0.1, w_kind="uniform", w_scale=4.0)),
    4: Workload(4, "stream", B=128, T=800, V=5000, dtype="f16", seed=4,
                search_beam=16.0, output_beam=10.0, min_active=200, max_active=10_000,
                lattice=True, streaming=True, chunk=16,
                graph=dict(kind="same_as", of=2)),
    5: Workload(5, "hlg_zipf15", B=64, T=500, V=5000, dtype="f16", seed=5,
                search_beam=20.0, output_beam=8.0, min_active=200, max_active=10_000,
                lattice=False,
                graph=dict(kind="zipf", N=2_000_000, s=1.5, cap=2000,
                           word_max=200_000, p_word=0.1, w_kind="exp")),
}


def workload(i: int) -> Workload:
    return WORKLOADS[i]


# --------------------------------------------------------------------------
# graphs
# --------------------------------------------------------------------------

def graph_from_arcs(N, V, src, dst, ilabel, olabel, weight, final, start=0):
    """Assemble a CSR graph dict from arc columns (stable-sorted by source)."""
    src = np.asarray(src, dtype=np.int64)
    order = np.argsort(src, kind="stable")
    counts = np.bincount(src, minlength=N)
    row_splits = np.zeros(N + 1, dtype=np.int64)
    np.cumsum(counts, out=row_splits[1:])
    return dict(
        num_states=int(N), start_state=int(start), vocab_size=int(V),
        num_arcs=int(len(src)),
        row_splits=row_splits,
        ilabel=np.ascontiguousarray(np.asarray(ilabel, dtype=np.int32)[order]),
        olabel=np.ascontiguousarray(np.asarray(olabel, dtype=np.int32)[order]),
        weight=np.ascontiguousarray(np.asarray(weight, dtype=np.float32)[order]),
        dst=np.ascontiguousarray(np.asarray(dst, dtype=np.int32)[order]),
        final=np.ascontiguousarray(np.asarray(final, dtype=np.float32)),
    )


def zipf_exponent(mean: float, cap: int) -> float:
    """Exponent s of a Zipf law on [1, cap] whose mean is ``mean`` (bisection)."""
    k = np.arange(1, cap + 1, dtype=np.float64)

    def m(s):
        p = k ** (-s)
        return float((k * p).sum() / p.sum())

    lo, hi = 1.0001, 6.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if m(mid) > mean:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _weights(rng, n, spec):
    if spec["w_kind"] == "uniform":
        return -rng.uniform(0.0, spec["w_scale"], size=n)
    if spec["w_kind"] == "exp":
        return -rng.exponential(1.0, size=n)
    raise ValueError(spec["w_kind"])


def _finals(rng, N):
    final = np.full(N, -np.inf, dtype=np.float32)
    final[rng.permutation(N)[: N // 10]] = 0.0
    return final


def _with_blank_loops(N, V, nb_src, nb_dst, nb_il, nb_ol, nb_w, final,
                      eps_src=None, eps_dst=None, eps_ol=None, eps_w=None):
    """Per state: blank self-loop, then emitting arcs (draw order), then epsilon arcs."""
    loops = np.arange(N, dtype=np.int64)
    parts_src = [loops, np.asarray(nb_src, dtype=np.int64)]
    parts_dst = [loops, nb_dst]
    parts_il = [np.zeros(N, np.int32), nb_il]
    parts_ol = [np.zeros(N, np.int32), nb_ol]
    parts_w = [np.zeros(N, np.float32), np.asarray(nb_w, np.float32)]
    # class key keeps loop < emitting < epsilon inside each state under the
    # stable sort by source state
    cls = [np.zeros(N, np.int8), np.ones(len(nb_src), np.int8)]
    if eps_src is not None:
        parts_src.append(np.asarray(eps_src, dtype=np.int64))
        parts_dst.append(eps_dst)
        parts_il.append(np.full(len(eps_src), -1, np.int32))
        parts_ol.append(eps_ol)
        parts_w.append(np.asarray(eps_w, np.float32))
        cls.append(np.full(len(eps_src), 2, np.int8))
    src = np.concatenate(parts_src)
    key = src * 3 + np.concatenate(cls)
    order = np.argsort(key, kind="stable")
    counts = np.bincount(src, minlength=N)
    row_splits = np.zeros(N + 1, dtype=np.int64)
    np.cumsum(counts, out=row_splits[1:])
    return dict(
        num_states=int(N), start_state=0, vocab_size=int(V), num_arcs=int(len(src)),
        row_splits=row_splits,
        ilabel=np.ascontiguousarray(np.concatenate(parts_il).astype(np.int32)[order]),
        olabel=np.ascontiguousarray(np.concatenate(parts_ol).astype(np.int32)[order]),
        weight=np.ascontiguousarray(np.concatenate(parts_w).astype(np.float32)[order]),
        dst=np.ascontiguousarray(np.concatenate(parts_dst).astype(np.int32)[order]),
        final=final,
    )


def _word_labels(rng, n, spec):
    mask = rng.random(n) < spec["p_word"]
    words = rng.integers(1, spec["word_max"] + 1, size=n)
    return np.where(mask, words, 0).astype(np.int32)


def _fit_total(deg, total, lo, hi):
    """Trim or pad the LAST states' degrees (within [lo, hi]) to hit ``total``."""
    deg = deg.copy()
    diff = int(total - deg.sum())
    i = len(deg) - 1
    while diff != 0 and i >= 0:
        if diff > 0:
            step = min(diff, hi - int(deg[i]))
        else:
            step = -min(-diff, int(deg[i]) - lo)
        deg[i] += step
        diff -= step
        i -= 1
    if diff != 0:
        raise ValueError("cannot reach the requested arc count")
    return deg


def make_graph(i: int) -> dict:
    wl = WORKLOADS[i]
    spec = wl.graph
    if spec["kind"] == "same_as":
        return make_graph(spec["of"])
    rng = np.random.default_rng([wl.seed, 0])
    V = wl.V
    N = spec["N"]
    if spec["kind"] in ("uniform", "poisson", "zipf"):
        if spec["kind"] == "uniform":
            deg = np.full(N, spec["deg"], dtype=np.int64)
        elif spec["kind"] == "poisson":
            deg = rng.poisson(spec["lam"], size=N).astype(np.int64)
        else:
            # the exponent as given, or solved for the requested mean (and the
            # total then trimmed to the requested arc count)
            s = spec["s"] if "s" in spec else zipf_exponent(spec["mean_nb"], spec["cap"])
            k = np.arange(1, spec["cap"] + 1, dtype=np.float64)
            cdf = np.cumsum(k ** (-s))
            cdf /= cdf[-1]
            deg = np.searchsorted(cdf, rng.random(N), side="right").astype(np.int64) + 1
            deg = np.minimum(deg, spec["cap"])
            if "A" in spec:
                deg = _fit_total(deg, spec["A"] - N, 1, spec["cap"])
        n_nb = int(deg.sum())
        nb_src = np.repeat(np.arange(N, dtype=np.int64), deg)
        nb_dst = rng.integers(0, N, size=n_nb).astype(np.int32)
        nb_il = rng.integers(1, V, size=n_nb).astype(np.int32)
        nb_ol = _word_labels(rng, n_nb, spec)
        nb_w = _weights(rng, n_nb, spec)
        final = _finals(rng, N)
        return _with_blank_loops(N, V, nb_src, nb_dst, nb_il, nb_ol, nb_w, final)
    if spec["kind"] == "tlg":
        ne, nz = spec["n_emit"], spec["n_eps"]
        em_src = rng.integers(0, N, size=ne)
        em_dst = rng.integers(0, N, size=ne).astype(np.int32)
        em_il = rng.integers(1, V, size=ne).astype(np.int32)
        a = rng.integers(0, N, size=nz)
        b = rng.integers(0, N - 1, size=nz)
        b = b + (b >= a)                       # distinct from a
        eps_src = np.minimum(a, b)
        eps_dst = np.maximum(a, b).astype(np.int32)   # src < dst: acyclic
        ol = _word_labels(rng, ne + nz, spec)
        w = _weights(rng, ne + nz, spec)
        final = _finals(rng, N)
        return _with_blank_loops(N, V, em_src, em_dst, em_il, ol[:ne], w[:ne], final,
                                 eps_src, eps_dst, ol[ne:], w[ne:])
    raise ValueError(spec["kind"])


# --------------------------------------------------------------------------
# log-posteriors and lengths
# --------------------------------------------------------------------------

def _log_softmax64(x):
    m = x.max(axis=-1, keepdims=True)
    z = x - m
    return z - np.log(np.exp(z).sum(axis=-1, keepdims=True))


def make_lane_log_probs(i: int, b: int, T: int | None = None, V: int | None = None,
                        seed: int | None = None, dtype: str | None = None):
    """Lane ``b`` of workload ``i``: [T, V] peaky-CTC log-posteriors."""
    wl = WORKLOADS[i]
    T = wl.T if T is None else T
    V = wl.V if V is None else V
    seed = wl.seed if seed is None else seed
    dtype = wl.dtype if dtype is None else dtype
    rng = np.random.default_rng([seed, 1, b])
    logits = rng.normal(0.0, 2.0, size=(T, V))
    boost = rng.random(T) < 0.7
    logits[boost, 0] += 3.0
    lp = _log_softmax64(logits)
    return lp.astype(np.float16 if dtype == "f16" else np.float32)


def make_log_probs(i: int, lanes=None, T: int | None = None):
    wl = WORKLOADS[i]
    lanes = range(wl.B) if lanes is None else lanes
    return np.stack([make_lane_log_probs(i, b, T=T) for b in lanes])


def make_lens(i: int) -> np.ndarray:
    wl = WORKLOADS[i]
    if wl.streaming:
        rng = np.random.default_rng([wl.seed, 2])
        return rng.integers(200, 801, size=wl.B).astype(np.int32)
    return np.full(wl.B, wl.T, dtype=np.int32)


def dyadic_log_probs(rng, T, V, lo=-8.0, hi=0.0, step=0.125):
    """Log-probs that are multiples of 1/8 (every fp32 sum of a few is exact)."""
    n = int(round((hi - lo) / step))
    return (lo + step * rng.integers(0, n + 1, size=(T, V))).astype(np.float32)


def random_tiny_graph(rng, N, V, max_deg=3, p_eps=0.0, p_final=0.5, dyadic=True,
                      p_word=0.5, word_max=9, allow_empty=False, relabel=False):
    """A small random graph for brute-force checks (epsilon arcs go to higher
    state ids only, so the epsilon subgraph is acyclic).  With ``relabel`` the
    states are renamed by a random permutation afterwards (the start state
    too), so that an epsilon-topological order no longer follows the ids."""
    src, dst, il, ol, w = [], [], [], [], []
    for s in range(N):
        deg = int(rng.integers(0 if allow_empty else 1, max_deg + 1))
        for _ in range(deg):
            eps = p_eps > 0 and s < N - 1 and rng.random() < p_eps
            if eps:
                d = int(rng.integers(s + 1, N))
                lab = -1
            else:
                d = int(rng.integers(0, N))
                lab = int(rng.integers(0, V))
            src.append(s)
            dst.append(d)
            il.append(lab)
            ol.append(int(rng.integers(1, word_max + 1)) if rng.random() < p_word else 0)
            if dyadic:
                w.append(-0.125 * int(rng.integers(0, 33)))
            else:
                w.append(-float(rng.uniform(0, 4)))
    final = np.where(rng.random(N) < p_final,
                     (-0.125 * rng.integers(0, 9, size=N)) if dyadic else -rng.uniform(0, 2, size=N),
                     -np.inf).astype(np.float32)
    if not np.isfinite(final).any():
        final[int(rng.integers(0, N))] = 0.0
    if not relabel:
        return graph_from_arcs(N, V, np.array(src, dtype=np.int64), dst, il, ol, w, final)
    perm = rng.permutation(N)
    final_p = np.empty_like(final)
    final_p[perm] = final
    return graph_from_arcs(N, V, perm[np.array(src, dtype=np.int64)], perm[np.array(dst, dtype=np.int64)],
                           il, ol, w, final_p, start=int(perm[0]))
