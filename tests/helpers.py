"""Independent reference computations used to pin the oracle.

Nothing here imports the oracle or the CUDA decoder: these are brute-force
path enumeration and a dense (unpruned) Viterbi written directly from the
definition of the decoding problem (best-scoring path through the graph,
end = (score + weight) + log_prob, fp32 arithmetic).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
INF_BEAM = dict(search_beam=1e30, min_active=0, max_active=2**31 - 1)


def f32(x):
    return np.float32(x)


def arcs_of(g, s):
    return range(int(g["row_splits"][s]), int(g["row_splits"][s + 1]))


def enumerate_paths(g, lp, T):
    """All complete paths of a tiny graph over T frames.

    Returns a list of (total fp32 score, final state, arcs, transitions),
    where transitions are (frame, arc id, kind) with kind in {"emit", "eps",
    "final"} and the frame of an emitting arc is the frame it consumes.
    """
    il, w, dst, fin = g["ilabel"], g["weight"], g["dst"], g["final"]
    A = len(il)

    def eps_ext(state, score, arcs, trans, frame):
        out = [(state, score, arcs, trans)]
        for a in arcs_of(g, state):
            if il[a] < 0:
                e = f32(score + w[a])
                out += eps_ext(int(dst[a]), e, arcs + [a], trans + [(frame, a, "eps")], frame)
        return out

    front = eps_ext(int(g["start_state"]), f32(0.0), [], [], 0)
    for t in range(T):
        new = []
        for (s, sc, arcs, trans) in front:
            for a in arcs_of(g, s):
                if il[a] >= 0:
                    e = f32(f32(sc + w[a]) + lp[t][il[a]])
                    new += eps_ext(int(dst[a]), e, arcs + [a], trans + [(t, a, "emit")], t + 1)
        front = new
    complete = []
    for (s, sc, arcs, trans) in front:
        if fin[s] > -np.inf:
            complete.append((f32(sc + fin[s]), s, arcs, trans + [(T, A + s, "final")]))
    return complete, front


def best_path(complete):
    """Max score; ties: lowest final state, then reverse-lexicographically
    smallest arc sequence (what per-token lowest-arc-id recombination picks
    when every sum is exact)."""
    if not complete:
        return None
    top = max(p[0] for p in complete)
    cands = [p for p in complete if p[0] == top]
    cands.sort(key=lambda p: (p[1], tuple(reversed(p[2]))))
    return cands[0]


def dense_viterbi(g, lp, T):
    """Unpruned Viterbi over every state (epsilon-free graphs), numpy fp32.
    Ties at a state keep the lowest arc id; final ties keep the lowest state."""
    N = int(g["num_states"])
    rs = g["row_splits"]
    src = np.repeat(np.arange(N), np.diff(rs)).astype(np.int64)
    il, w, dst, fin = g["ilabel"], g["weight"].astype(F32), g["dst"].astype(np.int64), g["final"]
    assert (il >= 0).all(), "dense_viterbi handles epsilon-free graphs"
    ids = np.arange(len(il), dtype=np.int64)
    score = np.full(N, -np.inf, dtype=F32)
    score[int(g["start_state"])] = 0.0
    bps = []
    for t in range(T):
        ok = score[src] > -np.inf
        e = (score[src] + w) + lp[t][il].astype(F32)
        e = e.astype(F32)
        new = np.full(N, -np.inf, dtype=F32)
        np.maximum.at(new, dst[ok], e[ok])
        best = ok & (e == new[dst])
        bp = np.full(N, np.iinfo(np.int64).max, dtype=np.int64)
        np.minimum.at(bp, dst[best], ids[best])
        bps.append(bp)
        score = new
    fe = (score + fin.astype(F32)).astype(F32)
    if not np.isfinite(fe).any():
        return None
    s = int(np.argmax(fe))          # first maximum = lowest state
    arcs = []
    for t in range(T - 1, -1, -1):
        a = int(bps[t][s])
        arcs.append(a)
        s = int(src[a])
    return float(fe.max()), arcs[::-1]


def words_of(g, arcs):
    ol = g["olabel"]
    return [int(ol[a]) for a in arcs if ol[a] != 0]
