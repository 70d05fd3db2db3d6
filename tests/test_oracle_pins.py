"""Pins of the CPU oracle against facts that do not come from the oracle.

* brute-force path enumeration on tiny graphs (with and without epsilon arcs)
  at an unbounded beam: the oracle's score equals the best path's score, and
  with dyadic data (exact fp32 sums) its arcs equal the tie-broken best path;
* an unpruned dense Viterbi (numpy) at an unbounded beam on workloads 0/1;
* closed forms: a one-state graph (score = sum of per-frame maxima, path =
  per-frame argmax) and a linear chain (the forced path);
* hand-derived values of the dynamic-beam rule and of the strict admission
  test (tests/golden/*.json, each citing the page section it follows);
* the final-step rules (allow_partial, no final state);
* lattice: brute-force best path through every record decides keep/drop;
* streaming: chunking invariance and equality with the offline decode when the
  last-frames rule cannot fire.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from tests import helpers as H

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _p(**kw):
    base = dict(search_beam=20.0, output_beam=8.0, min_active=30, max_active=10000,
                allow_partial=True, lattice=False)
    base.update(kw)
    return oracle.params(**base)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed", range(40))
@pytest.mark.parametrize("p_eps,relabel", [(0.0, False), (0.35, False), (0.5, True)])
def test_bruteforce_dyadic_exact_path(seed, p_eps, relabel):
    """Relabelled graphs put epsilon arcs from higher to lower state ids, so a
    closure that visits states in id order instead of epsilon-topological
    order (§5.5) relaxes some state before its score is final."""
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(2, 7)) + (3 if relabel else 0)
    V = int(rng.integers(2, 5))
    T = int(rng.integers(1, 5))
    g = synth.random_tiny_graph(rng, N, V, max_deg=3, p_eps=p_eps, dyadic=True, relabel=relabel)
    lp = synth.dyadic_log_probs(rng, T, V)
    complete, _ = H.enumerate_paths(g, lp, T)
    G = oracle.Graph(g)
    r = oracle.decode(G, lp, T, _p(**H.INF_BEAM, allow_partial=False))
    bp = H.best_path(complete)
    if bp is None:
        assert r["ok"] == 0
        return
    assert r["ok"] == 1 and r["reached_final"] == 1
    assert np.float32(r["score"]) == bp[0]
    assert list(r["arcs"]) == list(bp[2])
    assert list(r["words"]) == H.words_of(g, bp[2])


@pytest.mark.parametrize("seed", range(30))
def test_bruteforce_float_score(seed):
    """Non-dyadic data: the best score is still exactly the brute-force max
    (fp32 addition is monotone, so per-state maxima compose)."""
    rng = np.random.default_rng(5000 + seed)
    N, V, T = int(rng.integers(2, 7)), int(rng.integers(2, 5)), int(rng.integers(1, 5))
    g = synth.random_tiny_graph(rng, N, V, max_deg=3, p_eps=0.3 if seed % 2 else 0.0,
                                dyadic=False)
    lp = np.log(rng.dirichlet(np.ones(V), size=T)).astype(np.float32)
    complete, _ = H.enumerate_paths(g, lp, T)
    r = oracle.decode(oracle.Graph(g), lp, T, _p(**H.INF_BEAM, allow_partial=False))
    bp = H.best_path(complete)
    if bp is None:
        assert r["ok"] == 0
    else:
        assert np.float32(r["score"]) == bp[0]


# ---------------------------------------------------------------- dense Viterbi

@pytest.mark.parametrize("wl_index,lane,T", [(0, 0, 50), (1, 0, 60), (1, 3, 60)])
def test_dense_viterbi_unbounded_beam(wl_index, lane, T):
    g = synth.make_graph(wl_index)
    lp = synth.make_lane_log_probs(wl_index, lane, T=T).astype(np.float32)
    ref = H.dense_viterbi(g, lp, T)
    r = oracle.decode(oracle.Graph(g), lp, T, _p(**H.INF_BEAM))
    assert ref is not None and r["reached_final"] == 1
    assert np.float32(r["score"]) == np.float32(ref[0])
    assert list(r["arcs"]) == ref[1]


# ---------------------------------------------------------------- closed forms

def test_one_state_closed_form():
    rng = np.random.default_rng(7)
    V, T = 12, 40
    # one state, V self-loops ordered by ilabel, olabel = ilabel
    g = synth.graph_from_arcs(1, V, np.zeros(V, np.int64), np.zeros(V, np.int32),
                              np.arange(V), np.arange(V), np.zeros(V), np.zeros(1))
    lp = np.log(rng.dirichlet(np.ones(V), size=T)).astype(np.float32)
    lp[5, 3] = lp[5, 7] = lp[5].max() + np.float32(0.5)   # an exact tie -> lower label
    r = oracle.decode(oracle.Graph(g), lp, T, _p(search_beam=5.0))
    s = np.float32(0.0)
    for t in range(T):
        s = np.float32(s + lp[t].max())
    assert np.float32(r["score"]) == s
    assert list(r["arcs"]) == [int(np.argmax(lp[t])) for t in range(T)]
    assert r["arcs"][5] == 3
    assert list(r["words"]) == [int(np.argmax(lp[t])) for t in range(T) if np.argmax(lp[t]) != 0]


def test_linear_chain_forced_path_and_partial():
    rng = np.random.default_rng(11)
    T, V = 25, 6
    N = T + 1
    src = np.arange(T)
    il = rng.integers(1, V, size=T)
    w = -rng.uniform(0, 2, size=T).astype(np.float32)
    fin = np.full(N, -np.inf, np.float32)
    fin[T] = np.float32(-0.25)
    g = synth.graph_from_arcs(N, V, src, src + 1, il, np.arange(1, T + 1), w, fin)
    lp = np.log(rng.dirichlet(np.ones(V), size=T)).astype(np.float32)
    s = np.float32(0.0)
    for t in range(T):
        s = np.float32(np.float32(s + w[t]) + lp[t, il[t]])
    G = oracle.Graph(g)
    r = oracle.decode(G, lp, T, _p(min_active=0))
    assert r["reached_final"] == 1 and np.float32(r["score"]) == np.float32(s + fin[T])
    assert list(r["arcs"]) == list(range(T)) and list(r["words"]) == list(range(1, T + 1))
    # one frame short: no final state in the frontier -> allow_partial result
    s2 = np.float32(0.0)
    for t in range(T - 1):
        s2 = np.float32(np.float32(s2 + w[t]) + lp[t, il[t]])
    r2 = oracle.decode(G, lp, T - 1, _p(min_active=0))
    assert r2["ok"] == 1 and r2["reached_final"] == 0 and np.float32(r2["score"]) == s2
    assert list(r2["words"]) == list(range(1, T))
    r3 = oracle.decode(G, lp, T - 1, _p(min_active=0, allow_partial=False))
    assert r3["ok"] == 0 and len(r3["words"]) == 0 and r3["score"] == -np.inf


# ---------------------------------------------------------------- golden rules

def _fan_graph():
    # state 0: blank loop + arcs to 1..5 (ilabel 1); states 1..5: blank loop
    src = [0] + [0] * 5 + list(range(1, 6))
    dst = [0] + list(range(1, 6)) + list(range(1, 6))
    il = [0] + [1] * 5 + [0] * 5
    return synth.graph_from_arcs(6, 2, np.array(src), dst, il, [0] * 11, [0.0] * 11,
                                 np.zeros(6, np.float32))


def _dead_end_graph():
    # state 0: one arc (ilabel 1) to state 1; state 1: no arcs
    return synth.graph_from_arcs(2, 2, np.array([0]), [1], [1], [0], [0.0], np.zeros(2, np.float32))


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "beam_rule.json")))["cases"],
                         ids=lambda c: c["name"])
def test_golden_dynamic_beam(case):
    spec = json.load(open(os.path.join(GOLD, "beam_rule.json")))
    g = _dead_end_graph() if case.get("graph") == "dead_end" else _fan_graph()
    T = case["T"]
    lp = np.full((T, 2), -1.0, np.float32)
    p = _p(search_beam=spec["search_beam"], min_active=case["min_active"],
           max_active=case["max_active"])
    d = oracle.Decoder(oracle.Graph(g), p, None if case.get("streaming") else T)
    d.advance(lp)
    tr = d.trace()
    np.testing.assert_allclose(tr["beam"], case["beam"], rtol=2e-6)
    assert list(tr["n"]) == case["n"]


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "admission_boundary.json")))["cases"],
                         ids=lambda c: c["name"])
def test_golden_admission_boundary(case):
    spec = json.load(open(os.path.join(GOLD, "admission_boundary.json")))
    src, dst, il, ol, w = (list(c) for c in zip(*case["arcs"]))
    N = case["num_states"]
    fin = np.zeros(N, np.float32) if case["finals"] is None else \
        np.array([-np.inf if f is None else f for f in case["finals"]], np.float32)
    g = synth.graph_from_arcs(N, 2, np.array(src), dst, il, ol, w, fin)
    lp = np.full((spec["T"], 2), -0.5, np.float32)
    p = _p(search_beam=spec["search_beam"], min_active=spec["min_active"],
           max_active=spec["max_active"], lattice=True, output_beam=1e30)
    d = oracle.Decoder(oracle.Graph(g), p, spec["T"])
    d.advance(lp)
    tr = d.trace()
    assert tr["max_end"][0] == np.float32(case["max_end"])
    assert tr["cutoff"][0] == np.float32(case["cutoff"])
    r = d.finalize()
    recs = d.lattice(kept=False)
    assert sorted(recs[recs["flags"] == 0]["dst_state"].tolist()) == case["emit_states"]
    assert sorted(recs[recs["flags"] == oracle.REC_EPS]["dst_state"].tolist()) == case["eps_states"]
    assert np.float32(r["score"]) == np.float32(case["score"]) and list(r["words"]) == case["words"]


_NONMONO = json.load(open(os.path.join(GOLD, "beam_not_monotone.json")))


@pytest.mark.parametrize("case", _NONMONO["cases"], ids=lambda c: f"beam {c['search_beam']:g}")
def test_golden_best_score_is_not_monotone_in_the_beam(case):
    """A wider beam admits a branch whose higher maximum at the next step
    prunes the prefix of the narrower search's best path: beam 1 gives -5.5,
    beam 2 gives -13, an unbounded beam -5.5 again (hand-derived in the
    fixture).  A search that pruned against a per-token or stale maximum
    would not reproduce it."""
    spec = _NONMONO
    src, dst, il, ol, w = (list(c) for c in zip(*spec["arcs"]))
    N = spec["num_states"]
    fin = np.array([-np.inf if f is None else f for f in spec["finals"]], np.float32)
    g = synth.graph_from_arcs(N, 2, np.array(src), dst, il, ol, w, fin)
    p = _p(search_beam=case["search_beam"], min_active=spec["min_active"],
           max_active=spec["max_active"], allow_partial=False)
    d = oracle.Decoder(oracle.Graph(g), p, None)
    d.advance(np.full((spec["T"], 2), -0.5, np.float32))
    r = d.finalize()
    assert r["ok"] == 1 and r["reached_final"] == case["reached_final"]
    assert np.float32(r["score"]) == np.float32(case["score"])
    assert list(r["words"]) == case["words"]


@pytest.mark.parametrize("seed", range(40))
def test_pruned_search_never_beats_the_unpruned_optimum(seed):
    """What does hold for every beam: a pruned search returns a real path, so
    its score is at most the unpruned optimum, and if it reaches a final
    state so does the unpruned search.  (The best score is not monotone in
    the beam; see the golden case above.)"""
    rng = np.random.default_rng(9000 + seed)
    N, V, T = int(rng.integers(3, 30)), int(rng.integers(2, 6)), int(rng.integers(2, 12))
    g = synth.random_tiny_graph(rng, N, V, max_deg=4, p_eps=0.3 if seed % 2 else 0.0, dyadic=False)
    lp = np.log(rng.dirichlet(np.ones(V), size=T)).astype(np.float32)
    OG = oracle.Graph(g)
    best = oracle.decode(OG, lp, T, _p(**H.INF_BEAM, allow_partial=False))
    for beam in (0.5, 1.0, 2.0, 4.0, 8.0):
        r = oracle.decode(OG, lp, T, _p(search_beam=beam, min_active=0, max_active=2**31 - 1,
                                        allow_partial=False))
        if r["ok"]:
            assert best["ok"] == 1 and r["score"] <= best["score"], (beam, r["score"], best["score"])


# ---------------------------------------------------------------- lattice

@pytest.mark.parametrize("seed", range(30))
@pytest.mark.parametrize("p_eps", [0.0, 0.3])
def test_lattice_keep_matches_bruteforce(seed, p_eps):
    """Unbounded search beam: every reachable transition is persisted once;
    a record is kept iff the best complete path through it is within
    output_beam of the best path (dyadic data, exact sums)."""
    rng = np.random.default_rng(9000 + seed)
    N, V, T = int(rng.integers(2, 6)), int(rng.integers(2, 4)), int(rng.integers(1, 4))
    g = synth.random_tiny_graph(rng, N, V, max_deg=3, p_eps=p_eps, dyadic=True)
    lp = synth.dyadic_log_probs(rng, T, V, lo=-4.0)
    out_beam = float(rng.choice([0.0, 0.5, 1.0, 2.5, 1e30]))
    complete, _ = H.enumerate_paths(g, lp, T)
    d = oracle.Decoder(oracle.Graph(g), _p(**H.INF_BEAM, allow_partial=False, lattice=True,
                                           output_beam=out_beam), T)
    d.advance(lp)
    r = d.finalize()
    bp = H.best_path(complete)
    if bp is None:
        assert r["ok"] == 0 and len(d.lattice()) == 0
        return
    thr = np.float32(bp[0] - np.float32(out_beam))
    through = {}
    for tot, _, _, trans in complete:
        for (fr, a, kind) in trans:
            k = (fr, a)
            if k not in through or tot > through[k]:
                through[k] = tot
    allr = d.lattice(kept=False)
    kept = d.lattice(kept=True)
    got = {(int(x["t"]), int(x["arc_id"])) for x in kept}
    want = {k for (k, v) in through.items() if v >= thr}
    # only persisted transitions can be kept; unreachable-to-final ones are dropped
    persisted = {(int(x["t"]), int(x["arc_id"])) for x in allr}
    assert want <= persisted
    assert got == want
    # the 1-best path's transitions are all kept
    assert {(fr, a) for (fr, a, _) in bp[3]} <= got


def test_lattice_record_scores_and_flags():
    rng = np.random.default_rng(3)
    g = synth.random_tiny_graph(rng, 5, 3, max_deg=3, p_eps=0.3, dyadic=True)
    lp = synth.dyadic_log_probs(rng, 3, 3, lo=-4.0)
    d = oracle.Decoder(oracle.Graph(g), _p(**H.INF_BEAM, lattice=True, output_beam=1e30), 3)
    d.advance(lp)
    d.finalize()
    A = len(g["ilabel"])
    for x in d.lattice(kept=False):
        a = int(x["arc_id"])
        if x["flags"] & oracle.REC_FINAL:
            assert a == A + x["src_state"] and x["score"] == g["final"][x["src_state"]]
        elif x["flags"] & oracle.REC_REDIRECT:
            assert a == A + x["src_state"] and x["score"] == 0.0 and x["dst_state"] == -1
        elif x["flags"] & oracle.REC_EPS:
            assert g["ilabel"][a] == -1 and x["score"] == g["weight"][a]
        else:
            assert g["ilabel"][a] >= 0
            assert x["score"] == np.float32(g["weight"][a] + lp[x["t"], g["ilabel"][a]])
            assert x["dst_state"] == g["dst"][a]


# ---------------------------------------------------------------- streaming

@pytest.mark.parametrize("chunk", [1, 7, 16])
def test_streaming_chunk_invariance(chunk):
    wl = synth.workload(1)
    g = synth.make_graph(1)
    G = oracle.Graph(g)
    T = 80
    lp = synth.make_lane_log_probs(1, 2, T=T).astype(np.float32)
    p = _p(search_beam=wl.search_beam, min_active=wl.min_active, max_active=wl.max_active,
           lattice=True)
    whole = oracle.Decoder(G, p, None)
    whole.advance(lp)
    rw = whole.finalize()
    d = oracle.Decoder(G, p, None)
    partials = []
    for s in range(0, T, chunk):
        d.advance(lp[s:s + chunk])
        partials.append(d.partial())
    r = d.finalize()
    assert np.float32(r["score"]) == np.float32(rw["score"]) and list(r["words"]) == list(rw["words"])
    np.testing.assert_array_equal(d.lattice(), whole.lattice())
    # the last partial is the best token of the final frontier
    assert partials[-1]["ok"] == 1


def test_streaming_equals_offline_when_last_frames_rule_is_inert():
    """With min_active >= max_active / 2 the offline-only clause cannot change
    min_active, so online and offline decoding must agree exactly."""
    g = synth.make_graph(1)
    G = oracle.Graph(g)
    T = 60
    lp = synth.make_lane_log_probs(1, 5, T=T).astype(np.float32)
    p = _p(search_beam=20.0, min_active=4000, max_active=7000)
    off = oracle.decode(G, lp, T, p)
    d = oracle.Decoder(G, p, None)
    d.advance(lp)
    on = d.finalize()
    assert np.float32(on["score"]) == np.float32(off["score"]) and list(on["arcs"]) == list(off["arcs"])


# ---------------------------------------------------------------- graph checks

def test_rejects_epsilon_cycle_and_bad_arcs():
    g = synth.graph_from_arcs(3, 2, np.array([0, 1, 2]), [1, 2, 0], [-1, -1, -1], [0, 0, 0],
                              [0.0, 0.0, 0.0], np.zeros(3, np.float32))
    with pytest.raises(ValueError, match="cycle"):
        oracle.Graph(g)
    g = synth.graph_from_arcs(2, 2, np.array([0]), [5], [1], [0], [0.0], np.zeros(2, np.float32))
    with pytest.raises(ValueError, match="destination"):
        oracle.Graph(g)
    g = synth.graph_from_arcs(2, 2, np.array([0]), [1], [2], [0], [0.0], np.zeros(2, np.float32))
    with pytest.raises(ValueError, match="ilabel"):
        oracle.Graph(g)


def test_eps_rank_is_topological():
    g = synth.make_graph(0)
    rng = np.random.default_rng(0)
    g2 = synth.random_tiny_graph(rng, 30, 3, max_deg=4, p_eps=0.5)
    rank, has = oracle.Graph(g2).eps_rank()
    assert has
    src = np.repeat(np.arange(30), np.diff(g2["row_splits"]))
    e = g2["ilabel"] < 0
    assert (rank[src[e]] < rank[g2["dst"][e]]).all()
    assert sorted(rank.tolist()) == list(range(30))
    assert not oracle.Graph(g).eps_rank()[1]


# ---------------------------------------------------------------- small golden cases

def _case_graph(c):
    arcs = c["arcs"]
    fl = lambda v: -np.inf if v == "-inf" else float(v)
    return synth.graph_from_arcs(
        c["num_states"], c["vocab"], np.array([a[0] for a in arcs], np.int64),
        [a[1] for a in arcs], [a[2] for a in arcs], [a[3] for a in arcs],
        [a[4] for a in arcs], np.array([fl(v) for v in c["final"]], np.float32), start=c["start"])


def _case_lp(c):
    return np.array([[-np.inf if v == "-inf" else float(v) for v in row] for row in c["log_probs"]],
                    np.float32)


SMALL = json.load(open(os.path.join(GOLD, "small_cases.json")))["cases"]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c["name"])
def test_golden_small_cases(case):
    g = _case_graph(case)
    lp = _case_lp(case)
    T = len(lp)
    p = _p(search_beam=case["search_beam"], min_active=case["min_active"],
           max_active=case["max_active"])
    d = oracle.Decoder(oracle.Graph(g), p, None if case.get("streaming") else T)
    d.advance(lp)
    if "beam" in case:
        tr = d.trace()
        np.testing.assert_allclose(tr["beam"], case["beam"], rtol=2e-6)
        assert list(tr["n"]) == case["n"]
    if "words" in case:
        part = d.partial()
        r = d.finalize()
        assert r["ok"] == 1
        assert np.float32(r["score"]) == np.float32(case["score"])
        assert list(r["words"]) == case["words"]
        assert r["reached_final"] == case["reached_final"]
        if not case["reached_final"]:
            assert list(part["words"]) == case["words"]


def test_work_counters_closed_forms():
    """The oracle's work counters (they define arcs expanded/s and the
    algorithmic bytes) on graphs whose counts are fixed by construction."""
    rng = np.random.default_rng(21)
    V, T = 9, 30
    # one final state with V self-loops, beam wide enough to admit everything:
    # every step has n = 1 token, D = V candidates, a = V admitted, m = 1 state
    g = synth.graph_from_arcs(1, V, np.zeros(V, np.int64), np.zeros(V, np.int32),
                              np.arange(V), np.arange(V), np.zeros(V), np.zeros(1))
    lp = np.log(rng.dirichlet(np.ones(V), size=T)).astype(np.float32)
    r = oracle.decode(oracle.Graph(g), lp, T, _p(search_beam=1e30, min_active=0, max_active=10**9))
    st = r["stats"]
    assert (st["frames"], st["sum_n"], st["sum_D"], st["sum_a"], st["sum_m"]) == (T, T, T * V, T * V, T)
    assert st["finals"] == 1 and st["eps_relaxed"] == 0
    assert st["arcs_expanded"] == T * V + 1
    # a linear chain: one candidate per step, all admitted; no final state
    N = T + 1
    src = np.arange(T)
    g2 = synth.graph_from_arcs(N, V, src, src + 1, rng.integers(1, V, size=T), np.zeros(T, np.int64),
                               -rng.uniform(0, 1, size=T).astype(np.float32), np.full(N, -np.inf, np.float32))
    st2 = oracle.decode(oracle.Graph(g2), lp, T, _p(search_beam=1e30))["stats"]
    assert (st2["sum_n"], st2["sum_D"], st2["sum_a"], st2["sum_m"], st2["finals"]) == (T, T, T, T, 0)
    # a start state with two epsilon arcs to states with one each (a diamond):
    # the start closure relaxes 2 + 1 + 1 epsilon arcs, then nothing emits
    g3 = synth.graph_from_arcs(4, V, np.array([0, 0, 1, 2]), np.array([1, 2, 3, 3]), np.full(4, -1),
                               np.zeros(4, np.int64), np.array([-1.0, -2.0, -0.5, -0.25], np.float32),
                               np.array([-np.inf, -np.inf, -np.inf, 0.0], np.float32))
    st3 = oracle.decode(oracle.Graph(g3), lp, 1, _p(search_beam=1e30))["stats"]
    assert st3["eps_relaxed"] == 4 and st3["sum_m"] == 0 and st3["finals"] == 0
    # pruning: the first admission-boundary case (hand-derived in
    # tests/golden/admission_boundary.json) expands n = 1 token into D = 4
    # candidates, admits a = 2 of them into m = 2 states
    w = [0.0, -12.5, -12.375, -13.0]
    g4 = synth.graph_from_arcs(5, 2, np.zeros(4, np.int64), [1, 2, 3, 4], [1] * 4, [1, 2, 3, 4], w,
                               np.zeros(5, np.float32))
    st4 = oracle.decode(oracle.Graph(g4), np.full((1, 2), -0.5, np.float32), 1,
                        _p(search_beam=10.0, min_active=2, max_active=100))["stats"]
    assert (st4["sum_n"], st4["sum_D"], st4["sum_a"], st4["sum_m"]) == (1, 4, 2, 2)
    # recombination: three admitted arcs into one state give m = 1
    g5 = synth.graph_from_arcs(2, 2, np.zeros(3, np.int64), [1, 1, 1], [1, 1, 1], [0, 0, 0],
                               [0.0, -1.0, -2.0], np.zeros(2, np.float32))
    st5 = oracle.decode(oracle.Graph(g5), np.full((1, 2), -0.5, np.float32), 1,
                        _p(search_beam=1e30))["stats"]
    assert (st5["sum_n"], st5["sum_D"], st5["sum_a"], st5["sum_m"]) == (1, 3, 3, 1)


def test_blank_skip_rule_by_hand():
    """Blank-skip pre-slicing (§3: blank-dominated frames are removed before
    the search, WeNet-style, threshold 0.98): a frame is dropped when its
    blank posterior is above the threshold.  Expected frames written out from the posteriors."""
    import oracle
    thr = 0.98
    lthr = np.float32(np.log(0.98))
    p_blank = [0.99, 0.97, 0.985, 0.5, 0.999]          # frame 4 lies past lens[0]
    V = 3
    lp = np.zeros((2, 6, V), np.float32)
    for t, pb in enumerate(p_blank):
        rest = (1.0 - pb) / (V - 1)
        lp[0, t] = np.log([pb, rest, rest])
    lp[0, 5] = [lthr, -1.0, -1.0]                      # exactly at log(threshold): kept (strict '>')
    lens = np.array([4, 0], np.int32)
    rows, frames = oracle.blank_skip(lp, lens, thr)
    assert list(frames[0]) == [1, 3]
    assert np.array_equal(rows[0], lp[0, [1, 3]])
    assert len(frames[1]) == 0 and rows[1].shape == (0, V)
    lens = np.array([6, 6], np.int32)
    lp[1, :, 0] = np.nextafter(lthr, np.float32(0.0))  # just above log(threshold): dropped
    rows, frames = oracle.blank_skip(lp, lens, thr)
    assert list(frames[0]) == [1, 3, 5]
    assert len(frames[1]) == 0
    # threshold 1: no log-probability lies above log(1) = 0, every frame is kept
    rows, frames = oracle.blank_skip(lp, lens, 1.0)
    assert [list(f) for f in frames] == [list(range(6)), list(range(6))]
