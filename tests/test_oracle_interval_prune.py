"""Pins of the oracle's interval lattice prune (page "GPU WFST Beam-Search
Decoder", §7 lattice paragraph: every lat_prune_interval frames a loose
prune runs over a window of recent frames; the final output_beam prune stays
exact).  The reading: the interval pass drops only records that the final
prune can never keep, so the final lattice must not change; the golden case
fixes which records it drops (hand derivation in tests/golden/)."""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "interval_prune.json")


def _golden_graph(spec):
    src, dst, il, ol, w = (list(c) for c in zip(*spec["arcs"]))
    fin = np.array([-np.inf if f is None else f for f in spec["finals"]], np.float32)
    return synth.graph_from_arcs(spec["num_states"], 2, np.array(src), dst, il, ol, w, fin)


def test_golden_interval_prune_drops_exactly_the_derived_records():
    spec = json.load(open(GOLDEN))
    g = _golden_graph(spec)
    lp = np.tile(np.array(spec["lp_row"], np.float32), (spec["T"], 1))
    OG = oracle.Graph(g)
    want = np.array([tuple(r) for r in spec["final_lattice"]], dtype=oracle.LAT_DTYPE)
    for case in spec["cases"]:
        p = oracle.params(**spec["params"], allow_partial=True, lattice=True,
                          lat_prune_interval=case["lat_prune_interval"])
        r = oracle.decode(OG, lp, spec["T"], p, lattice_out=True)
        assert r["stats"]["records_dropped"] == case["dropped"], case
        assert list(r["words"]) == spec["words"] and r["score"] == spec["score"]
        lat = r["lattice"]
        for k in want.dtype.names:
            assert np.array_equal(lat[k], want[k]), (case, k)
        # what the interval pass dropped is gone from the unpruned record set
        d = oracle.Decoder(OG, p, spec["T"])
        d.advance(lp)
        d.finalize()
        assert len(d.lattice(kept=False)) == 7 + 1 - case["dropped"]


def _tiny(seed):
    rng = np.random.default_rng(6100 + seed)
    N = int(rng.integers(2, 40))
    V = int(rng.integers(2, 9))
    g = synth.random_tiny_graph(rng, N, V, max_deg=int(rng.integers(1, 6)), p_eps=float(rng.choice([0.0, 0.3])),
                                dyadic=bool(seed % 2 == 0), allow_empty=bool(seed % 3 == 0),
                                p_final=float(rng.choice([0.0, 0.2, 0.6])), relabel=bool(seed % 4 == 1))
    T = int(rng.integers(1, 30))
    if seed % 2 == 0:
        lp = synth.dyadic_log_probs(rng, T, V, lo=-4.0)
    else:
        lp = np.log(rng.dirichlet(np.ones(V), size=T)).astype(np.float32)
    p = dict(search_beam=float(rng.choice([1.0, 2.5, 6.0, 20.0])), output_beam=float(rng.choice([0.0, 1.0, 4.0])),
             min_active=int(rng.integers(0, 5)), max_active=int(rng.integers(1, 12)),
             allow_partial=bool(seed % 5 != 0), lattice=True)
    return g, lp, T, p


def _same_result(a, b, where):
    assert a["ok"] == b["ok"] and list(a["words"]) == list(b["words"]), where
    if a["ok"]:
        assert a["score"] == b["score"], where
        for k in a["lattice"].dtype.names:
            assert np.array_equal(a["lattice"][k], b["lattice"][k]), (where, k)


def test_interval_prune_never_changes_the_final_lattice():
    """On random tiny graphs (with and without epsilon arcs, states renamed,
    dyadic and non-dyadic scores) every interval leaves words, scores and
    the final lattice as they are without it."""
    dropped = 0
    for seed in range(240):
        g, lp, T, p = _tiny(seed)
        OG = oracle.Graph(g)
        ref = oracle.decode(OG, lp, T, oracle.params(**p), lattice_out=True)
        for n in (1, 2, 5):
            r = oracle.decode(OG, lp, T, oracle.params(**p, lat_prune_interval=n), lattice_out=True)
            _same_result(r, ref, f"seed {seed} interval {n}")
            dropped += r["stats"]["records_dropped"]
    assert dropped > 1000   # the pass does drop records


def test_interval_prune_on_workloads_0_and_3_streaming():
    """Workload 0 (lattice on) offline and online, and workload 3's epsilon
    graph online over 40 frames: the same final lattices with the interval
    prune at 4 and 16 frames."""
    cases = [(0, synth.make_log_probs(0)[0], 50, None), (0, synth.make_log_probs(0)[0], 50, "online")]
    lp3 = synth.make_log_probs(3, lanes=[5], T=40)[0]
    cases.append((3, lp3, 40, "online"))
    for wi, lp, T, mode in cases:
        wl = synth.workload(wi)
        OG = oracle.Graph(synth.make_graph(wi))
        base = dict(search_beam=wl.search_beam, output_beam=wl.output_beam, min_active=wl.min_active,
                    max_active=wl.max_active, allow_partial=True, lattice=True)

        def run(n):
            d = oracle.Decoder(OG, oracle.params(**base, lat_prune_interval=n), None if mode else T)
            d.advance(lp[:T])
            r = d.finalize()
            r["lattice"] = d.lattice()
            r["stats"] = d.stats()
            return r
        ref = run(0)
        for n in (4, 16):
            r = run(n)
            _same_result(r, ref, f"workload {wi} {mode} interval {n}")
            assert r["stats"]["records_dropped"] > 0


def test_interval_prune_bounds_a_long_stream():
    """A 2400-frame stream over workload 0's graph: with the interval prune
    the records held are about twice the final lattice's size instead of
    about five times it, and the final lattice is the same."""
    wl = synth.workload(0)
    OG = oracle.Graph(synth.make_graph(0))
    T = 2400
    lp = synth.make_lane_log_probs(0, 7, T=T)
    out = {}
    for n in (0, 50):
        d = oracle.Decoder(OG, oracle.params(wl.search_beam, wl.output_beam, wl.min_active, wl.max_active,
                                             True, True, n), None)
        d.advance(lp)
        st = d.stats()
        d.finalize()
        out[n] = (st["records"] - st["records_dropped"], d.lattice())
    live0, lat0 = out[0]
    live, lat = out[50]
    assert len(lat) == len(lat0) and all(np.array_equal(lat[k], lat0[k]) for k in lat.dtype.names)
    assert live0 > 4 * len(lat0)
    assert live < 2.5 * len(lat0)
