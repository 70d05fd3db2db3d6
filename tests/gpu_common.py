"""Shared helpers of the GPU parity tests: run the CUDA decoder through the C
ABI and the oracle on the same seeded inputs and compare."""
from __future__ import annotations

import numpy as np

import oracle
import synth

SCORE_TOL = 1e-4       # absolute, on fp32 path scores (same fp32 sums in the same order)


def wl_params(wl, lattice=None, allow_partial=True):
    return dict(search_beam=wl.search_beam, output_beam=wl.output_beam,
                min_active=wl.min_active, max_active=wl.max_active,
                allow_partial=allow_partial, lattice=wl.lattice if lattice is None else lattice)


def gpu_decoder(W, g, p, max_lanes, max_frames, caps=None, graph=None, streaming=False, options=0):
    G = graph if graph is not None else W.Graph(g, device=0)
    params = W.make_params(p["search_beam"], p["output_beam"], p["min_active"], p["max_active"],
                           p["allow_partial"], p["lattice"], streaming, options)
    return G, W.Decoder(G, params, max_lanes, max_frames, caps)


def oracle_lane(OG, lp, length, p, streaming=False):
    op = oracle.params(**p)
    if not streaming:
        return oracle.decode(OG, lp, int(length), op, lattice_out=p["lattice"])
    d = oracle.Decoder(OG, op, None)
    if length:
        d.advance(np.asarray(lp)[:length])
    r = d.finalize()
    if p["lattice"]:
        r["lattice"] = d.lattice()
    r["stats"] = d.stats()
    return r


def assert_lane_equal(got, ref, where=""):
    assert got["overflow"] == 0, f"{where}: capacity overflow {got['overflow']}"
    assert got["ok"] == ref["ok"], f"{where}: ok {got['ok']} vs {ref['ok']}"
    if not ref["ok"]:
        return
    assert got["reached_final"] == ref["reached_final"], f"{where}: reached_final"
    assert list(got["words"]) == list(ref["words"]), f"{where}: words {list(got['words'])} vs {list(ref['words'])}"
    assert abs(got["score"] - float(ref["score"])) <= SCORE_TOL, f"{where}: score {got['score']} vs {ref['score']}"


def assert_lattice_equal(lat, ref_lat, where=""):
    assert len(lat) == len(ref_lat), f"{where}: lattice size {len(lat)} vs {len(ref_lat)}"
    for k in ("t", "src_state", "dst_state", "arc_id", "flags"):
        assert np.array_equal(lat[k], ref_lat[k]), f"{where}: lattice field {k} differs"
    assert np.all(np.abs(lat["score"] - ref_lat["score"]) <= SCORE_TOL), f"{where}: lattice scores"
