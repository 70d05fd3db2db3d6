"""The interval lattice prune on the GPU (lat_prune_interval, page "GPU WFST
Beam-Search Decoder" §7) against the oracle's: the same final lattices as
without it, and on epsilon-free graphs exactly the oracle's number of
records held (the GPU compacts the dropped records out of its arena)."""
import os

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_common import assert_lane_equal, assert_lattice_equal, gpu_decoder, oracle_lane, wl_params
from tests.test_gpu_parity import _tiny_case

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def W():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import wfst_beam_search_gb300 as W
    W.load()
    return W


def _cuda(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda:0")


def _decoder(W, g, p, lanes, frames, n, graph=None, streaming=False):
    G = graph if graph is not None else W.Graph(g, device=0)
    params = W.make_params(p["search_beam"], p["output_beam"], p["min_active"], p["max_active"],
                           p["allow_partial"], True, streaming, 0, 0, n)
    return G, W.Decoder(G, params, lanes, frames)


def _oracle(OG, lp, T, p, n, online=False):
    d = oracle.Decoder(OG, oracle.params(**dict(p, lattice=True), lat_prune_interval=n), None if online else T)
    if T:
        d.advance(np.asarray(lp)[:T].astype(np.float32))
    r = d.finalize()
    r["lattice"] = d.lattice()
    r["stats"] = d.stats()
    return r


def test_workload0_offline_intervals(W):
    wl = synth.workload(0)
    g = synth.make_graph(0)
    lp = synth.make_log_probs(0, lanes=range(3))
    lens = np.array([wl.T, 37, 16], np.int32)
    p = wl_params(wl)
    OG = oracle.Graph(g)
    G = W.Graph(g, device=0)
    for n in (1, 4, 16):
        _, D = _decoder(W, g, p, 3, wl.T, n, graph=G)
        out = D.decode(_cuda(lp), lens)
        held = 0
        for b in range(3):
            ref = _oracle(OG, lp[b], lens[b], p, n)
            assert_lane_equal(out[b], ref, f"interval {n} lane {b}")
            assert_lattice_equal(D.lattice(b), ref["lattice"], f"interval {n} lane {b}")
            held += ref["stats"]["records"] - ref["stats"]["records_dropped"]
        assert D.stats()["lattice_records_held"] == held, n
        D.close()


def test_tiny_graphs_with_epsilon_arcs_and_intervals(W):
    for seed in range(40):
        g, lp, lens, p = _tiny_case(seed, 0.4 if seed % 2 else 0.0)
        OG = oracle.Graph(g)
        for n in (1, 3):
            G, D = _decoder(W, g, p, len(lens), lp.shape[1], n)
            out = D.decode(_cuda(lp), lens)
            for b in range(len(lens)):
                ref = _oracle(OG, lp[b], lens[b], p, n)
                where = f"seed {seed} interval {n} lane {b}"
                assert_lane_equal(out[b], ref, where)
                if ref["ok"]:
                    assert_lattice_equal(D.lattice(b), ref["lattice"], where)
            D.close()
            G.close()


def test_workload3_epsilon_lattice_with_interval(W):
    wl = synth.workload(3)
    g = synth.make_graph(3)
    T = 64
    lanes = [2, 11]
    lp = synth.make_log_probs(3, lanes=lanes, T=T)
    lens = np.array([T, 50], np.int32)
    p = wl_params(wl, lattice=True)
    OG = oracle.Graph(g)
    G, D = _decoder(W, g, p, 2, T, 8)
    out = D.decode(_cuda(lp), lens)
    for b in range(2):
        ref = _oracle(OG, lp[b], lens[b], p, 8)
        assert_lane_equal(out[b], ref, f"workload 3 lane {lanes[b]}")
        assert_lattice_equal(D.lattice(b), ref["lattice"], f"workload 3 lane {lanes[b]}")
        assert ref["stats"]["records_dropped"] > 0


def test_streaming_workload4_channels_with_interval(W):
    wl = synth.workload(4)
    g = synth.make_graph(4)
    n_ch = 4
    lens = synth.make_lens(4)[:n_ch]
    lp = synth.make_log_probs(4, lanes=range(n_ch))
    p = wl_params(wl)
    G, D = _decoder(W, g, p, n_ch, wl.T, 32, streaming=True)
    chans = [D.stream_create() for _ in range(n_ch)]
    T = int(lens.max())
    for s in range(0, T, wl.chunk):
        cl = np.clip(lens - s, 0, wl.chunk).astype(np.int32)
        D.stream_advance(chans, _cuda(lp[:, s:s + wl.chunk]), cl, want_partial=(s // wl.chunk) % 2 == 0)
    fin = D.stream_finalize(chans)
    OG = oracle.Graph(g)
    for i in range(n_ch):
        ref = _oracle(OG, lp[i], int(lens[i]), p, 32, online=True)
        assert_lane_equal(fin[i], ref, f"channel {i}")
        assert_lattice_equal(D.lattice(chans[i]), ref["lattice"], f"channel {i}")


def test_long_stream_arena_stays_near_the_lattice(W):
    """A 2400-frame stream on workload 0's graph, 48-frame chunks, interval 50:
    the final lattice equals the oracle's, the arena holds exactly the
    oracle's live records, about twice the final lattice, where without the
    interval prune it holds every admitted candidate."""
    wl = synth.workload(0)
    g = synth.make_graph(0)
    T, chunk = 2400, 48
    lp = synth.make_lane_log_probs(0, 7, T=T)[None]
    p = wl_params(wl)
    OG = oracle.Graph(g)
    G = W.Graph(g, device=0)
    held = {}
    for n in (0, 50):
        _, D = _decoder(W, g, p, 1, T, n, graph=G, streaming=True)
        ch = D.stream_create()
        for s in range(0, T, chunk):
            D.stream_advance([ch], _cuda(lp[:, s:s + chunk]), [chunk], want_partial=False)
        f = D.stream_finalize([ch])[0]
        held[n] = D.stats()["lattice_records_held"]
        ref = _oracle(OG, lp[0], T, p, n, online=True)
        assert_lane_equal(f, ref, f"interval {n}")
        lat = D.lattice(ch)
        assert_lattice_equal(lat, ref["lattice"], f"interval {n}")
        assert held[n] == ref["stats"]["records"] - ref["stats"]["records_dropped"], n
        D.close()
    assert held[50] < 2.5 * len(lat) and held[0] > 4 * len(lat), held
