"""Lazily committed tables (page "GPU WFST Beam-Search Decoder" §6.2): the
frontier, winners-log and lattice tables reserve worst-case address ranges
and commit device memory only for their current capacities; growth maps
more memory in place, so lanes keep their contents and only overflowed
lanes run again; streaming channels grow between calls."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_common import assert_lane_equal, assert_lattice_equal, gpu_decoder, oracle_lane, wl_params

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


def test_workload2_decoder_commits_a_fraction_of_its_worst_case(W):
    """The 64-lane decoder of workload 2: the eager layout (a frontier of N
    tokens and a log of 4 * max_active entries per frame, in every lane)
    held ~20 GB; committed now: the recombination table (4.1 GB, touched
    densely) plus the lazy tables' initial capacities, and the first decode
    needs no growth."""
    wl = synth.workload(2)
    g = synth.make_graph(2)
    G, D = gpu_decoder(W, g, wl_params(wl), wl.B, wl.T)
    m = D.mem_stats()
    N, L, mf = g["num_states"], wl.B, wl.T + 2
    eager = 2 * L * N * 16 + L * N * 8 + 2 * L * N * 20 + L * mf * 4 * wl.max_active * 8
    assert m["reserved"] >= m["lazy_committed"] > 0
    assert m["bytes"] < 0.45 * eager, (m, eager)
    lanes = list(range(8))
    lp = synth.make_log_probs(2, lanes=lanes, T=160)
    out = D.decode(_cuda(lp), np.full(8, 160, np.int32))
    assert all(o["overflow"] == 0 and o["ok"] for o in out)
    assert D.mem_stats()["grows"] == 0


def test_growth_in_place_reruns_only_overflowed_lanes(W):
    """Workload 0 with a lattice and small capacities: a long lane overflows
    the winners log and the lattice arena, short lanes do not; after growth
    every lane equals the oracle (lattices included), and the short lanes'
    records survived the growth untouched (they were not decoded again: the
    decoder's frame counter counts only the rerun lane twice)."""
    wl = synth.workload(0)
    g = synth.make_graph(0)
    T = 50
    lp = synth.make_log_probs(0, lanes=range(3), T=T)
    lens = np.array([T, 4, 6], np.int32)
    p = wl_params(wl)
    OG = oracle.Graph(g)
    refs = [oracle_lane(OG, lp[b], lens[b], p) for b in range(3)]
    need_log = refs[0]["stats"]["tokens"]
    need_lat = refs[0]["stats"]["records"]
    small = max(refs[1]["stats"]["tokens"], refs[2]["stats"]["tokens"]) + 8
    G, D = gpu_decoder(W, g, p, 3, T, caps=W.Capacity(0, small, max(refs[1]["stats"]["records"],
                                                                    refs[2]["stats"]["records"]) + 8, 0))
    assert need_log > D.mem_stats()["log_cap"] and need_lat > D.mem_stats()["lattice_cap"]
    out = D.decode(_cuda(lp), lens)
    for b in range(3):
        assert_lane_equal(out[b], refs[b], f"lane {b}")
        assert_lattice_equal(D.lattice(b), refs[b]["lattice"], f"lane {b}")
    st = D.stats()
    m = D.mem_stats()
    assert m["grows"] >= 1 and m["log_cap"] >= need_log
    # frames of every round: lanes 1 and 2 once, lane 0 once per round
    rounds = m["grows"] + 1
    assert st["frames"] == int(lens[1] + lens[2]) + rounds * int(lens[0])


def test_streaming_channels_grow_between_calls(W):
    """A 600-frame lattice stream in 24-frame chunks on a decoder made with a
    small winners log and lattice arena (each holds two chunks): the tables
    double between calls whenever a channel has used half of them, so no
    chunk overflows, and the results equal the oracle's."""
    wl = synth.workload(0)
    g = synth.make_graph(0)
    T, chunk = 600, 24
    lp = synth.make_log_probs(0, lanes=range(2), T=T)
    p = wl_params(wl)
    G, D = gpu_decoder(W, g, p, 2, T, caps=W.Capacity(0, 1 << 14, 1 << 16, 0), streaming=True)
    m0 = D.mem_stats()
    chans = [D.stream_create() for _ in range(2)]
    for s in range(0, T, chunk):
        outs = D.stream_advance(chans, _cuda(lp[:, s:s + chunk]), np.full(2, chunk, np.int32), want_partial=True)
        assert all(o["overflow"] == 0 for o in outs), s
    fin = D.stream_finalize(chans)
    m1 = D.mem_stats()
    assert m1["log_cap"] > m0["log_cap"] and m1["lattice_cap"] > m0["lattice_cap"]
    assert m1["lazy_committed"] > m0["lazy_committed"]
    OG = oracle.Graph(g)
    for i in range(2):
        ref = oracle_lane(OG, lp[i], T, p, streaming=True)
        assert_lane_equal(fin[i], ref, f"channel {i}")
        assert_lattice_equal(D.lattice(chans[i]), ref["lattice"], f"channel {i}")
