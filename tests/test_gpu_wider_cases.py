"""GPU parity on inputs outside the other files' generators: tiny graphs
whose states are renamed by a random permutation (start state other than 0,
epsilon arcs into lower state ids), and the hand-derived case where the best
score falls as the beam widens (tests/golden/beam_not_monotone.json)."""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_common import assert_lane_equal, assert_lattice_equal, gpu_decoder, oracle_lane
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


def test_tiny_random_graphs_relabelled(W):
    """States renamed by a random permutation: epsilon arcs also run from
    higher to lower state ids and the start state is not state 0."""
    for seed in range(40):
        g, lp, lens, p = _tiny_case(seed, 0.4, relabel=True)
        G, D = gpu_decoder(W, g, p, max_lanes=6, max_frames=lp.shape[1])
        OG = oracle.Graph(g)
        out = D.decode(torch.from_numpy(np.ascontiguousarray(lp)).to("cuda:0"), lens)
        for b in range(len(lens)):
            ref = oracle_lane(OG, lp[b], lens[b], p)
            where = f"relabelled seed {seed} lane {b}"
            assert_lane_equal(out[b], ref, where)
            if ref["ok"]:
                assert_lattice_equal(D.lattice(b), ref["lattice"], where)
        D.close()
        G.close()


def test_best_score_not_monotone_in_the_beam(W):
    """The hand-derived case on a streaming channel (online beam rules):
    beam 1 gives -5.5, beam 2 gives -13, an unbounded beam -5.5, because the
    decoder prunes against the step's exact maximum over all of the lane's
    candidates."""
    spec = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "beam_not_monotone.json")))
    src, dst, il, ol, w = (list(c) for c in zip(*spec["arcs"]))
    N, T = spec["num_states"], spec["T"]
    fin = np.array([-np.inf if f is None else f for f in spec["finals"]], np.float32)
    g = synth.graph_from_arcs(N, 2, np.array(src), dst, il, ol, w, fin)
    lp = torch.full((1, T, 2), -0.5, dtype=torch.float32, device="cuda:0")
    G = W.Graph(g, device=0)
    for case in spec["cases"]:
        p = dict(search_beam=case["search_beam"], output_beam=0.0, min_active=spec["min_active"],
                 max_active=spec["max_active"], allow_partial=False, lattice=False)
        _, D = gpu_decoder(W, g, p, 1, T, graph=G, streaming=True)
        ch = D.stream_create()
        D.stream_advance([ch], lp, [T], want_partial=False)
        f = D.stream_finalize([ch])[0]
        D.stream_release(ch)
        assert f["ok"] == 1 and f["reached_final"] == case["reached_final"], case
        assert np.float32(f["score"]) == np.float32(case["score"]), (case["search_beam"], f["score"])
        assert list(f["words"]) == case["words"], (case["search_beam"], f["words"])
        D.close()
    G.close()
