"""The decode kernel's three instantiations run the same search: a decode of
an epsilon-free graph without lattices or GC runs the plain kind, one with
lattices the general kind, one with the winners-log GC the ancestor-GC kind.
On workload 1's graph and log-probs all three give the same words, scores
and flags on every lane, and lane 0 equals the oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_common import assert_lane_equal, oracle_lane, wl_params

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def W():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import wfst_beam_search_gb300 as W
    W.load()
    return W


def test_kernel_kinds_agree_on_workload1(W):
    wl = synth.workload(1)
    g = synth.make_graph(1)
    lp_host = synth.make_log_probs(1)
    lens = synth.make_lens(1)
    G = W.Graph(g, device=0)
    lp = torch.from_numpy(np.ascontiguousarray(lp_host)).to("cuda:0")
    outs = {}
    for name, lattice, gc in (("plain", False, 0), ("general", True, 0), ("ancestor GC", False, 8)):
        params = W.make_params(wl.search_beam, wl.output_beam, wl.min_active, wl.max_active, True, lattice,
                               gc_interval=gc)
        D = W.Decoder(G, params, wl.B, wl.T)
        outs[name] = D.decode(lp, lens)
        D.close()
    for b in range(wl.B):
        ref = outs["plain"][b]
        assert ref["ok"] == 1, f"lane {b}"
        for name in ("general", "ancestor GC"):
            got = outs[name][b]
            where = f"{name} kind, lane {b}"
            assert np.array_equal(got["words"], ref["words"]), where
            assert got["score"] == ref["score"], where
            assert (got["ok"], got["reached_final"], got["overflow"]) == \
                   (ref["ok"], ref["reached_final"], ref["overflow"]), where
    p = wl_params(wl, lattice=False)
    assert_lane_equal(outs["plain"][0], oracle_lane(oracle.Graph(g), lp_host[0], lens[0], p), "plain kind, lane 0")
    G.close()
