"""wfst_decode_static (the offline decode whose working memory is the
library's statically declared device region) against wfst_decode on the same
inputs: identical words, flags and scores, on two calls in a row, so that
whatever the first call leaves in the region cannot change the second.

This file is collected last (tests/conftest.py) so that it also runs after
every other test in one process, and it must pass when run alone."""
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


def _cuda(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda:0")


def _same(a, b, where):
    assert a["ok"] == b["ok"], where
    assert a["reached_final"] == b["reached_final"], where
    assert a["overflow"] == b["overflow"] == 0, where
    assert a["n_words"] == b["n_words"], where
    assert list(a["words"]) == list(b["words"]), where
    if a["ok"]:
        assert a["score"] == b["score"], where   # same kernel, same fp32 sums


def _params(W, p):
    return W.make_params(p["search_beam"], p["output_beam"], p["min_active"], p["max_active"],
                         p["allow_partial"], False, False)


def _tiny_case(seed):
    rng = np.random.default_rng(91000 + seed)
    N = int(rng.integers(2, 40))
    V = int(rng.integers(2, 9))
    g = synth.random_tiny_graph(rng, N, V, max_deg=int(rng.integers(1, 6)), p_eps=0.3 * (seed % 2),
                                dyadic=bool(seed % 2 == 0), allow_empty=False,
                                p_final=float(rng.choice([0.0, 0.2, 0.6])))
    B = int(rng.integers(1, 9))
    T = int(rng.integers(1, 14))
    lens = rng.integers(0, T + 1, size=B).astype(np.int32)
    lens[0] = T
    lp = np.log(rng.dirichlet(np.ones(V), size=(B, T))).astype(np.float32)
    p = dict(search_beam=float(rng.choice([2.5, 6.0, 20.0])), output_beam=0.0,
             min_active=int(rng.integers(0, 5)), max_active=int(rng.integers(1, 12)),
             allow_partial=True, lattice=False)
    return g, lp, lens, p


def test_static_matches_decoder_on_two_calls_in_a_row(W):
    wl = synth.workload(0)
    g = synth.make_graph(0)
    G = W.Graph(g, device=0)
    p = wl_params(wl, lattice=False)
    params = _params(W, p)
    T = wl.T
    lp_a = np.stack([synth.make_lane_log_probs(0, b) for b in range(4)]).astype(np.float32)
    lp_b = np.stack([synth.make_lane_log_probs(0, 10 + b) for b in range(6)]).astype(np.float32)
    lens_a = np.array([T, T - 7, 1, T], np.int32)
    lens_b = np.array([T - 3, T, 0, 12, T, 31], np.int32)
    D = W.Decoder(G, params, 8, T)
    OG = oracle.Graph(g)
    for name, lp, lens in (("first", lp_a, lens_a), ("second", lp_b, lens_b)):
        got = W.decode_static(G, params, _cuda(lp), lens)
        ref = D.decode(_cuda(lp), lens)
        for b in range(len(lens)):
            _same(got[b], ref[b], f"{name} call, lane {b}")
            assert_lane_equal(got[b], oracle_lane(OG, lp[b], lens[b], p), f"{name} call, lane {b}")


def test_static_matches_decoder_on_tiny_graphs(W):
    # consecutive calls with changing graphs and shapes re-lay the region out
    for seed in range(24):
        g, lp, lens, p = _tiny_case(seed)
        G = W.Graph(g, device=0)
        params = _params(W, p)
        D = W.Decoder(G, params, 8, lp.shape[1])
        for rep in range(2):
            got = W.decode_static(G, params, _cuda(lp), lens)
            ref = D.decode(_cuda(lp), lens)
            for b in range(len(lens)):
                _same(got[b], ref[b], f"seed {seed} call {rep} lane {b}")


def test_static_fp16_input(W):
    wl = synth.workload(0)
    g = synth.make_graph(0)
    G = W.Graph(g, device=0)
    params = _params(W, wl_params(wl, lattice=False))
    lp = np.stack([synth.make_lane_log_probs(0, b) for b in range(3)]).astype(np.float16)
    lens = np.array([wl.T, 20, wl.T], np.int32)
    D = W.Decoder(G, params, 4, wl.T)
    for rep in range(2):
        got = W.decode_static(G, params, _cuda(lp), lens)
        ref = D.decode(_cuda(lp), lens)
        for b in range(3):
            _same(got[b], ref[b], f"call {rep} lane {b}")


def test_static_rejects_what_does_not_fit(W):
    wl = synth.workload(0)
    g = synth.make_graph(0)
    G = W.Graph(g, device=0)
    params = _params(W, wl_params(wl, lattice=False))
    lp = _cuda(np.stack([synth.make_lane_log_probs(0, b) for b in range(9)]).astype(np.float32))
    with pytest.raises(W.WfstError) as e:
        W.decode_static(G, params, lp, np.full(9, wl.T, np.int32))
    assert e.value.code == -5 and "WFST_STATIC_MAX_LANES" in str(e.value)
    # a graph whose tables exceed the region: CAPACITY with the bytes needed
    big = synth.make_graph(1)
    GB = W.Graph(big, device=0)
    V = synth.workload(1).V
    lpb = torch.zeros((8, 200, V), dtype=torch.float32, device="cuda:0")
    with pytest.raises(W.WfstError) as e:
        W.decode_static(GB, params, lpb, np.full(8, 200, np.int32))
    assert e.value.code == -5 and "bytes of scratch" in str(e.value)
    # host log-probs are refused (the call copies nothing in)
    with pytest.raises(W.WfstError) as e:
        W.decode_static(G, params, np.zeros((1, 5, wl.V), np.float32), np.array([5], np.int32))
    assert e.value.code == -1
    # lattice output needs a decoder
    lat = W.make_params(wl.search_beam, wl.output_beam, wl.min_active, wl.max_active, True, True, False)
    with pytest.raises(W.WfstError):
        W.decode_static(G, lat, lp[:1], np.array([wl.T], np.int32))
    # the region still decodes correctly after the refusals
    lens = np.array([wl.T], np.int32)
    got = W.decode_static(G, params, lp[:1], lens)
    ref = W.Decoder(G, params, 1, wl.T).decode(lp[:1], lens)
    _same(got[0], ref[0], "after refusals")


def test_static_log_fills_the_region_and_refuses_overflow(W):
    """A wide beam on workload 1's graph (50k states): with max_active 10
    the frontier decays after ~25 frames and a 60-frame lane needs about
    1.08M winners-log entries, more than the decoder's default for that
    max_active (1Mi) but within what the region leaves one lane, so the
    static call equals wfst_decode and the oracle.  With max_active
    unbounded every frame holds ~50k tokens (~3M entries): the static call
    returns CAPACITY, while wfst_decode grows its log and stays exact."""
    g = synth.make_graph(1)
    G = W.Graph(g, device=0)
    OG = oracle.Graph(g)
    T = 60
    lp = synth.make_log_probs(1, lanes=[0], T=T)
    lens = np.array([T], np.int32)
    for max_active, fits in ((10, True), (2**30, False)):
        p = dict(search_beam=1000.0, output_beam=0.0, min_active=0, max_active=max_active,
                 allow_partial=True, lattice=False)
        params = _params(W, p)
        D = W.Decoder(G, params, 1, T)
        ref = D.decode(_cuda(lp), lens)
        assert_lane_equal(ref[0], oracle_lane(OG, lp[0], T, p), f"decoder, max_active {max_active}")
        for rep in range(2):
            if fits:
                got = W.decode_static(G, params, _cuda(lp), lens)
                _same(got[0], ref[0], f"max_active {max_active} call {rep}")
            else:
                with pytest.raises(W.WfstError) as e:
                    W.decode_static(G, params, _cuda(lp), lens)
                assert e.value.code == -5 and "winners log" in str(e.value)
        D.close()
