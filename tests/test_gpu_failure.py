"""Failure detection on the device, tested without a GPU fault: every grid
barrier wait of the persistent decode kernel is bounded.  The decoder's test
hook makes the next call's barriers unreachable (one arrival more than the
grid makes) with a 200 ms limit, so the first wait gives up, the kernel sets
its abort flag and every CTA returns.  The call must report TIMEOUT, and the
same decoder must then decode exactly as the oracle does (the entry tables,
epsilon marks and channels were reset)."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_common import assert_lane_equal, assert_lattice_equal, gpu_decoder, oracle_lane, wl_params
from tests.test_gpu_parity import _tiny_case

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LIMIT_NS = 200_000_000


@pytest.fixture(scope="module")
def W():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import wfst_beam_search_gb300 as W
    W.load()
    return W


def _cuda(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda:0")


def _expect_timeout(W, fn):
    with pytest.raises(W.WfstError) as e:
        fn()
    assert e.value.code == -6, str(e.value)
    assert "barrier" in str(e.value)


def test_offline_barrier_timeout_then_exact_decode(W):
    wl = synth.workload(0)
    g = synth.make_graph(0)
    lp = synth.make_log_probs(0, lanes=range(3))
    lens = np.array([wl.T, 31, wl.T], np.int32)
    p = wl_params(wl)
    G, D = gpu_decoder(W, g, p, 3, wl.T)
    OG = oracle.Graph(g)
    for rep in range(2):
        D.arm_barrier_timeout(LIMIT_NS)
        _expect_timeout(W, lambda: D.decode(_cuda(lp), lens))
        out = D.decode(_cuda(lp), lens)
        for b in range(3):
            ref = oracle_lane(OG, lp[b], lens[b], p)
            assert_lane_equal(out[b], ref, f"after timeout {rep}, lane {b}")
            assert_lattice_equal(D.lattice(b), ref["lattice"], f"after timeout {rep}, lane {b}")


def test_epsilon_graph_barrier_timeout_mid_decode(W):
    """An epsilon graph: a timeout after a decode that advanced the lanes'
    worklist pass ids; the next decode must not see stale dedupe marks."""
    g, lp, lens, p = _tiny_case(1, 0.4)
    G, D = gpu_decoder(W, g, p, len(lens), lp.shape[1])
    OG = oracle.Graph(g)
    D.decode(_cuda(lp), lens)
    D.arm_barrier_timeout(LIMIT_NS)
    _expect_timeout(W, lambda: D.decode(_cuda(lp), lens))
    out = D.decode(_cuda(lp), lens)
    for b in range(len(lens)):
        ref = oracle_lane(OG, lp[b], lens[b], p)
        assert_lane_equal(out[b], ref, f"eps lane {b}")
        if ref["ok"]:
            assert_lattice_equal(D.lattice(b), ref["lattice"], f"eps lane {b}")


def test_streaming_barrier_timeout_closes_channels(W):
    wl = synth.workload(0)
    g = synth.make_graph(0)
    p = wl_params(wl, lattice=False)
    T, chunk = 48, 16
    lp = synth.make_log_probs(0, lanes=range(2), T=T)
    G, D = gpu_decoder(W, g, p, 2, T, streaming=True)   # path buffer for a whole-stream backtrack
    chans = [D.stream_create() for _ in range(2)]
    D.stream_advance(chans, _cuda(lp[:, :chunk]), np.full(2, chunk, np.int32), want_partial=True)
    D.arm_barrier_timeout(LIMIT_NS)
    _expect_timeout(W, lambda: D.stream_advance(chans, _cuda(lp[:, chunk:2 * chunk]),
                                                np.full(2, chunk, np.int32), want_partial=True))
    # the abandoned call closed every channel: the stream starts over
    with pytest.raises(W.WfstError):
        D.stream_advance(chans, _cuda(lp[:, :chunk]), np.full(2, chunk, np.int32))
    chans = [D.stream_create() for _ in range(2)]
    assert sorted(chans) == [0, 1]
    for s in range(0, T, chunk):
        D.stream_advance(chans, _cuda(lp[:, s:s + chunk]), np.full(2, chunk, np.int32), want_partial=False)
    fin = D.stream_finalize(chans)
    OG = oracle.Graph(g)
    for i in range(2):
        ref = oracle_lane(OG, lp[i], T, p, streaming=True)
        assert_lane_equal(fin[i], ref, f"stream {i} after timeout")
