"""Streaming channels on the GPU against the oracle's online decoding:
per-chunk partial hypotheses, final results and lattices, channel lifecycle."""
import os

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_common import SCORE_TOL, assert_lane_equal, assert_lattice_equal, gpu_decoder, wl_params

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def W():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import wfst_beam_search_gb300 as W
    W.load()
    return W


def _run_stream(W, D, lp, lens, chunk, channels):
    n = len(channels)
    partials = []
    T = int(lens.max())
    for s in range(0, T, chunk):
        cl = np.clip(lens - s, 0, chunk).astype(np.int32)
        lpc = torch.from_numpy(np.ascontiguousarray(lp[:, s:s + chunk])).to("cuda:0")
        partials.append(D.stream_advance(channels, lpc, cl, want_partial=True))
    final = D.stream_finalize(channels)
    return partials, final


def _oracle_stream(OG, p, lp, length, chunk, T):
    d = oracle.Decoder(OG, oracle.params(**p), None)
    parts = []
    for s in range(0, T, chunk):
        cl = max(0, min(chunk, length - s))
        if cl:
            d.advance(lp[s:s + cl].astype(np.float32))
        parts.append(d.partial())
    r = d.finalize()
    return parts, r, (d.lattice() if p["lattice"] else None)


def test_workload4_streaming_partials_final_lattice(W):
    wl = synth.workload(4)
    g = synth.make_graph(4)
    n_ch = 6
    lens = synth.make_lens(4)[:n_ch]
    lp = synth.make_log_probs(4, lanes=range(n_ch))
    p = wl_params(wl)
    G, D = gpu_decoder(W, g, p, n_ch, wl.T, streaming=True)
    channels = [D.stream_create() for _ in range(n_ch)]
    assert sorted(channels) == list(range(n_ch))
    partials, final = _run_stream(W, D, lp, lens, wl.chunk, channels)
    OG = oracle.Graph(g)
    T = int(lens.max())
    for i in (0, 1):
        parts, r, lat = _oracle_stream(OG, p, lp[i], int(lens[i]), wl.chunk, T)
        for k, (gp, op) in enumerate(zip(partials, parts)):
            assert gp[i]["ok"] == op["ok"], f"channel {i} chunk {k}"
            assert list(gp[i]["words"]) == list(op["words"]), f"channel {i} chunk {k} partial words"
            assert abs(gp[i]["score"] - op["score"]) <= SCORE_TOL, f"channel {i} chunk {k} partial score"
        assert_lane_equal(final[i], r, f"channel {i} final")
        assert_lattice_equal(D.lattice(channels[i]), lat, f"channel {i} lattice")
    for c in channels:
        D.stream_release(c)


def test_stream_lifecycle_and_chunking_invariance(W):
    wl = synth.workload(1)
    g = synth.make_graph(1)
    p = wl_params(wl, lattice=True)
    lp = synth.make_log_probs(1, lanes=range(3), T=48)
    lens = np.array([48, 30, 5], np.int32)
    G, D = gpu_decoder(W, g, p, 3, 64, streaming=True)
    chans = [D.stream_create() for _ in range(3)]
    assert D.stream_create() == -1          # every channel busy
    _, f16 = _run_stream(W, D, lp, lens, 16, chans)
    lat16 = [D.lattice(c) for c in chans]
    for c in chans:
        D.stream_release(c)
    chans = [D.stream_create() for _ in range(3)]
    _, f5 = _run_stream(W, D, lp, lens, 5, chans)
    OG = oracle.Graph(g)
    for i, c in enumerate(chans):
        assert list(f5[i]["words"]) == list(f16[i]["words"]) and f5[i]["score"] == f16[i]["score"]
        _, r, lat = _oracle_stream(OG, p, lp[i], int(lens[i]), 48, 48)
        assert_lane_equal(f5[i], r, f"lifecycle channel {i}")
        assert_lattice_equal(D.lattice(c), lat, f"lifecycle lattice {i}")
        assert_lattice_equal(lat16[i], lat, f"lifecycle lattice chunk16 {i}")
    for c in chans:
        D.stream_release(c)


def test_workload4_full_128_channels_every_channel(W):
    """The streaming workload in the launch configuration the benchmark times:
    128 channels, 16-frame chunks, partials every chunk, lattices.  Every
    channel's every partial, its final result and its lattice equal the
    oracle's online decode of the same chunks (oracle channels on host
    threads)."""
    wl = synth.workload(4)
    g = synth.make_graph(4)
    lens = synth.make_lens(4)
    lp = synth.make_log_probs(4)
    p = wl_params(wl)
    G, D = gpu_decoder(W, g, p, wl.B, wl.T, streaming=True)
    channels = [D.stream_create() for _ in range(wl.B)]
    partials, final = _run_stream(W, D, lp, lens, wl.chunk, channels)
    assert all(f["ok"] and f["overflow"] == 0 for f in final)
    lats = [D.lattice(c) for c in channels]
    OG = oracle.Graph(g)
    T = int(lens.max())
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=max(1, min(os.cpu_count() or 1, 32))) as ex:
        refs = list(ex.map(lambda i: _oracle_stream(OG, p, lp[i], int(lens[i]), wl.chunk, T), range(wl.B)))
    for i, (parts, r, lat) in enumerate(refs):
        assert len(parts) == len(partials)
        for k, op in enumerate(parts):
            gp = partials[k][i]
            assert gp["ok"] == op["ok"], f"channel {i} chunk {k}"
            assert list(gp["words"]) == list(op["words"]), f"channel {i} chunk {k} partial words"
            if op["ok"]:
                assert abs(gp["score"] - op["score"]) <= SCORE_TOL, f"channel {i} chunk {k} partial score"
        assert_lane_equal(final[i], r, f"channel {i} final")
        assert_lattice_equal(lats[i], lat, f"channel {i} lattice")
    for c in channels:
        D.stream_release(c)


def test_streaming_search_matches_oracle_and_restarts_on_overflow(W):
    """StreamingSearch on real channels: without overflow its per-chunk words
    and final result are the oracle's streaming results; on a decoder whose
    frontier capacity is far too small, flagged chunks restart the channel
    and the stream still ends with a result."""
    wl = synth.workload(0)
    g = synth.make_graph(0)
    T, chunk = 300, 16
    lp = synth.make_lane_log_probs(0, 3, T=T)
    p = wl_params(wl, lattice=False)
    G, D = gpu_decoder(W, g, p, 2, chunk, caps=W.Capacity(0, 0, 0, 4096), streaming=True)
    s = W.StreamingSearch(D)
    outs = [s.feed(torch.from_numpy(np.ascontiguousarray(lp[t:t + chunk])).to("cuda:0"))
            for t in range(0, T, chunk)]
    f = s.finish()
    parts, r, _ = _oracle_stream(oracle.Graph(g), p, lp, T, chunk, T)
    assert f["restarts"] == 0
    for k, (o, op) in enumerate(zip(outs, parts)):
        assert o["words"] == list(op["words"]), f"chunk {k}"
    assert f["words"] == list(r["words"]) and abs(f["score"] - r["score"]) <= SCORE_TOL
    _, D2 = gpu_decoder(W, g, p, 2, chunk, caps=W.Capacity(4, 0, 0, 4096), graph=G, streaming=True)
    s2 = W.StreamingSearch(D2)
    for t in range(0, T, chunk):
        s2.feed(torch.from_numpy(np.ascontiguousarray(lp[t:t + chunk])).to("cuda:0"))
    f2 = s2.finish()
    assert s2.restarts > 0 and isinstance(f2["words"], list)

