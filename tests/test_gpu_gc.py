"""Winners-log GC (params.gc_interval > 0) on the GPU against the oracle.

The GC turns each lane's winners log into a ring and, every gc_interval
frames, cuts every chain at the lane's convergence point, moving the words
below it into a finalized list ("GPU WFST Beam-Search Decoder", §6.3
"Winners-log GC for long-form audio" and §8.1 "Per-chunk GC").  It must not
change any result: partial hypotheses per chunk, final words and scores equal
the oracle's (which keeps every frame), while the ring holds only a small part
of the entries the stream appends, so it wraps many times."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_common import SCORE_TOL, assert_lane_equal, wl_params

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def W():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import wfst_beam_search_gb300 as W
    W.load()
    return W


def _params(W, p, streaming, gc, options=0):
    return W.make_params(p["search_beam"], p["output_beam"], p["min_active"], p["max_active"],
                         p["allow_partial"], False, streaming, options, gc_interval=gc)


def _stream(W, D, lp, lens, chunk, channels):
    partials = []
    for s in range(0, int(lens.max()), chunk):
        cl = np.clip(lens - s, 0, chunk).astype(np.int32)
        lpc = torch.from_numpy(np.ascontiguousarray(lp[:, s:s + chunk])).to("cuda:0")
        partials.append(D.stream_advance(channels, lpc, cl, want_partial=True))
    return partials, D.stream_finalize(channels)


def _oracle_stream(OG, p, lp, length, chunk, T):
    d = oracle.Decoder(OG, oracle.params(**p), None)
    parts = []
    for s in range(0, T, chunk):
        cl = max(0, min(chunk, length - s))
        if cl:
            d.advance(np.ascontiguousarray(lp[s:s + cl], dtype=np.float32))
        parts.append(d.partial())
    r = d.finalize()
    return parts, r, d.stats()


def _check_stream(partials, final, i, parts, r, where, every=1):
    for k in range(0, len(parts), every):
        gp, op = partials[k][i], parts[k]
        assert gp["ok"] == op["ok"], f"{where} chunk {k}: ok"
        assert gp["overflow"] == 0, f"{where} chunk {k}: overflow {gp['overflow']}"
        assert list(gp["words"]) == list(op["words"]), f"{where} chunk {k}: partial words"
        assert abs(gp["score"] - op["score"]) <= SCORE_TOL, f"{where} chunk {k}: partial score"
    assert_lane_equal(final[i], r, f"{where} final")


def _peaky_log_probs(seed, n, T, V, boost):
    """[n, T, V] log-posteriors with one boosted symbol per frame (blank in
    70% of frames): a sharper CTC output than the workloads' recipe."""
    rng = np.random.default_rng(seed)
    logits = rng.normal(0.0, 1.0, size=(n, T, V))
    top = np.where(rng.random((n, T)) < 0.7, 0, rng.integers(1, V, size=(n, T)))
    np.put_along_axis(logits, top[..., None], np.take_along_axis(logits, top[..., None], -1) + boost, -1)
    m = logits.max(-1, keepdims=True)
    return (logits - m - np.log(np.exp(logits - m).sum(-1, keepdims=True))).astype(np.float32)


def test_gc_long_stream_ring_wraps(W):
    """One channel on the 200-state graph for 6000 frames in 16-frame chunks,
    GC every chunk, through a ring of 65536 entries: the stream appends about
    18 rings' worth of entries."""
    wl = synth.workload(0)
    g = synth.make_graph(0)
    T, chunk, ring = 6000, 16, 1 << 16
    lp = synth.make_lane_log_probs(0, 0, T=T)[None]
    lens = np.array([T], np.int32)
    p = wl_params(wl, lattice=False)
    G = W.Graph(g, device=0)
    D = W.Decoder(G, _params(W, p, True, 16), 1, chunk, W.Capacity(0, ring, 0, 4096, 0))
    assert D.mem_stats()["log_cap"] == ring
    ch = D.stream_create()
    partials, final = _stream(W, D, lp, lens, chunk, [ch])
    parts, r, st = _oracle_stream(oracle.Graph(g), p, lp[0], T, chunk, T)
    assert st["tokens"] > 10 * ring, st["tokens"]
    assert len(r["words"]) > 100
    _check_stream(partials, final, 0, parts, r, "long stream")
    D.stream_release(ch)


def _eps_graph(seed):
    """A small graph with epsilon arcs (to higher state ids: acyclic) and a
    blank self-loop on every state, so that long streams keep a frontier."""
    rng = np.random.default_rng(seed)
    N, V = 40, 8
    t = synth.random_tiny_graph(rng, N, V, max_deg=3, p_eps=0.3, p_final=0.3, dyadic=False)
    rs = np.asarray(t["row_splits"])
    src = np.repeat(np.arange(N), np.diff(rs))
    src = np.concatenate([src, np.arange(N)])
    dst = np.concatenate([np.asarray(t["dst"]), np.arange(N)])
    il = np.concatenate([np.asarray(t["ilabel"]), np.zeros(N, np.int64)])
    ol = np.concatenate([np.asarray(t["olabel"]), np.zeros(N, np.int64)])
    w = np.concatenate([np.asarray(t["weight"]), np.zeros(N)])
    order = np.argsort(src, kind="stable")
    return synth.graph_from_arcs(N, V, src[order], dst[order], il[order], ol[order], w[order],
                                 np.asarray(t["final"], np.float32))


def test_gc_epsilon_graph_stream(W):
    """Epsilon chains (several entries per frame on one path) through a
    1024-entry ring, 2000 frames in chunks of 7, GC every 4 frames."""
    g = _eps_graph(7)
    T, chunk, ring = 2000, 7, 1 << 10
    lp = _peaky_log_probs(2, 1, T, 8, 6.0)
    lens = np.array([T], np.int32)
    p = dict(search_beam=10.0, output_beam=0.0, min_active=0, max_active=20, allow_partial=True,
             lattice=False)
    G = W.Graph(g, device=0)
    assert G.has_eps
    D = W.Decoder(G, _params(W, p, True, 4), 1, chunk, W.Capacity(0, ring, 0, 4096, 0))
    ch = D.stream_create()
    partials, final = _stream(W, D, lp, lens, chunk, [ch])
    parts, r, st = _oracle_stream(oracle.Graph(g), p, lp[0], T, chunk, T)
    assert st["tokens"] > 4 * ring, st["tokens"]
    assert len(r["words"]) > 20
    _check_stream(partials, final, 0, parts, r, "epsilon stream")
    D.stream_release(ch)


def test_gc_offline_log_smaller_than_an_utterance(W):
    """Offline decodes of 8 lanes x 2000 frames on the 200-state graph (about
    190 tokens per frame) through a 65536-entry log with growth turned off:
    without GC every lane overflows the log; with GC every 16 frames the
    results equal the oracle's, and stay so when the decoder is reused."""
    wl = synth.workload(0)
    g = synth.make_graph(0)
    B, T = 8, 2000
    lp = np.stack([synth.make_lane_log_probs(0, b, T=T) for b in range(B)])
    lens = np.full(B, T, np.int32)
    lens[3] = 1500
    p = wl_params(wl, lattice=False)
    G = W.Graph(g, device=0)
    caps = W.Capacity(0, 1 << 16, 0, 4096, 0)
    dev = torch.from_numpy(lp).to("cuda:0")
    D0 = W.Decoder(G, _params(W, p, False, 0, W.OPT_NO_GROW), B, T, caps)
    assert all(r["overflow"] & W.OVF_ARENA for r in D0.decode(dev, lens))
    D = W.Decoder(G, _params(W, p, False, 16, W.OPT_NO_GROW), B, T, caps)
    out = D.decode(dev, lens)
    OG = oracle.Graph(g)
    for b in range(B):
        assert_lane_equal(out[b], oracle.decode(OG, lp[b], int(lens[b]), oracle.params(**p)), f"lane {b}")
    again = D.decode(dev, lens)
    for b in range(B):
        assert list(again[b]["words"]) == list(out[b]["words"]) and again[b]["score"] == out[b]["score"]


def test_gc_rejects_lattice_and_negative_interval(W):
    g = synth.make_graph(0)
    G = W.Graph(g, device=0)
    with pytest.raises(W.WfstError, match="INVALID_ARG"):
        W.Decoder(G, W.make_params(lattice=True, gc_interval=8), 1, 16)
    with pytest.raises(W.WfstError, match="INVALID_ARG"):
        W.Decoder(G, W.make_params(gc_interval=-1), 1, 16)


def test_gc_channel_reuse_and_ragged_channels(W):
    """Two channels of one GC decoder with different lengths, released and
    opened again for a second pair of streams: each stream starts from an
    empty finalized list and a fresh root, and every partial and final result
    equals the oracle's."""
    wl = synth.workload(0)
    g = synth.make_graph(0)
    p = wl_params(wl, lattice=False)
    G = W.Graph(g, device=0)
    D = W.Decoder(G, _params(W, p, True, 16), 2, 16, W.Capacity(0, 1 << 16, 0, 4096, 0))
    OG = oracle.Graph(g)
    for rnd, T in enumerate((3000, 1000)):
        lp = np.stack([synth.make_lane_log_probs(0, 10 + 2 * rnd + i, T=T) for i in range(2)])
        lens = np.array([T, T // 2 + 3], np.int32)
        chans = [D.stream_create(), D.stream_create()]
        partials, final = _stream(W, D, lp, lens, 16, chans)
        for i in range(2):
            parts, r, _ = _oracle_stream(OG, p, lp[i], int(lens[i]), 16, T)
            _check_stream(partials, final, i, parts, r, f"round {rnd} channel {i}", every=7)
        for c in chans:
            D.stream_release(c)


def test_gc_bounds_the_log_on_workload2_lanes(W):
    """Workload 2 (2M states, B=3 lanes x 500 frames): on an epsilon-free
    graph the GC tracks every token's ancestor among a checkpoint frame's
    tokens and cuts once all of a frame's tokens share one; the results equal
    the decode without GC, and the most log entries held live fall to about
    half (the chains converge 40-170 frames back on this workload)."""
    wl = synth.workload(2)
    g = synth.make_graph(2)
    lanes = [0, 1, 2]
    lp = synth.make_log_probs(2, lanes=lanes)
    lens = np.full(3, wl.T, np.int32)
    G = W.Graph(g, device=0)
    res = {}
    for gi in (0, 16):
        params = W.make_params(wl.search_beam, wl.output_beam, wl.min_active, wl.max_active, True, False, False,
                               0, gi)
        D = W.Decoder(G, params, 3, wl.T)
        out = D.decode(torch.from_numpy(lp).to("cuda:0"), lens)
        res[gi] = (out, D.stats()["log_high_water"])
        D.close()
    (o0, hw0), (o16, hw16) = res[0], res[16]
    for b in range(3):
        assert o16[b]["overflow"] == 0 and list(o16[b]["words"]) == list(o0[b]["words"])
        assert o16[b]["score"] == o0[b]["score"]
    assert hw16 < 0.6 * hw0, (hw16, hw0)
