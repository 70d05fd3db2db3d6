"""Blank-skip frame pre-slicing on the GPU (a pre-pass outside the decoder,
"GPU WFST Beam-Search Decoder" §3) against the oracle's rule: kept rows,
counts and frame maps bit-exact, for fp32 and fp16, strided inputs, ragged
and zero lengths; then the packed output decodes like the oracle's rows."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_common import assert_lane_equal, wl_params

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def W():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import wfst_beam_search_gb300 as W
    W.load()
    return W


def _blanky_log_probs(seed, B, T, V, p_frame=0.6):
    """log_softmax of N(0, 1) logits with a large blank boost on a random
    subset of frames, so that a fair share of frames pass 0.98."""
    rng = np.random.default_rng(seed)
    logits = rng.normal(0.0, 1.0, size=(B, T, V))
    boost = rng.random((B, T)) < p_frame
    logits[..., 0] += np.where(boost, rng.uniform(2.0, 14.0, size=(B, T)), 0.0)
    m = logits.max(-1, keepdims=True)
    return logits - m - np.log(np.exp(logits - m).sum(-1, keepdims=True))


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_blank_skip_matches_oracle(W, dtype):
    B, T, V = 9, 700, 37
    lp = _blanky_log_probs(1, B, T, V).astype(dtype)
    lens = np.array([700, 0, 1, 699, 513, 2, 700, 64, 300], np.int32)
    for thr in (0.98, 0.5, 0.999):
        dev = torch.from_numpy(lp).to("cuda:0")
        out, out_lens, fmap = W.blank_skip(dev, lens, threshold=thr)
        torch.cuda.synchronize()
        out, out_lens, fmap = out.cpu().numpy(), out_lens.cpu().numpy(), fmap.cpu().numpy()
        rows, frames = oracle.blank_skip(lp, lens, thr)
        for b in range(B):
            n = len(frames[b])
            assert out_lens[b] == n, (thr, b)
            assert np.array_equal(fmap[b, :n], frames[b]) and np.all(fmap[b, n:] == -1), (thr, b)
            assert np.array_equal(out[b, :n].view(np.uint8), rows[b].view(np.uint8)), (thr, b)
        assert 0 < out_lens.sum() < lens.sum()


def test_blank_skip_strided_input_and_blank_id(W):
    """A [B, T, V] view with padded rows and lanes (stride_t > V), blank id 3."""
    B, T, V = 4, 257, 20
    big = _blanky_log_probs(2, B, T + 3, V + 12).astype(np.float32)
    big[..., [0, 8]] = big[..., [8, 0]]               # the boosted symbol is id 3 of the view
    dev_big = torch.from_numpy(big).to("cuda:0")
    view = dev_big[:, 2:2 + T, 5:5 + V]
    host = big[:, 2:2 + T, 5:5 + V]
    lens = np.array([257, 100, 0, 256], np.int32)
    out, out_lens, fmap = W.blank_skip(view, lens, threshold=0.9, blank_id=3)
    torch.cuda.synchronize()
    rows, frames = oracle.blank_skip(host, lens, 0.9, blank=3)
    out, out_lens, fmap = out.cpu().numpy(), out_lens.cpu().numpy(), fmap.cpu().numpy()
    for b in range(B):
        n = len(frames[b])
        assert out_lens[b] == n
        assert np.array_equal(fmap[b, :n], frames[b])
        assert np.array_equal(out[b, :n], rows[b])


def test_blank_skip_then_decode(W):
    """The packed output of the pre-pass decodes like the oracle decodes the
    oracle's kept rows (workload 1's graph, 8 lanes)."""
    wl = synth.workload(1)
    g = synth.make_graph(1)
    B, T = 8, 200
    lp = _blanky_log_probs(3, B, T, wl.V).astype(np.float32)
    lens = np.array([200, 150, 199, 1, 0, 200, 77, 128], np.int32)
    p = wl_params(wl, lattice=False)
    dev = torch.from_numpy(lp).to("cuda:0")
    out, out_lens, _ = W.blank_skip(dev, lens, threshold=0.98)
    kept = out_lens.cpu().numpy()
    G = W.Graph(g, device=0)
    D = W.Decoder(G, W.make_params(p["search_beam"], p["output_beam"], p["min_active"], p["max_active"],
                                   True, False), B, T)
    res = D.decode(out, kept)
    rows, _ = oracle.blank_skip(lp, lens, 0.98)
    OG = oracle.Graph(g)
    for b in range(B):
        assert kept[b] == len(rows[b])
        ref = oracle.decode(OG, rows[b], int(kept[b]), oracle.params(**p))
        assert_lane_equal(res[b], ref, f"lane {b}")
