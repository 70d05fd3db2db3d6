"""The caller-side overflow policy of StreamingSearch (page "GPU WFST
Beam-Search Decoder", §7 overflow handling and §8.1): a chunk that comes
back flagged abandons its channel, keeps the hypothesis from before that
chunk as a prefix and runs the chunk once more on a newly opened channel.
Checked on the CPU against a scripted stand-in for the streaming decoder calls."""
import numpy as np

import wfst_beam_search_gb300 as W


class ScriptedDecoder:
    """Channels that emit one word per chunk (the chunk's first value); a
    channel overflows on the chunks listed in `burst` of its own life."""

    def __init__(self, burst=(), n_channels=2):
        self.burst = set(burst)
        self.free = list(range(n_channels))
        self.open = {}
        self.log = []

    def stream_create(self):
        if not self.free:
            return -1
        ch = self.free.pop(0)
        self.open[ch] = dict(words=[], chunks=0)
        self.log.append(("create", ch))
        return ch

    def stream_release(self, ch):
        del self.open[ch]
        self.free.append(ch)
        self.log.append(("release", ch))

    def stream_advance(self, chans, lp, lens, want_partial=True, words_cap=4096):
        (ch,) = chans
        st = self.open[ch]
        st["chunks"] += 1
        st["words"].append(int(lp[0][0][0]))
        ovf = W.OVF_KEPT if (st["chunks"] in self.burst and ch == 0) else 0
        self.log.append(("advance", ch, int(lp[0][0][0])))
        return [dict(words=np.array(st["words"], np.int32), score=-float(len(st["words"])), ok=1,
                     overflow=ovf)]

    def stream_finalize(self, chans, words_cap=4096):
        (ch,) = chans
        st = self.open[ch]
        return [dict(words=np.array(st["words"], np.int32), score=-1.0, ok=1, reached_final=1,
                     overflow=0)]


def _chunk(word):
    return np.full((4, 3), word, np.float32)


def test_no_overflow_keeps_one_channel():
    d = ScriptedDecoder()
    s = W.StreamingSearch(d)
    for w in (11, 12, 13):
        r = s.feed(_chunk(w))
    assert r["words"] == [11, 12, 13] and r["restarts"] == 0
    f = s.finish()
    assert f["words"] == [11, 12, 13] and f["restarts"] == 0
    assert d.log == [("create", 0), ("advance", 0, 11), ("advance", 0, 12), ("advance", 0, 13),
                     ("release", 0)]


def test_overflowed_chunk_is_decoded_again_on_a_fresh_channel():
    d = ScriptedDecoder(burst={3})
    s = W.StreamingSearch(d)
    outs = [s.feed(_chunk(w)) for w in (21, 22, 23, 24)]
    # chunk 3 overflowed on channel 0: channel 0 is dropped, its words before
    # that chunk become the prefix, chunk 3 runs again on channel 1
    assert outs[1]["words"] == [21, 22]
    assert outs[2]["words"] == [21, 22, 23] and outs[2]["restarts"] == 1 and outs[2]["overflow"] == 0
    assert outs[3]["words"] == [21, 22, 23, 24]
    f = s.finish()
    assert f["words"] == [21, 22, 23, 24] and f["restarts"] == 1
    assert ("release", 0) in d.log and ("advance", 1, 23) in d.log
    assert d.log.index(("release", 0)) < d.log.index(("advance", 1, 23))
    assert sorted(d.free) == [0, 1]
