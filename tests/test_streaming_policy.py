"""The caller-side overflow policy of StreamingSearch (page "GPU WFST
Beam-Search Decoder", §7 overflow handling and §8.1): a chunk that comes
back flagged abandons its channel, keeps the hypothesis from before that
chunk as a prefix and runs the chunk once more on a newly opened channel.
Checked on the CPU against a scripted stand-in for the streaming decoder calls."""
import numpy as np
import pytest

import wfst_beam_search_gb300 as W


class ScriptedDecoder:
    """Channels that emit one word per chunk (the chunk's first value); a
    channel overflows on the chunks listed in `burst` of its own life."""

    def __init__(self, burst=(), n_channels=2, bits=None, final_ok=1):
        # burst: chunk numbers (of a channel's own life) on which channel 0
        # overflows, or {channel: chunk numbers}
        self.burst = {c: set(v) for c, v in burst.items()} if isinstance(burst, dict) else {0: set(burst)}
        self.bits = W.OVF_KEPT if bits is None else bits
        self.final_ok = final_ok
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
        ovf = self.bits if st["chunks"] in self.burst.get(ch, ()) else 0
        self.log.append(("advance", ch, int(lp[0][0][0])))
        return [dict(words=np.array(st["words"], np.int32), score=-float(len(st["words"])), ok=1,
                     overflow=ovf)]

    def stream_finalize(self, chans, words_cap=4096):
        (ch,) = chans
        st = self.open[ch]
        return [dict(words=np.array(st["words"] if self.final_ok else [], np.int32), score=-1.0,
                     ok=self.final_ok, reached_final=self.final_ok, overflow=0)]


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


def test_path_overflow_is_reported_without_a_restart():
    """Bit 32 (best path longer than the path buffer) is only reported: a new
    channel would have no larger buffer."""
    d = ScriptedDecoder(burst={2}, bits=W.OVF_PATH)
    s = W.StreamingSearch(d)
    outs = [s.feed(_chunk(w)) for w in (31, 32, 33)]
    assert outs[1]["overflow"] == W.OVF_PATH and outs[1]["restarts"] == 0
    assert s.finish()["words"] == [31, 32, 33]
    assert [e for e in d.log if e[0] == "create"] == [("create", 0)]


def test_a_retried_chunk_that_overflows_again_is_reported_and_not_kept():
    """Channel 0 overflows on chunk 2; its retry on channel 1 overflows too
    (channel 1 overflows on its first and second chunks).  The flagged retry
    is reported, and its words never become part of the finished prefix."""
    d = ScriptedDecoder(burst={0: {2}, 1: {1, 2}}, n_channels=3)
    s = W.StreamingSearch(d)
    r1 = s.feed(_chunk(41))
    r2 = s.feed(_chunk(42))
    assert r1["words"] == [41]
    assert r2["restarts"] == 1 and r2["overflow"] == W.OVF_KEPT and r2["words"] == [41, 42]
    # chunk 3 overflows channel 1 again: the restart on channel 2 keeps the
    # prefix [41] only (never the flagged [42])
    r3 = s.feed(_chunk(43))
    assert r3["restarts"] == 2 and r3["overflow"] == 0 and r3["words"] == [41, 43]


def test_failed_final_step_falls_back_to_the_last_partial():
    d = ScriptedDecoder(final_ok=0)
    s = W.StreamingSearch(d)
    for w in (51, 52):
        s.feed(_chunk(w))
    f = s.finish()
    assert f["ok"] == 0 and f["words"] == [51, 52]


def test_no_free_channel_raises():
    d = ScriptedDecoder(n_channels=0)
    with pytest.raises(RuntimeError, match="busy"):
        W.StreamingSearch(d)
