"""Host bookkeeping of the closed-loop driver (no GPU): which context rows are appended when,
what commits, and how pruning caps acceptance. A fake session stands in for the C ABI; the
acceptance and pruning decisions come from the oracle's pinned functions."""
import numpy as np

import oracle
from dflash_synth import DraftConfig
from speculative_block_draft_gb300.driver import ClosedLoop, SyntheticTarget


class FakeSession:
    def __init__(self, cfg, drafts, conf):
        self.cfg = cfg
        self.drafts, self.conf = drafts, conf
        self.projected = []          # (req_ids, counts, taps rows)
        self.drafted_anchors = []

    def project(self, reqs, counts, taps):
        self.projected.append((list(reqs), list(counts), taps.shape[0]))
        return 0

    def draft(self, reqs, anchors, logits=False):
        self.drafted_anchors.append(list(anchors))
        return {"rc": 0, "tokens": self.drafts[: len(reqs)].copy(), "conf": self.conf[: len(reqs)].copy()}

    def draft_lengths(self, conf, thresholds, min_conf):
        return np.array([oracle.draft_length(c, thresholds, min_conf) for c in conf], dtype=np.int32)

    def accept(self, d, t):
        r = [oracle.accept(d[i], t[i]) for i in range(d.shape[0])]
        return np.array([x[0] for x in r], np.int32), np.array([x[1] for x in r], np.int32)

    def accept_kept(self, d, keep, t):
        r = [oracle.accept_kept(d[i], t[i], keep[i]) for i in range(d.shape[0])]
        return np.array([x[0] for x in r], np.int32), np.array([x[1] for x in r], np.int32)


def cfg():
    return DraftConfig("drv", n_layers=1, d=64, n_q_heads=1, n_kv_heads=1, head_dim=64, inter=64, n_taps=1,
                       target_hidden=64, vocab=100, gamma=5, window=0, ctx_len=8, wdtype="f32", adtype="f32",
                       seed=3)


def test_closed_loop_appends_committed_rows():
    c = cfg()
    drafts = np.array([[1, 2, 3, 4], [5, 6, 7, 8]], np.int32)
    conf = np.full((2, 4), 0.9, np.float32)
    s = FakeSession(c, drafts, conf)
    loop = ClosedLoop(s, SyntheticTarget(c))
    loop.start(0, 8, anchor=11)
    loop.start(1, 3, anchor=12)
    # round 0: the prompts are appended, then the blocks drafted from the anchors
    t = np.array([[1, 2, 9, 9, 9], [5, 6, 7, 8, 40]], np.int32)
    res = loop.step(targets=t)
    assert s.projected[-1][:2] == ([0, 1], [8, 3]) and s.drafted_anchors[-1] == [11, 12]
    assert list(res.accepted) == [2, 4] and list(res.next_anchor) == [9, 40]
    loop.commit(res)
    assert loop.req[0].committed == [11, 1, 2] and loop.req[1].committed == [12, 5, 6, 7, 8]
    # round 1: a + 1 committed positions of each request are appended at the right offsets
    res = loop.step(targets=np.zeros((2, 5), np.int32))
    assert s.projected[-1][:2] == ([0, 1], [3, 5]) and s.drafted_anchors[-1] == [9, 40]
    assert loop.req[0].pos == 11 and loop.req[1].pos == 8


def test_closed_loop_pruning_caps_acceptance():
    c = cfg()
    drafts = np.array([[1, 2, 3, 4]], np.int32)
    conf = np.array([[0.9, 0.8, 0.1, 0.9]], np.float32)     # position 2 is below 0.5: keep 2
    s = FakeSession(c, drafts, conf)
    loop = ClosedLoop(s, SyntheticTarget(c), min_conf=0.5)
    loop.start(0, 4, anchor=7)
    res = loop.step(targets=np.array([[1, 2, 3, 4, 5]], np.int32))   # the target agrees everywhere
    assert list(res.keep) == [2] and list(res.accepted) == [2] and list(res.next_anchor) == [3]
    loop.commit(res)
    assert loop.req[0].pending == 3 and loop.req[0].anchor == 3
