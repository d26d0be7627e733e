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


class RecordingTarget(SyntheticTarget):
    """The synthetic target, recording which positions' taps the driver asks for."""

    def __init__(self, cfg, agree):
        super().__init__(cfg, agree=agree)
        self.tap_calls = []

    def taps(self, req, pos0, count):
        self.tap_calls.append((req, pos0, count))
        return super().taps(req, pos0, count)


class RandomDraftSession(FakeSession):
    """Fresh random drafts and confidences every call (the synthetic target agrees with each draft
    with its probability p, so blocks are accepted at many lengths)."""

    def __init__(self, cfg, rng):
        super().__init__(cfg, None, None)
        self.rng = rng

    def draft(self, reqs, anchors, logits=False):
        self.drafted_anchors.append(list(anchors))
        n = self.cfg.n_draft
        d = self.rng.integers(0, self.cfg.vocab, size=(len(reqs), n), dtype=np.int32)
        c = self.rng.uniform(0.0, 1.0, size=(len(reqs), n)).astype(np.float32)
        return {"rc": 0, "tokens": d, "conf": c}


def test_closed_loop_many_rounds_bookkeeping():
    """Twenty rounds of four requests with random blocks, with and without pruning: every committed
    position's taps are appended exactly once and in order; each round commits the anchor and the
    accepted drafts (each equal to the target's token there); the bonus token is the next anchor."""
    c = cfg()
    for min_conf in (None, 0.3):
        rng = np.random.default_rng(11)
        target = RecordingTarget(c, agree=0.7)
        s = RandomDraftSession(c, rng)
        loop = ClosedLoop(s, target, min_conf=min_conf)
        prompts = {0: 8, 1: 1, 2: 5, 3: 13}
        for b, p in prompts.items():
            loop.start(b, p, anchor=20 + b)
        expect_committed = {b: [] for b in prompts}
        seen_a = set()
        for r in range(20):
            anchors_before = {b: loop.req[b].anchor for b in prompts}
            res = loop.step()
            assert s.drafted_anchors[-1] == [anchors_before[b] for b in sorted(prompts)]
            for i, b in enumerate(sorted(prompts)):
                a, keep = int(res.accepted[i]), int(res.keep[i])
                assert 0 <= a <= keep <= c.n_draft
                if min_conf is None:
                    assert keep == c.n_draft
                assert list(res.drafts[i][:a]) == list(res.targets[i][:a])
                assert a == keep or res.drafts[i][a] != res.targets[i][a]
                assert res.next_anchor[i] == res.targets[i][a]
                seen_a.add(a)
                expect_committed[b] += [anchors_before[b]] + [int(x) for x in res.drafts[i][:a]]
            loop.commit(res)
            for i, b in enumerate(sorted(prompts)):
                assert loop.req[b].anchor == res.next_anchor[i]
                assert loop.req[b].committed == expect_committed[b]
        assert len(seen_a) >= 3           # short and long accepted prefixes both occurred
        # taps: per request one contiguous run of positions 0 .. prompt + committed - 1 (the last
        # round's commits are still pending), each position once
        for b, p in prompts.items():
            calls = [(p0, n) for rb, p0, n in target.tap_calls if rb == b]
            pos = 0
            for p0, n in calls:
                assert p0 == pos and n > 0
                pos += n
            assert pos == loop.req[b].pos == p + len(expect_committed[b]) - loop.req[b].pending


class GreedyTarget(SyntheticTarget):
    """A deterministic stand-in target: its greedy token at position q of request b is a fixed hash
    f(b, q), whatever came before. It tracks the position of each request's anchor itself."""

    def __init__(self, cfg, prompts):
        super().__init__(cfg)
        self.q = {b: p - 1 for b, p in prompts.items()}      # the anchor is the prompt's last token

    def f(self, b, q):
        return int((b * 1000003 + q * 7919 + 17) % self.cfg.vocab)

    def verify(self, rnd, b, drafts):
        q = self.q[b]
        t = np.array([self.f(b, q + 1 + k) for k in range(self.cfg.n_draft + 1)], dtype=np.int32)
        a = 0
        while a < len(drafts) and drafts[a] == t[a]:
            a += 1
        self.q[b] = q + a + 1                                  # a drafts and the bonus token commit
        return t


class PeekingSession(FakeSession):
    """Drafts that equal the target's tokens with probability 0.6 each, else random."""

    def __init__(self, cfg, target, rng):
        super().__init__(cfg, None, None)
        self.t, self.rng = target, rng

    def draft(self, reqs, anchors, logits=False):
        n = self.cfg.n_draft
        d = self.rng.integers(0, self.cfg.vocab, size=(len(reqs), n)).astype(np.int32)
        for i, b in enumerate(reqs):
            for k in range(n):
                if self.rng.uniform() < 0.6:
                    d[i, k] = self.t.f(b, self.t.q[b] + 1 + k)
        return {"rc": 0, "tokens": d, "conf": self.rng.uniform(0.0, 1.0, size=(len(reqs), n)).astype(np.float32)}


def test_closed_loop_output_is_the_targets_greedy_sequence():
    """Greedy speculative decoding changes only how many tokens a round commits, never which: with
    random drafts, with and without confidence pruning (which keeps position 0 and only shortens
    what the target verifies), every request's committed tokens are the target's own greedy
    sequence from the prompt's last token on."""
    c = cfg()
    prompts = {0: 8, 1: 3, 2: 6}
    for min_conf in (None, 0.5):
        target = GreedyTarget(c, prompts)
        loop = ClosedLoop(PeekingSession(c, target, np.random.default_rng(5)), target, min_conf=min_conf)
        for b, p in prompts.items():
            loop.start(b, p, anchor=target.f(b, p - 1))
        lengths = []
        for _ in range(25):
            res = loop.step()
            if min_conf is not None:
                assert np.all(res.keep >= 1)
            loop.commit(res)
            lengths += [int(x) + 1 for x in res.accepted]
        for b, p in prompts.items():
            got = loop.req[b].committed + [loop.req[b].anchor]
            assert got == [target.f(b, p - 1 + j) for j in range(len(got))]
        assert max(lengths) > 1 and min(lengths) == 1        # rounds of several tokens and of one
