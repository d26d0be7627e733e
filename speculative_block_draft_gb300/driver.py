"""Closed-loop speculative decoding over the C ABI: the round driver either side of a draft.

A round for every active request (the loop of the DFlash pages: the target verifies the block
[anchor, d_1..d_n] and commits a + 1 tokens; the drafter's context then grows by the hidden
states of exactly those committed positions, and the bonus token becomes the next anchor):

  1. append the context rows of the positions committed by the previous verification
     (dflash_project_ctx; a + 1 rows, the first round: the prompt),
  2. draft one block from the anchor (dflash_draft_block),
  3. optionally prune the block by confidence (dflash_draft_lengths),
  4. the target verifies the kept drafts and returns its greedy tokens t_0..t_n,
  5. accept (dflash_accept / dflash_accept_kept): a, next anchor = t_a; a + 1 tokens commit.

The target is an object with two methods:
  verify(round, req, drafts) -> int32 [n + 1]   the target's greedy tokens after [anchor, drafts]
  taps(req, pos0, count)     -> [count, n_taps * H] the target's tapped hidden states at
                                positions pos0 .. pos0 + count - 1 (bf16 bits or fp32 rows)
The driver holds only host bookkeeping; every step of the round runs in the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class RoundResult:
    drafts: np.ndarray          # int32 [B, n]
    conf: np.ndarray            # float32 [B, n]
    keep: np.ndarray            # int32 [B]: drafts verified (n when not pruned)
    targets: np.ndarray         # int32 [B, n + 1]
    accepted: np.ndarray        # int32 [B]
    next_anchor: np.ndarray     # int32 [B]


@dataclass
class RequestState:
    pos: int = 0                # context rows appended to the drafter so far
    pending: int = 0            # committed positions whose rows are not appended yet
    anchor: int = 0             # last committed token
    committed: list = field(default_factory=list)


class ClosedLoop:
    """Drive rounds for requests 0..B-1 of a Session (speculative_block_draft_gb300.session)."""

    def __init__(self, session, target, thresholds=None, min_conf=None):
        self.s = session
        self.target = target
        self.thresholds = None if thresholds is None else np.asarray(thresholds, dtype=np.float32)
        self.min_conf = min_conf
        self.req: dict[int, RequestState] = {}
        self.round = 0

    @property
    def n(self) -> int:
        return self.s.cfg.n_draft

    def start(self, req: int, prompt_len: int, anchor: int):
        """A new request: its prompt's prompt_len positions are pending, anchor is its last token."""
        self.req[req] = RequestState(pos=0, pending=int(prompt_len), anchor=int(anchor))

    def _append_pending(self, reqs):
        counts = [self.req[b].pending for b in reqs]
        if sum(counts):
            rows = [self.target.taps(b, self.req[b].pos, c) for b, c in zip(reqs, counts) if c]
            rc = self.s.project(reqs, counts, np.concatenate(rows))
            if rc != 0:
                raise RuntimeError(f"dflash_project_ctx returned {rc}")
        for b, c in zip(reqs, counts):
            self.req[b].pos += c
            self.req[b].pending = 0

    def step(self, targets: np.ndarray | None = None) -> RoundResult:
        """One round for every request (appending, drafting, pruning, verifying, accepting); the
        result is committed by commit(). targets, when given, replaces the target's verification."""
        reqs = sorted(self.req)
        self._append_pending(reqs)
        anchors = np.array([self.req[b].anchor for b in reqs], dtype=np.int32)
        out = self.s.draft(reqs, anchors, logits=False)
        if out["rc"] != 0:
            raise RuntimeError(f"dflash_draft_block returned {out['rc']}")
        drafts, conf = out["tokens"], out["conf"]
        pruned = self.thresholds is not None or self.min_conf is not None
        if pruned:
            keep = self.s.draft_lengths(conf, self.thresholds, self.min_conf or 0.0)
        else:
            keep = np.full(len(reqs), self.n, dtype=np.int32)
        if targets is None:
            targets = np.stack([self.target.verify(self.round, b, drafts[i][:keep[i]]) for i, b in enumerate(reqs)])
        if pruned:
            a, nxt = self.s.accept_kept(drafts, keep, targets)
        else:
            a, nxt = self.s.accept(drafts, targets)
        return RoundResult(drafts, conf, keep, targets, a, nxt)

    def commit(self, res: RoundResult):
        """Commit a + 1 tokens per request: the anchor and the accepted drafts' positions become
        pending context rows, the bonus token becomes the next anchor."""
        for i, b in enumerate(sorted(self.req)):
            st = self.req[b]
            a = int(res.accepted[i])
            st.committed.extend([st.anchor] + [int(x) for x in res.drafts[i][:a]])
            st.pending += a + 1
            st.anchor = int(res.next_anchor[i])
        self.round += 1


class SyntheticTarget:
    """The seeded stand-in for the target model: taps from the shared generator, greedy tokens
    that agree with each draft with probability p (dflash_synth.target_tokens)."""

    def __init__(self, cfg, seed: int | None = None, agree: float | None = None):
        import dflash_synth as syn
        self.syn, self.cfg = syn, cfg
        self.seed = cfg.seed if seed is None else seed
        self.p = (cfg.agree or 0.0) if agree is None else agree

    def verify(self, rnd: int, req: int, drafts) -> np.ndarray:
        n = self.cfg.n_draft
        d = np.asarray(drafts, dtype=np.int32)
        full = np.concatenate([d, np.zeros(n - d.shape[0], np.int32)]) if d.shape[0] < n else d
        t = self.syn.target_tokens(self.seed, req, rnd, full, self.p, self.cfg.vocab)
        return np.asarray(t, dtype=np.int32)

    def taps(self, req: int, pos0: int, count: int):
        return self.syn.taps_rows(self.cfg, self.seed, req, pos0, count)
