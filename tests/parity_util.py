"""Shared GPU-vs-oracle parity harness (imported by the gpu tests and the smoke check).

Acceptance rule (the parity tolerances fixed for the drafter workloads):
  * logits max-abs <= 1e-4 (fp32 drafter) or 2e-2 (bf16 / 4-bit drafter);
  * a draft token must equal the oracle's wherever the oracle's top-1 - top-2 margin > 1e-2;
  * accept_len must equal the oracle's whenever every row up to and including the oracle's
    first mismatch has margin > 1e-2 (rows below the margin are reported, not failed);
  * confidence: |ln conf_gpu - ln conf_oracle| <= 2 * (max-abs logit error) + 1e-5. This bound
    follows from conf = 1 / sum_j exp(l_j - l_max): shifting every logit by at most e moves
    ln conf by at most 2e.
"""
from __future__ import annotations

import numpy as np

import dflash_synth as syn
import oracle

MARGIN = 1e-2


def logit_tol(cfg) -> float:
    return 1e-4 if cfg.wdtype == "f32" else 2e-2


def compare_block(cfg, gpu: dict, orc: dict, b: int, report: dict):
    lg = gpu["logits"][b].astype(np.float64)
    lo = orc["logits"]
    err = float(np.max(np.abs(lg - lo)))
    report["max_logit_err"] = max(report.get("max_logit_err", 0.0), err)
    assert err <= logit_tol(cfg), f"logit max-abs {err} > {logit_tol(cfg)}"
    confident = orc["margin"] > MARGIN
    tg, to = gpu["tokens"][b], orc["tokens"]
    assert np.array_equal(tg[confident], to[confident]), f"tokens differ at confident rows: {tg} vs {to}"
    report["low_margin_rows"] = report.get("low_margin_rows", 0) + int(np.sum(~confident))
    report["token_mismatch_low_margin"] = report.get("token_mismatch_low_margin", 0) + int(np.sum(tg != to))
    dc = np.abs(np.log(gpu["conf"][b].astype(np.float64)) - np.log(orc["conf"]))
    assert np.all(dc <= 2 * err + 1e-5), f"confidence off: {dc.max()} > {2 * err + 1e-5}"


def accept_checked(orc_tokens, gpu_tokens, margin, target, gpu_a, report):
    a_o, nxt_o = oracle.accept(orc_tokens, target)
    # rows up to and including the oracle's first mismatch must be confident
    upto = min(a_o + 1, len(orc_tokens))
    if np.all(margin[:upto] > MARGIN):
        assert gpu_a == a_o, f"accept_len {gpu_a} != oracle {a_o}"
    else:
        report["accept_unchecked"] = report.get("accept_unchecked", 0) + 1
    return a_o


class Pair:
    """The GPU session and the oracle session for one drafter, fed identical inputs."""

    def __init__(self, cfg, model, max_batch=None, ctx_capacity=None, oracle_ctx=None):
        from speculative_block_draft_gb300.session import Session
        self.cfg = cfg
        self.model = model
        self.gpu = Session(model, max_batch=max_batch or cfg.batch, ctx_capacity=ctx_capacity)
        self.orc = oracle.Oracle(model)
        self.os = oracle.OracleSession(self.orc)
        self.pos = {}
        self.oracle_ctx = oracle_ctx   # optional precomputed {req: (first_pos, k, v)}

    def taps(self, req, pos0, n):
        return syn.taps_rows(self.cfg, self.cfg.seed, req, pos0, n)

    def prefill(self, lengths):
        c = self.cfg
        reqs = list(range(len(lengths)))
        taps = [self.taps(b, 0, int(lengths[b])) for b in reqs]
        flat = np.concatenate(taps) if sum(int(x) for x in lengths) else np.zeros((0, c.n_taps * c.target_hidden))
        assert self.gpu.project(reqs, [int(x) for x in lengths], flat) == 0
        for b in reqs:
            P = int(lengths[b])
            self.pos[b] = P
            skip = P - c.window if (c.window > 0 and P > c.window) else 0
            if self.oracle_ctx is not None and b in self.oracle_ctx:
                first, k, v = self.oracle_ctx[b]
                assert first == skip and k.shape[1] == P - skip
                self.os.skip(b, skip)
                self.os.k[b], self.os.v[b] = k, v
                self.os.n_pos[b] = P
                continue
            if skip:
                self.os.skip(b, skip)
            if P - skip:
                self.os.project(b, syn.taps_to_f32(c, taps[b][skip:]).astype(np.float64))

    def append(self, counts):
        reqs = list(range(len(counts)))
        rows = [self.taps(b, self.pos[b], int(counts[b])) for b in reqs]
        assert self.gpu.project(reqs, [int(x) for x in counts], np.concatenate(rows)) == 0
        for b in reqs:
            self.pos[b] += int(counts[b])
            if int(counts[b]):
                self.os.project(b, syn.taps_to_f32(self.cfg, rows[b]).astype(np.float64))

    def round(self, r, report, check_accept=True):
        c = self.cfg
        B = len(self.pos)
        anchors = syn.anchors(c.seed, B, r, c.vocab)
        g = self.gpu.draft(list(range(B)), anchors, logits=True)
        assert g["rc"] == 0
        outs = []
        for b in range(B):
            # the Markov head drafts serially: the oracle follows the GPU's chain of previous
            # tokens, so a near-tie does not make every later row incomparable
            prev = g["tokens"][b] if c.markov_rank else None
            o = self.os.draft(b, int(anchors[b]), prev_tokens=prev)
            compare_block(c, g, o, b, report)
            outs.append(o)
        if check_accept:
            p = c.agree if c.agree is not None else 0.0
            targets = np.stack([syn.target_tokens(c.seed, b, r, outs[b]["tokens"], p, c.vocab) for b in range(B)])
            ga, gn = self.gpu.accept(g["tokens"], targets)
            for b in range(B):
                a_o = accept_checked(outs[b]["tokens"], g["tokens"][b], outs[b]["margin"], targets[b], int(ga[b]),
                                     report)
                if int(ga[b]) == a_o:
                    assert int(gn[b]) == int(targets[b][a_o])
        return g, outs


_MODELS = {}


def cached_model(cfg, norm_jitter=0.0):
    """make_model(cfg) drawn once per process and shared by the test files (the 4-bit 5120-wide
    drafter takes tens of seconds to draw)."""
    key = (cfg, norm_jitter)
    if key not in _MODELS:
        _MODELS[key] = syn.make_model(cfg, norm_jitter=norm_jitter)
    return _MODELS[key]
