"""Closed-loop rounds (append a + 1 committed rows, draft from the bonus token, verify, accept)
through the C ABI against an oracle mirror of the same loop. Targets are computed from the
oracle's drafts and given to both sides, so the two loops see the same verification; where a
low-margin row lets the GPU accept a different length (allowed by the parity rule), the GPU loop
is committed with the oracle's result to stay in lockstep and the case is counted."""
import numpy as np
import pytest

import dflash_synth as syn
from dflash_synth import DraftConfig

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import speculative_block_draft_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.build()
    yield


def loop_pair(cfg, rounds, thresholds=None, min_conf=None, prompt=24):
    import oracle
    from parity_util import MARGIN, compare_block
    from speculative_block_draft_gb300.driver import ClosedLoop, SyntheticTarget
    from speculative_block_draft_gb300.session import Session
    B = cfg.batch
    model = syn.make_model(cfg, norm_jitter=0.1)
    sess = Session(model, max_batch=B, ctx_capacity=prompt + rounds * cfg.gamma + 64)
    tgt = SyntheticTarget(cfg)
    loop = ClosedLoop(sess, tgt, thresholds=thresholds, min_conf=min_conf)
    orc = oracle.OracleSession(oracle.Oracle(model))
    anchors0 = syn.anchors(cfg.seed, B, 0, cfg.vocab)
    mirror = {b: {"pos": 0, "pending": prompt, "anchor": int(anchors0[b])} for b in range(B)}
    for b in range(B):
        loop.start(b, prompt, int(anchors0[b]))
    report, forced, total_acc = {}, 0, 0
    for r in range(rounds):
        outs, targets = [], []
        for b in range(B):
            m = mirror[b]
            if m["pending"]:
                rows = tgt.taps(b, m["pos"], m["pending"])
                orc.project(b, syn.taps_to_f32(cfg, rows).astype(np.float64))
                m["pos"] += m["pending"]
                m["pending"] = 0
            o = orc.draft(b, m["anchor"])
            outs.append(o)
        res_probe = None
        # the oracle's drafts decide the verification both loops see
        keep_o = [cfg.n_draft] * B
        targets = np.stack([tgt.verify(r, b, outs[b]["tokens"]) for b in range(B)])
        res = loop.step(targets=targets)
        gpu = {"tokens": res.drafts, "conf": res.conf}
        for b in range(B):
            assert sess.h.ctx_len(b) == mirror[b]["pos"]
            confident = outs[b]["margin"] > MARGIN
            assert np.array_equal(res.drafts[b][confident], outs[b]["tokens"][confident])
            if thresholds is not None or min_conf is not None:
                keep_o[b] = oracle.draft_length(res.conf[b], thresholds, min_conf or 0.0)
                assert res.keep[b] == keep_o[b]
        for b in range(B):
            a_o, nxt_o = oracle.accept_kept(outs[b]["tokens"], targets[b], keep_o[b])
            upto = min(a_o + 1, keep_o[b])
            if np.all(outs[b]["margin"][:upto] > MARGIN):
                assert int(res.accepted[b]) == a_o and int(res.next_anchor[b]) == nxt_o
            elif int(res.accepted[b]) != a_o:
                forced += 1
            res.accepted[b], res.next_anchor[b] = a_o, nxt_o
            res.drafts[b][:a_o] = outs[b]["tokens"][:a_o]
            m = mirror[b]
            m["pending"] += a_o + 1
            m["anchor"] = nxt_o
            total_acc += a_o
        loop.commit(res)
    for b in range(B):
        assert loop.req[b].pos + loop.req[b].pending == mirror[b]["pos"] + mirror[b]["pending"]
        assert loop.req[b].anchor == mirror[b]["anchor"]
    assert sess.check() == 0
    sess.close()
    return total_acc, forced


def cfg(name, **kw):
    base = dict(n_layers=2, d=256, n_q_heads=4, n_kv_heads=2, head_dim=64, inter=512, n_taps=2, target_hidden=256,
                vocab=1000, gamma=6, window=0, ctx_len=24, wdtype="q4", adtype="bf16", seed=77, agree=0.8, batch=3)
    base.update(kw)
    return DraftConfig(name, **base)


def test_closed_loop_matches_oracle():
    acc, forced = loop_pair(cfg("loop_q4"), rounds=6)
    print(f"accepted drafts {acc}, low-margin forced commits {forced}")
    assert acc > 0


def test_closed_loop_windowed_with_pruning():
    c = cfg("loop_win", window=32, gamma=8, agree=0.9, batch=2, wdtype="bf16")
    acc, forced = loop_pair(c, rounds=6, min_conf=0.05)
    print(f"accepted drafts {acc}, low-margin forced commits {forced}")


def test_closed_loop_all_rows():
    acc, forced = loop_pair(cfg("loop_all", draft_all_rows=True, gamma=5), rounds=5)
    print(f"accepted drafts {acc}, low-margin forced commits {forced}")
