"""The allocation-free entry point (dflash_greedy_from_logits_noalloc) against the library's
normal path. It serves callers that cannot allocate device memory on their request path and so
cannot give dflash_create a workspace; its scratch is a fixed array inside the library shared
by every call. This file is collected last on purpose: a first-failure run has already run every
other test, and the test also passes alone in a fresh process."""
import numpy as np
import pytest

import dflash_synth as syn

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkg():
    import speculative_block_draft_gb300 as p
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p.build()
    return p


def test_noalloc_greedy_matches_draft_block_twice(pkg):
    from speculative_block_draft_gb300.session import Session
    cfg = syn.DraftConfig("noalloc", n_layers=2, d=256, n_q_heads=4, n_kv_heads=2, head_dim=64, inter=512, n_taps=2,
                          target_hidden=256, vocab=5000, gamma=5, window=0, ctx_len=40, batch=6, wdtype="q4",
                          adtype="bf16", seed=21)
    s = Session(syn.make_model(cfg, norm_jitter=0.1), max_batch=cfg.batch)
    req = list(range(cfg.batch))
    taps = np.concatenate([syn.taps_rows(cfg, cfg.seed, b, 0, cfg.ctx_len) for b in req])
    assert s.project(req, [cfg.ctx_len] * cfg.batch, taps) == 0
    ref = s.draft(req, syn.anchors(cfg.seed, cfg.batch, 0, cfg.vocab), logits=True)   # the existing entry point
    rows = cfg.batch * cfg.n_draft
    logits = torch.from_numpy(ref["logits"].reshape(rows, cfg.vocab)).cuda()
    for call in range(2):                         # two calls in a row share the scratch array
        tok = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        conf = torch.zeros(rows, dtype=torch.float32, device="cuda")
        assert pkg.greedy_from_logits_noalloc(logits, tok, conf) == 0
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), ref["tokens"].reshape(-1)), call
        # same fp32 logits, different summation order: confidence agrees to fp32 rounding
        dc = np.abs(np.log(conf.cpu().numpy().astype(np.float64)) - np.log(ref["conf"].reshape(-1).astype(np.float64)))
        assert dc.max() <= 1e-5, (call, dc.max())
    too_many = torch.zeros((pkg.DFLASH_NOALLOC_MAX_ROWS + 1, 16), dtype=torch.float32, device="cuda")
    out = torch.zeros(pkg.DFLASH_NOALLOC_MAX_ROWS + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.DFlashError) as e:
        pkg.greedy_from_logits_noalloc(too_many, out)
    assert e.value.status == pkg.DFLASH_ECAPACITY
    s.close()


def _oracle_rows(logits):
    import oracle
    out = [oracle.argmax_conf(row) for row in logits.astype(np.float64)]
    return np.array([o[0] for o in out]), np.array([o[1] for o in out])


@pytest.mark.parametrize("vocab", [2, 17, 63, 64, 65, 5000])
def test_noalloc_small_vocab_ties_and_masked_entries(pkg, vocab):
    """Against the oracle's argmax / confidence: vocabularies below the 64 CTAs of a row (some
    CTAs get no entries), exact ties (the lowest index wins), -inf entries at the start of CTA
    ranges (masked out, no NaN), and a fully masked row (token -1, confidence 0)."""
    rng = np.random.default_rng(vocab)
    rows = 12
    lg = rng.normal(size=(rows, vocab)).astype(np.float32)
    lg[1, :] = 0.5                                                # all equal: token 0, conf 1/V
    top = lg[2].max() + 1.0
    lg[2, [vocab - 1, vocab // 2, min(1, vocab - 1)]] = top      # exact tie at three indices
    starts = sorted({c * vocab // 64 for c in range(64)})
    if len(starts) == vocab:                                      # vocab <= 64: every entry starts a range
        starts = starts[::2]
    lg[3, starts] = -np.inf                                       # masked CTA starts
    lg[4, 0] = -np.inf                                            # masked first entry
    lg[5, :] = -np.inf
    lg[5, vocab - 1] = 2.0                                        # one live entry, the last
    lg[6, :] = -np.inf                                            # nothing live
    d_lg = torch.from_numpy(lg).cuda()
    for call in range(2):
        tok = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
        conf = torch.full((rows,), -1.0, dtype=torch.float32, device="cuda")
        assert pkg.greedy_from_logits_noalloc(d_lg, tok, conf) == 0
        torch.cuda.synchronize()
        t, c = tok.cpu().numpy(), conf.cpu().numpy().astype(np.float64)
        live = [r for r in range(rows) if r != 6]
        ot, oc = _oracle_rows(lg[live])
        assert np.array_equal(t[live], ot), (call, t, ot)
        assert np.all(np.isfinite(c[live]))
        assert np.max(np.abs(np.log(c[live]) - np.log(oc))) <= 1e-5, call
        assert t[6] == -1 and c[6] == 0.0
        assert t[2] == min(1, vocab - 1)
        assert abs(c[1] - 1.0 / vocab) <= 1e-5 / vocab
