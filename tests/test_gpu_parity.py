"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Small configurations span several tiles, ragged tails, ring wrap-around, padding strips, split-K
and row chunking; the full-size workloads (page-3 default bf16, the page-1 4-bit drafter, the
block/head sweep and the batched case) run in the launch configuration the bench times.
"""
import numpy as np
import pytest

import dflash_synth as syn
from dflash_synth import CONFIGS, DraftConfig

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import speculative_block_draft_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.build()
    yield


def small(name, **kw):
    base = dict(n_layers=2, d=256, n_q_heads=4, n_kv_heads=2, head_dim=64, inter=512, n_taps=2, target_hidden=256,
                vocab=1000, gamma=5, window=0, ctx_len=70, wdtype="q4", adtype="bf16", seed=99)
    base.update(kw)
    return DraftConfig(name, **base)


def run(cfg, rounds=3, jitter=0.1, max_batch=None, ctx_capacity=None, lengths=None, model=None, oracle_ctx=None,
        appends=None):
    from parity_util import Pair
    model = model or syn.make_model(cfg, norm_jitter=jitter)
    pair = Pair(cfg, model, max_batch=max_batch, ctx_capacity=ctx_capacity, oracle_ctx=oracle_ctx)
    lengths = syn.ctx_lengths(cfg) if lengths is None else lengths
    pair.prefill(lengths)
    report = {}
    for r in range(rounds):
        if r:
            counts = appends(r) if appends else syn.append_counts(cfg, r)
            pair.append(counts)
        pair.round(r, report)
    assert pair.gpu.check() == 0
    pair.gpu.close()
    print(f"\n[{cfg.name}] {report}")
    return report


# ---------------------------------------------------------------------------------------------
# small cases: every code path, several tiles, ragged tails
# ---------------------------------------------------------------------------------------------
def test_c1_tiny_fp32():
    rep = run(CONFIGS["c1"], rounds=3)
    assert rep["max_logit_err"] < 1e-4


@pytest.mark.parametrize("wdtype", ["q4", "bf16"])
@pytest.mark.parametrize("hd", [64, 128, 256])
def test_small_formats_and_head_dims(wdtype, hd):
    cfg = small(f"s_{wdtype}_{hd}", wdtype=wdtype, head_dim=hd, n_q_heads=512 // hd, n_kv_heads=max(1, 256 // hd),
                d=512, target_hidden=512, inter=1024)
    run(cfg, rounds=2)


@pytest.mark.parametrize("wdtype", ["q4", "bf16", "f32"])
def test_small_gated_gelu_ffn(wdtype):
    """The page's gated-GELU FFN (tanh-form GELU on the gate) instead of SwiGLU."""
    kw = dict(adtype="f32") if wdtype == "f32" else {}
    run(small(f"s_gelu_{wdtype}", wdtype=wdtype, ffn="gelu", d=512, target_hidden=512, inter=1024,
              n_q_heads=8, n_kv_heads=2, **kw), rounds=2)


def test_small_draft_all_rows():
    """Drafts from all gamma block rows (gamma tokens per block), the page-3 forwardRows form."""
    run(small("s_allrows", draft_all_rows=True, gamma=6, agree=0.5), rounds=2)


@pytest.mark.parametrize("wdtype", ["q4", "bf16", "f32"])
def test_small_markov_head(wdtype):
    """Markov sequential head (rank 128): serial drafts, each argmax over base logits plus
    W1[previous token] W2; the oracle follows the GPU's chain of previous tokens."""
    kw = dict(adtype="f32") if wdtype == "f32" else {}
    run(small(f"s_markov_{wdtype}", wdtype=wdtype, markov_rank=128, gamma=6, **kw), rounds=2)


def test_small_markov_head_batched_all_rows():
    """Markov head over several requests (one chain each) with drafts from every block row."""
    run(small("s_markov_b", markov_rank=64, batch=3, ctx_len=50, draft_all_rows=True, agree=0.5), rounds=2)


def test_small_mha_no_gqa():
    """Multi-head attention without grouping (one K/V head per query head)."""
    run(small("s_mha", n_q_heads=8, n_kv_heads=8, head_dim=64, d=512, target_hidden=512, inter=1024), rounds=2)


def test_small_d_ne_h_bf16():
    """tok_proj / out_proj present (d != H)."""
    run(small("s_proj", wdtype="bf16", target_hidden=512), rounds=2)


@pytest.mark.parametrize("gamma", [2, 4, 8, 16])
def test_small_block_sizes(gamma):
    run(small(f"s_g{gamma}", gamma=gamma, n_q_heads=4, n_kv_heads=4 if gamma == 16 else 2), rounds=2)


def test_sliding_window_ring_wraps():
    """window 100 in a ring of 128 rows; 12 rounds of 7 new rows wrap the ring several times."""
    cfg = small("s_ring", window=100, ctx_len=90)
    run(cfg, rounds=12, ctx_capacity=100, appends=lambda r: np.array([7]))


def test_empty_context():
    cfg = small("s_p0", ctx_len=0)
    run(cfg, rounds=2, lengths=np.array([0]), appends=lambda r: np.array([0]))


def test_batch_ragged_and_row_chunks():
    """8 requests x gamma 5 = 40 block rows (> 32: row chunks), ragged contexts, U{1..8} appends."""
    cfg = small("s_batch", batch=8, ctx_len=300, ctx_min=1, window=128, append_min=1, append_max=8, agree=0.6)
    run(cfg, rounds=3, ctx_capacity=160)


@pytest.mark.parametrize("case", ["hd64", "hd128_gelu", "allrows_b3", "b4_g8_32rows", "g16", "markov", "d_ne_h"])
def test_small_skinny_tc05(case):
    """Draft calls of at most 32 block rows on the tcgen05 projection kernel (config skinny_tc05):
    several 128-row tiles cut between CTAs (ragged last tiles: vocab 1000, d 256 / 512), 16 and 32
    contraction rows, drafting-row maps of one to four requests, the gated-GELU FFN, the Markov
    head's base logits, and d != H (the head then stays on the GEMV)."""
    kw = {"hd64": dict(),
          "hd128_gelu": dict(ffn="gelu", d=512, target_hidden=512, inter=1024, n_q_heads=4, n_kv_heads=2,
                             head_dim=128),
          "allrows_b3": dict(draft_all_rows=True, batch=3, ctx_len=50, agree=0.5),
          "b4_g8_32rows": dict(batch=4, gamma=8, ctx_len=60, ctx_min=5, window=48, agree=0.6),
          "g16": dict(gamma=16, n_kv_heads=4),
          "markov": dict(markov_rank=128, gamma=6),
          "d_ne_h": dict(target_hidden=512)}[case]
    run(small(f"s_pj_{case}", skinny_tc05=True, **kw), rounds=2, ctx_capacity=64 if case == "b4_g8_32rows" else None)


def test_deterministic_repeat():
    """Same inputs, two handles: bit-identical logits, tokens and confidence."""
    from speculative_block_draft_gb300.session import Session
    cfg = small("s_det")
    m = syn.make_model(cfg, norm_jitter=0.1)
    outs = []
    for _ in range(2):
        s = Session(m)
        s.project([0], [70], syn.taps_rows(cfg, cfg.seed, 0, 0, 70))
        outs.append(s.draft([0], np.array([3], dtype=np.int32)))
        s.close()
    for k in ("tokens", "conf", "logits"):
        assert np.array_equal(outs[0][k], outs[1][k])


def test_accept_kernel_exhaustive_vs_oracle():
    import oracle
    from speculative_block_draft_gb300.session import Session
    cfg = small("s_acc", gamma=8)
    s = Session(syn.make_model(cfg), max_batch=1)
    rng = np.random.default_rng(0)
    d = rng.integers(0, 3, size=(4096, 7)).astype(np.int32)
    t = rng.integers(0, 3, size=(4096, 8)).astype(np.int32)
    a, nxt = s.accept(d, t)
    want = np.zeros(8, dtype=np.int64)
    for i in range(4096):
        assert (a[i], nxt[i]) == oracle.accept(d[i], t[i])
        want[oracle.accept(d[i], t[i])[0]] += 1
    # the device histogram of accepted lengths counts every block once, at its length
    assert s.h.accept_histogram(stream=s.stream) == list(want)
    s.accept(d[:100], t[:100])
    want += np.bincount(a[:100], minlength=8)
    assert s.h.accept_histogram(stream=s.stream) == list(want)
    s.close()


def test_draft_lengths_and_kept_accept_vs_oracle():
    """Confidence-scheduled pruning and capped acceptance, bit-exact (integer results; the same
    fp32 confidences and thresholds go to both sides), gamma 8 and 16, per-position thresholds
    and the uniform minConf, with exact ties."""
    import oracle
    from speculative_block_draft_gb300.session import Session
    rng = np.random.default_rng(11)
    for gamma in (8, 16):
        cfg = small(f"s_prune{gamma}", gamma=gamma)
        s = Session(syn.make_model(cfg), max_batch=1)
        n, B = gamma - 1, 2048
        conf = rng.random((B, n)).astype(np.float32)
        th = (rng.random(n) * 0.5).astype(np.float32)
        conf[:64, 1] = th[1]                          # ties keep the position
        for thresholds, min_conf in ((th, 0.0), (None, 0.3), (None, 0.0), (None, 1.5)):
            keep = s.draft_lengths(conf, thresholds, min_conf)
            for i in range(B):
                assert keep[i] == oracle.draft_length(conf[i], thresholds, min_conf)
        keep = s.draft_lengths(conf, th)
        d = rng.integers(0, 3, size=(B, n)).astype(np.int32)
        t = rng.integers(0, 3, size=(B, n + 1)).astype(np.int32)
        a, nxt = s.accept_kept(d, keep, t)
        for i in range(B):
            assert (a[i], nxt[i]) == oracle.accept_kept(d[i], t[i], keep[i])
        s.close()


def test_pruning_on_drafted_confidence():
    """The pruning step on a real round: confidences from dflash_draft_block decide the kept
    lengths exactly as the oracle decides them from the same fp32 values."""
    import oracle
    from speculative_block_draft_gb300.session import Session
    cfg = small("s_prune_round", gamma=8, ctx_len=40, batch=4)
    s = Session(syn.make_model(cfg, norm_jitter=0.1), max_batch=4)
    for b in range(4):
        assert s.project([b], [40], syn.taps_rows(cfg, cfg.seed, b, 0, 40)) == 0
    out = s.draft([0, 1, 2, 3], syn.anchors(cfg.seed, 4, 0, cfg.vocab), logits=False)
    conf = out["conf"]
    mid = float(np.median(conf[:, 1:]))
    keep = s.draft_lengths(conf, None, mid)
    for i in range(4):
        assert keep[i] == oracle.draft_length(conf[i], None, mid)
    s.close()


def test_abi_errors_and_decline(monkeypatch):
    import speculative_block_draft_gb300 as pkg
    from speculative_block_draft_gb300.session import Session
    cfg = small("s_err", ctx_len=10)
    s = Session(syn.make_model(cfg), max_batch=2, ctx_capacity=64)
    h = s.h
    taps = syn.taps_rows(cfg, cfg.seed, 0, 0, 10)
    assert s.project([0], [10], taps) == 0
    # temperature > 0 and the kill switch decline without touching the outputs
    anchor = torch.zeros(1, dtype=torch.int32, device="cuda")
    draft = torch.full((1, cfg.gamma - 1), -7, dtype=torch.int32, device="cuda")
    assert h.draft_block([0], anchor, draft, temperature=0.4) == pkg.DFLASH_DECLINED
    monkeypatch.setenv("DFLASH_DISABLE", "1")
    assert h.draft_block([0], anchor, draft) == pkg.DFLASH_DECLINED
    monkeypatch.delenv("DFLASH_DISABLE")
    torch.cuda.synchronize()
    assert int(draft.min()) == -7 and h.stats()["declined"] == 2
    # rejected calls change no state
    with pytest.raises(pkg.DFlashError) as e:
        h.project_ctx([0, 0], [1, 1], torch.zeros(2, 512, dtype=torch.int16, device="cuda"))
    assert e.value.status == pkg.DFLASH_EINVAL
    with pytest.raises(pkg.DFlashError) as e:
        h.project_ctx([5], [1], torch.zeros(1, 512, dtype=torch.int16, device="cuda"))
    assert e.value.status == pkg.DFLASH_EINVAL
    with pytest.raises(pkg.DFlashError) as e:   # window 0: capacity 64 rows per request
        h.project_ctx([0], [60], torch.zeros(60, 512, dtype=torch.int16, device="cuda"))
    assert e.value.status == pkg.DFLASH_ECAPACITY
    assert h.ctx_len(0) == 10
    assert h.draft_block([], anchor, draft) == 0
    assert h.reset_request(1) == 0 and h.ctx_len(1) == 0
    assert s.check() == 0
    s.close()


def test_bounded_wait_runs_out_reports_and_recovers():
    """A device wait that runs out is reported, never a hang, and the next round is exact again
    (the "A Refusal Is Not A Failure" page's closing rule: an acceleration path declines, never
    fails). With the wait limit shortened to 20 ms, CTA 0 of every projection launch of one draft
    call waits on an mbarrier that nothing completes. The down projection here (K = 4096 over
    16 strips) splits K four ways over global partials and tickets, so the stalled CTA leaves a
    strip's ticket short of its count: the following round is only right if dflash_check_errors
    cleared the tickets."""
    import time

    import speculative_block_draft_gb300 as pkg
    from parity_util import Pair
    cfg = small("s_stall", inter=4096, ctx_len=40)
    pair = Pair(cfg, syn.make_model(cfg, norm_jitter=0.1), ctx_capacity=64)
    pair.prefill(syn.ctx_lengths(cfg))
    report = {}
    pair.round(0, report)
    s = pair.gpu
    s.h.set_wait_limit(20000, stream=s.stream)
    s.h.debug_stall(0)
    t0 = time.time()
    g = s.draft([0], syn.anchors(cfg.seed, 1, 1, cfg.vocab), logits=False)
    assert g["rc"] == 0
    with pytest.raises(pkg.DFlashError) as e:
        s.check()
    assert e.value.status == pkg.DFLASH_ETIMEOUT
    assert time.time() - t0 < 30.0
    assert s.check() == 0                       # the word was cleared
    s.h.set_wait_limit(0, stream=s.stream)
    pair.round(1, report)                       # the hook was one-shot; tickets were cleared
    pair.round(2, report)
    assert s.check() == 0
    print(f"\n[s_stall] {report}, stalled call {time.time() - t0:.2f} s")
    s.close()


# ---------------------------------------------------------------------------------------------
# full-size workloads
# ---------------------------------------------------------------------------------------------
def test_c2_p3_default_bf16_full():
    rep = run(CONFIGS["c2"], rounds=2, jitter=0.1)
    print("c2", rep)


_C3_MODEL = {}


def c3_model():
    """The 4-bit 5120-wide drafter shared by the full-size cases, with every norm weight drawn
    N(1, 0.1) so that the 5120-wide strip and cluster-split epilogues are checked against
    distinct attn_norm, ff_norm, ctx_norm and out_norm values."""
    from parity_util import cached_model
    return cached_model(CONFIGS["c3"], norm_jitter=0.1)


@pytest.mark.parametrize("skinny", [False, True], ids=["gemv", "tc05"])
def test_c3_dflash2_q4_full(skinny):
    """The bench workload: 4-bit 5120-wide drafter, block 8, window 2048 over context 4096; on the
    mma.sync GEMV and on the tcgen05 projection kernel (config skinny_tc05)."""
    cfg = syn.with_overrides(CONFIGS["c3"], skinny_tc05=skinny)
    m = c3_model()
    rep = run(cfg, rounds=2, model=syn.HostModel(cfg, m.mats, dict(m.vecs)))
    print("c3", skinny, rep)


def _c4_oracle_ctx(cfg, model):
    """Window rows of the sweep's context (positions 6144..8191): the K/V rows do not depend on
    gamma or on how head_dim splits the 1024 K/V features, so all sweep points share them."""
    import oracle
    key = ("c4ctx", cfg.window)
    if key not in _C3_MODEL:
        P = cfg.ctx_len
        first = P - cfg.window if cfg.window else 0
        taps = syn.taps_to_f32(cfg, syn.taps_rows(cfg, cfg.seed, 0, first, P - first)).astype(np.float64)
        k, v = oracle.Oracle(model).ctx_rows(taps)
        _C3_MODEL[key] = (first, k, v)
    return {0: _C3_MODEL[key]}


@pytest.mark.parametrize("cfg", syn.configs.C4[:6], ids=lambda c: c.name)
def test_c4_sweep_full(cfg):
    m = c3_model()
    model = syn.HostModel(cfg, m.mats, dict(m.vecs))
    model.vecs["block_pos"] = syn.normal(cfg.seed, "block_pos", (32, cfg.d), 0.02)[: cfg.gamma].copy()
    model.vecs["mask_emb"] = syn.normal(cfg.seed, "mask_emb", (32, cfg.d), 0.02)[: cfg.gamma - 1].copy()
    rep = run(cfg, rounds=1, model=model, oracle_ctx=_c4_oracle_ctx(cfg, m))
    print(cfg.name, rep)


@pytest.mark.slow
def test_c4_full_context_window0():
    cfg = syn.configs.C4[6]
    m = c3_model()
    model = syn.HostModel(cfg, m.mats, dict(m.vecs))
    rep = run(cfg, rounds=1, model=model, oracle_ctx=_c4_oracle_ctx(cfg, m),
              ctx_capacity=cfg.ctx_len + 64)
    print(cfg.name, rep)


@pytest.mark.parametrize("tc05", [False, True], ids=["gemv", "tc05"])
def test_c5_batched_sampled_requests(tc05):
    """32 requests, gamma 5, ragged contexts in [512, 16384], U{1..8} appends, agreement 0.6.
    The GPU runs all 32; the oracle recomputes requests 0 and 17 (requests are independent).
    tc05: the 160 block rows run every projection and the head once on the tcgen05 contraction,
    and context appends over 32 rows run W_c on it too."""
    from parity_util import MARGIN, Pair, accept_checked, compare_block
    import oracle
    cfg = syn.with_overrides(CONFIGS["c5"], large_batch_tc05=tc05)
    m = c3_model()
    model = syn.HostModel(cfg, m.mats, dict(m.vecs))
    model.vecs["block_pos"] = syn.normal(cfg.seed, "block_pos", (32, cfg.d), 0.02)[: cfg.gamma].copy()
    model.vecs["mask_emb"] = syn.normal(cfg.seed, "mask_emb", (32, cfg.d), 0.02)[: cfg.gamma - 1].copy()
    from speculative_block_draft_gb300.session import Session
    s = Session(model, max_batch=cfg.batch, ctx_capacity=cfg.window + 64)
    lengths = syn.ctx_lengths(cfg)
    B = cfg.batch
    # the window is all that matters: rows before P - W never enter attention
    first = [max(0, int(P) - cfg.window) for P in lengths]
    rows = [syn.taps_rows(cfg, cfg.seed, b, first[b], int(lengths[b]) - first[b]) for b in range(B)]
    # the GPU walks through the skipped prefix too (positions decide ring slots and the window);
    # those rows never enter attention, so zero taps stand in for them
    zeros = torch.zeros((4096, cfg.n_taps * cfg.target_hidden), dtype=torch.int16, device="cuda")
    for b in range(B):
        done = 0
        while done < first[b]:
            n = min(4096, first[b] - done)
            with torch.cuda.stream(s.stream):
                assert s.h.project_ctx([b], [n], zeros, stream=s.stream) == 0
            done += n
    s.stream.synchronize()
    assert s.project(list(range(B)), [r.shape[0] for r in rows], np.concatenate(rows)) == 0
    counts = syn.append_counts(cfg, 1)
    app = [syn.taps_rows(cfg, cfg.seed, b, int(lengths[b]), int(counts[b])) for b in range(B)]
    assert s.project(list(range(B)), [int(c) for c in counts], np.concatenate(app)) == 0
    anchors = syn.anchors(cfg.seed, B, 1, cfg.vocab)
    g = s.draft(list(range(B)), anchors, logits=True)
    orc = oracle.Oracle(model)
    rep = {}
    for b in (0, 17):
        taps = np.concatenate([rows[b], app[b]])
        k, v = orc.ctx_rows(syn.taps_to_f32(cfg, taps).astype(np.float64))
        if k.shape[1] > cfg.window:
            k, v = k[:, -cfg.window:], v[:, -cfg.window:]
        o = orc.draft(int(anchors[b]), np.ascontiguousarray(k), np.ascontiguousarray(v))
        compare_block(cfg, g, o, b, rep)
        t = syn.target_tokens(cfg.seed, b, 1, o["tokens"], cfg.agree, cfg.vocab)
        ga, _ = s.accept(g["tokens"][b:b + 1], t[None, :])
        accept_checked(o["tokens"], g["tokens"][b], o["margin"], t, int(ga[0]), rep)
    assert s.check() == 0
    s.close()
    print("c5", rep)
