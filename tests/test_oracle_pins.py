"""Pins of the CPU oracle to facts that do not come from the oracle itself: closed forms,
library routines (torch SDPA / SiLU), brute force, invariants and the page-1 worked examples.
Each test names the mistake it would catch."""
import itertools
import os

import numpy as np
import pytest
import torch

import dflash_synth as syn
import oracle
from dflash_synth import DraftConfig, HostMatrix

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(wdtype="f32", d=64, H=64, gamma=4, window=0, hq=4, hkv=2, L=2, vocab=97):
    return DraftConfig("tiny", n_layers=L, d=d, n_q_heads=hq, n_kv_heads=hkv, head_dim=d // hq,
                       inter=128, n_taps=2, target_hidden=H, vocab=vocab, gamma=gamma, window=window,
                       ctx_len=5, wdtype=wdtype, adtype="f32", seed=7)


def model(cfg, jitter=0.3):
    return syn.make_model(cfg, cfg.seed, norm_jitter=jitter)


def taps(cfg, n, pos0=0, req=0):
    return syn.taps_to_f32(cfg, syn.taps_rows(cfg, cfg.seed, req, pos0, n)).astype(np.float64)


# ------------------------------------------------------------------------------------------
# storage formats
# ------------------------------------------------------------------------------------------
def test_q4_hand_cases():
    """Nibble order (low nibble = lowest input), group indexing and w = s*q + b.
    Catches a reversed nibble order, a wrong group index, or scale/bias swapped."""
    words = np.zeros((2, 128 // 8), dtype=np.uint32)
    words[0, 0] = 0x76543210          # q = 0..7 for k = 0..7
    words[0, 1] = 0xFEDCBA98          # q = 8..15 for k = 8..15
    words[1, 8] = 0x0000000F          # row 1, group 1, k = 64 -> q = 15
    scale = np.array([[0x3F00, 0x4000], [0x3F80, 0x3E80]], dtype=np.uint16)  # 0.5, 2.0 | 1.0, 0.25
    bias = np.array([[0xBF80, 0x0000], [0x0000, 0x4040]], dtype=np.uint16)   # -1, 0 | 0, 3.0
    m = HostMatrix("q4", 2, 128, words, scale, bias)
    for k in range(16):
        assert oracle.weight(m, 0, k) == 0.5 * k - 1.0
    assert oracle.weight(m, 0, 16) == -1.0           # q = 0 in group 0
    assert oracle.weight(m, 0, 64) == 0.0            # group 1: s = 2, b = 0, q = 0
    assert oracle.weight(m, 1, 64) == 0.25 * 15 + 3.0
    assert oracle.weight(m, 1, 65) == 3.0
    bf = HostMatrix("bf16", 1, 3, np.array([[0x3F80, 0x4049, 0xC000]], dtype=np.uint16))
    assert [oracle.weight(bf, 0, k) for k in range(3)] == [1.0, 3.140625, -2.0]


def test_q4_matches_source_within_half_step():
    """The oracle reads back what the group-64 quantiser wrote: every dequantised weight lies
    within half a quantisation step (plus bf16 rounding of s, b) of the fp32 draw."""
    w = syn.normal(3, "qtest", (8, 256), 0.02)
    hm = HostMatrix("q4", 8, 256, *syn.quantize_q4g64(w))
    deq = oracle.dense(hm)
    s = syn.bf16_bits_to_f32(hm.scale).astype(np.float64)
    step = np.repeat(s, 64, axis=1)
    err = np.abs(deq - w)
    assert np.all(err <= 0.5 * step * 1.02 + 4e-3 * np.abs(w) + 1e-7)
    assert np.mean(err) < 0.3 * np.mean(step)


# ------------------------------------------------------------------------------------------
# RMSNorm, SiLU, attention, argmax/confidence
# ------------------------------------------------------------------------------------------
def test_rmsnorm_closed_form():
    y = oracle.rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 2.0], dtype=np.float32), 0.0)
    r = np.sqrt(12.5)
    assert np.allclose(y, [3 / r, 8 / r], rtol=0, atol=1e-15)
    x = np.random.default_rng(0).normal(size=64)
    ones = np.ones(64, dtype=np.float32)
    y1 = oracle.rmsnorm(x, ones, 0.0)
    assert abs(np.sqrt(np.mean(y1 ** 2)) - 1.0) < 1e-14           # unit RMS
    assert np.allclose(oracle.rmsnorm(7.5 * x, ones, 0.0), y1, atol=1e-14)   # scale invariance
    assert np.allclose(oracle.rmsnorm(np.zeros(4), ones[:4], 1e-6), 0.0)     # eps guards 0/0


def test_silu_vs_torch():
    xs = np.linspace(-30, 30, 121)
    ref = torch.nn.functional.silu(torch.tensor(xs, dtype=torch.float64)).numpy()
    got = np.array([oracle.silu(x) for x in xs])
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-300)


@pytest.mark.parametrize("hq,hkv,hd,nq,nk", [(4, 4, 16, 3, 7), (4, 2, 16, 4, 9), (6, 2, 8, 5, 1), (8, 1, 32, 8, 40)])
def test_attention_vs_torch_sdpa(hq, hkv, hd, nq, nk):
    """Non-causal SDPA with contiguous GQA groups against torch's own routine (fp64).
    Catches a wrong scale, a transposed score, or a wrong head-group map."""
    rng = np.random.default_rng(hq * 100 + nk)
    q = rng.normal(size=(nq, hq * hd))
    k = rng.normal(size=(nk, hkv * hd))
    v = rng.normal(size=(nk, hkv * hd))
    got = oracle.attention(q, k, v, hq, hkv, hd)
    tq = torch.tensor(q).view(nq, hq, hd).transpose(0, 1)
    tk = torch.tensor(k).view(nk, hkv, hd).transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
    tv = torch.tensor(v).view(nk, hkv, hd).transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=False)
    ref = ref.transpose(0, 1).reshape(nq, hq * hd).numpy()
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_attention_causal_variant_vs_masked_sdpa():
    """The test-only causal variant: query i sees the context keys and block keys 0..i."""
    rng = np.random.default_rng(5)
    hq, hkv, hd, nctx, g = 4, 2, 8, 3, 4
    q = rng.normal(size=(g, hq * hd))
    k = rng.normal(size=(nctx + g, hkv * hd))
    v = rng.normal(size=(nctx + g, hkv * hd))
    got = oracle.attention(q, k, v, hq, hkv, hd, causal_block_start=nctx)
    mask = torch.tensor([[j <= nctx + i for j in range(nctx + g)] for i in range(g)])
    tq = torch.tensor(q).view(g, hq, hd).transpose(0, 1)
    tk = torch.tensor(k).view(-1, hkv, hd).transpose(0, 1).repeat_interleave(2, dim=0)
    tv = torch.tensor(v).view(-1, hkv, hd).transpose(0, 1).repeat_interleave(2, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    assert np.allclose(got, ref.transpose(0, 1).reshape(g, -1).numpy(), atol=1e-12)


def test_attention_rows_sum_to_one():
    """With V = identity over keys the output is the probability row itself."""
    rng = np.random.default_rng(1)
    nk, hd = 12, 16
    q = rng.normal(size=(6, hd)) * 3
    k = rng.normal(size=(nk, hd))
    v = np.zeros((nk, hd))
    v[np.arange(nk), np.arange(nk)] = 1.0
    p = oracle.attention(q, k, v, 1, 1, hd)[:, :nk]
    assert np.all(p >= 0)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-12


def test_argmax_conf_closed_forms():
    V = 1000
    tok, conf, margin = oracle.argmax_conf(np.full(V, 0.25))
    assert (tok, margin) == (0, 0.0) and abs(conf - 1.0 / V) < 1e-15     # all equal: 1/V, index 0
    for c in (0.5, 3.0, 20.0):
        row = np.zeros(V)
        row[417] = c
        tok, conf, margin = oracle.argmax_conf(row)
        assert tok == 417 and margin == c
        # the sum over V terms rounds about once per term: a few V ulps
        assert abs(conf - 1.0 / (1.0 + (V - 1) * np.exp(-c))) < 4 * V * 2.3e-16
    row = np.zeros(V)
    row[[5, 9]] = 2.0                                                   # tie: lowest index wins
    assert oracle.argmax_conf(row)[0] == 5


# ------------------------------------------------------------------------------------------
# acceptance
# ------------------------------------------------------------------------------------------
def test_accept_exhaustive_binary():
    """Every d in {0,1}^n, t in {0,1}^(n+1), n <= 7, against the direct definition
    a = max{k : d[:k] == t[:k]}."""
    for n in range(0, 8):
        for d in itertools.product((0, 1), repeat=n):
            for t in itertools.product((0, 1), repeat=n + 1):
                a_ref = max(k for k in range(n + 1) if list(d[:k]) == list(t[:k]))
                a, nxt = oracle.accept(np.array(d, dtype=np.int32), np.array(t, dtype=np.int32))
                assert (a, nxt) == (a_ref, t[a_ref])


def test_accept_page1_worked_examples():
    """block 8 = 1 verify token + 7 proposals; accepted 7 -> committed 8, accepted 5 -> 6."""
    rows = [list(map(int, ln.split())) for ln in open(os.path.join(GOLDEN, "accept_worked_examples.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert rows == [[8, 7, 8], [8, 5, 6]]
    rng = np.random.default_rng(0)
    for block, accepted, committed in rows:
        n = block - 1
        d = rng.integers(0, 1000, size=n).astype(np.int32)
        t = np.concatenate([d, rng.integers(1000, 2000, size=1)]).astype(np.int32)
        if accepted < n:
            t[accepted] = d[accepted] + 1
        a, nxt = oracle.accept(d, t)
        assert a == accepted and a + 1 == committed and nxt == t[accepted]
    cfg = tiny(gamma=8)
    o = oracle.Oracle(model(cfg))
    out = o.draft(3, *o.ctx_rows(taps(cfg, 2)))
    assert out["tokens"].shape == (7,)          # a block of 8 drafts 7 tokens


def test_synthetic_target_agreement_statistics():
    """E[a] = sum_{k=1..n} p^k when each position agrees independently with probability p."""
    rng = np.random.default_rng(11)
    for p, n, expect in ((0.7, 7, 2.1412), (0.7, 4, 1.7731), (0.6, 4, 1.3056)):
        assert abs(sum(p ** k for k in range(1, n + 1)) - expect) < 1e-3
        acc = []
        for trial in range(12000):
            d = rng.integers(0, 50, size=n).astype(np.int32)
            t = syn.target_tokens(99, 0, trial, d, p, 50)
            acc.append(oracle.accept(d, t)[0])
        acc = np.array(acc, dtype=np.float64)
        assert abs(acc.mean() - expect) < 3 * acc.std() / np.sqrt(len(acc)) + 1e-3


# ------------------------------------------------------------------------------------------
# drafter structure
# ------------------------------------------------------------------------------------------
def _raw(hm):
    assert hm.fmt == "f32"
    return hm.data.astype(np.float64)


def _rms(x, w, eps):
    return x / np.sqrt(np.mean(x * x) + eps) * w


def test_ctx_projection_one_hot_taps():
    """One-hot taps select one column of W_c; then ctx_norm, then the layer's attn_norm (the
    same norm the block rows use), then W_k / W_v. Catches a transposed W_c, a dropped or
    swapped norm, or K/V swapped."""
    cfg = tiny()
    m = model(cfg)
    o = oracle.Oracle(m)
    j = 37
    t = np.zeros((1, cfg.n_taps * cfg.target_hidden))
    t[0, j] = 1.0
    k, v = o.ctx_rows(t)
    x = _raw(m.mats["W_c"])[:, j]
    hctx = _rms(x, m.vecs["ctx_norm"], cfg.eps)
    for i in range(cfg.n_layers):
        n = _rms(hctx, m.vecs[f"bb.{i}.attn_norm"], cfg.eps)
        assert np.allclose(k[i, 0], _raw(m.mats[f"bb.{i}.k"]) @ n, atol=1e-13)
        assert np.allclose(v[i, 0], _raw(m.mats[f"bb.{i}.v"]) @ n, atol=1e-13)


@pytest.mark.parametrize("H", [64, 128])
def test_identity_layers_reduce_to_head_of_block_rows(H):
    """With W_o = W_down = 0 every layer is the identity on H_d, so draft k's logits are
    lm_head (out_proj) RMSNorm(mask_emb[k-1] + block_pos[k]; out_norm): pins the block rows,
    the draft-row selection (rows 1..gamma-1), out_norm/out_proj and the head orientation."""
    cfg = tiny(H=H)
    m = model(cfg)
    for i in range(cfg.n_layers):
        m.mats[f"bb.{i}.o"].data[:] = 0
        m.mats[f"bb.{i}.down"].data[:] = 0
    o = oracle.Oracle(m)
    anchor = 11
    out = o.draft(anchor, *o.ctx_rows(taps(cfg, 3)), trace=True)
    e = _raw(m.mats["embed"])[anchor]
    row0 = (_raw(m.mats["tok_proj"]) @ e if H != cfg.d else e) + m.vecs["block_pos"][0]
    assert np.allclose(out["trace"][-1][0], row0, atol=1e-14)
    for k in range(1, cfg.gamma):
        h = _rms(m.vecs["mask_emb"][k - 1].astype(np.float64) + m.vecs["block_pos"][k], m.vecs["out_norm"], cfg.eps)
        if H != cfg.d:
            h = _raw(m.mats["out_proj"]) @ h
        ref = _raw(m.mats["lm_head"]) @ h
        assert np.allclose(out["logits"][k - 1], ref, atol=1e-13)
        assert out["tokens"][k - 1] == int(np.argmax(ref))


@pytest.mark.parametrize("window,n_ctx", [(0, 5), (3, 5), (8, 5), (0, 0), (2, 1)])
def test_uniform_attention_pins_key_set(window, n_ctx):
    """W_q = 0 makes every score 0, so attention returns the plain mean of the value rows over
    the key set. With W_o = I and W_down = 0 the layer adds exactly that mean: pins the key set
    (windowed context rows ++ all gamma block rows), the GQA head map and the residual add."""
    cfg = tiny(window=window, L=1, hq=4, hkv=2)
    m = model(cfg)
    m.mats["bb.0.q"].data[:] = 0
    m.mats["bb.0.o"].data[:] = np.eye(cfg.d, dtype=np.float32)
    m.mats["bb.0.down"].data[:] = 0
    o = oracle.Oracle(m)
    kc, vc = o.ctx_rows(taps(cfg, n_ctx))
    out = o.draft(5, kc, vc, trace=True)
    h0 = out["trace"][0]
    lo = max(0, n_ctx - window) if window else 0
    nd = np.stack([_rms(h0[r], m.vecs["bb.0.attn_norm"], cfg.eps) for r in range(cfg.gamma)])
    vd = nd @ _raw(m.mats["bb.0.v"]).T
    vals = np.concatenate([vc[0, lo:n_ctx], vd])                       # [keys][Hkv*hd]
    hd, grp = cfg.head_dim, cfg.n_q_heads // cfg.n_kv_heads
    mean = vals.mean(axis=0)
    add = np.concatenate([mean[(h // grp) * hd:(h // grp + 1) * hd] for h in range(cfg.n_q_heads)])
    assert np.allclose(out["trace"][1], h0 + add[None, :], atol=1e-13)


@pytest.mark.parametrize("hq,hkv,window,n_ctx", [(4, 4, 0, 5), (4, 4, 3, 6), (4, 2, 4, 7), (4, 1, 0, 0), (2, 2, 0, 3)])
def test_block_scores_from_live_q_k_v_projections(hq, hkv, window, n_ctx):
    """Eq 3 of the dflash.ts page with every attention projection live: Q = n W_q^T,
    K = [K_ctx; n W_k^T], V = [V_ctx; n W_v^T], n = RMSNorm(H_d; attn_norm). W_q and W_k are
    scaled up so the softmax is far from uniform (the scores decide the output); W_o = I and
    W_down = 0 make the layer add exactly the attention output. The restatement below builds
    the projections from the raw matrices and calls torch's scaled_dot_product_attention.
    Catches K_d built from W_v or W_q, Q built from W_k, a transposed projection, block keys
    missing from the key set, or a wrong context slice."""
    cfg = tiny(window=window, L=1, hq=hq, hkv=hkv)
    m = model(cfg)
    m.mats["bb.0.q"].data[:] *= 25.0
    m.mats["bb.0.k"].data[:] *= 25.0
    m.mats["bb.0.o"].data[:] = np.eye(cfg.d, dtype=np.float32)
    m.mats["bb.0.down"].data[:] = 0
    o = oracle.Oracle(m)
    kc, vc = o.ctx_rows(taps(cfg, n_ctx))
    out = o.draft(5, kc, vc, trace=True)
    h0 = out["trace"][0]
    n = np.stack([_rms(h0[r], m.vecs["bb.0.attn_norm"], cfg.eps) for r in range(cfg.gamma)])
    lo = max(0, n_ctx - window) if window else 0
    q = n @ _raw(m.mats["bb.0.q"]).T
    k = np.concatenate([kc[0, lo:n_ctx], n @ _raw(m.mats["bb.0.k"]).T])
    v = np.concatenate([vc[0, lo:n_ctx], n @ _raw(m.mats["bb.0.v"]).T])
    hd, G, nk = cfg.head_dim, cfg.gamma, k.shape[0]
    tq = torch.tensor(q).view(G, hq, hd).transpose(0, 1)
    tk = torch.tensor(k).view(nk, hkv, hd).transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
    tv = torch.tensor(v).view(nk, hkv, hd).transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
    att = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=False)
    att = att.transpose(0, 1).reshape(G, hq * hd).numpy()
    p = torch.softmax(tq @ tk.transpose(1, 2) / np.sqrt(hd), dim=-1)
    assert float(p.max()) > 0.5 or nk == 1          # the scores are far from uniform
    assert np.allclose(out["trace"][1], h0 + att, rtol=0, atol=1e-12)


def _torch_drafter(cfg, m, anchor, tap_rows, all_rows=False, gelu=False):
    """The whole draft block written with torch's own routines (F.linear, F.rms_norm, SDPA,
    SiLU / GELU, softmax) in float64 from the raw matrices: the context rows' projection and
    norms (Eq 2 of the dflash.ts page), the block rows, every layer of Eq 3 with its gated FFN,
    out_norm (+ out_proj) and the borrowed head."""
    F = torch.nn.functional
    T = lambda a: torch.tensor(np.asarray(a, dtype=np.float64))
    W = lambda n: T(_raw(m.mats[n]))
    vec = lambda n: T(m.vecs[n])
    eps, d, hd = cfg.eps, cfg.d, cfg.head_dim
    hq, hkv, G = cfg.n_q_heads, cfg.n_kv_heads, cfg.gamma
    hctx = F.rms_norm(F.linear(T(tap_rows), W("W_c")), (d,), vec("ctx_norm"), eps)
    e = W("embed")[anchor]
    h = torch.empty(G, d, dtype=torch.float64)
    h[0] = (F.linear(e, W("tok_proj")) if cfg.target_hidden != d else e) + vec("block_pos")[0]
    for k in range(1, G):
        h[k] = vec("mask_emb")[k - 1] + vec("block_pos")[k]
    n_ctx = hctx.shape[0]
    lo = max(0, n_ctx - cfg.window) if cfg.window else 0
    for i in range(cfg.n_layers):
        an = vec(f"bb.{i}.attn_norm")
        nc = F.rms_norm(hctx[lo:], (d,), an, eps)
        n = F.rms_norm(h, (d,), an, eps)
        q = F.linear(n, W(f"bb.{i}.q"))
        k = torch.cat([F.linear(nc, W(f"bb.{i}.k")), F.linear(n, W(f"bb.{i}.k"))])
        v = torch.cat([F.linear(nc, W(f"bb.{i}.v")), F.linear(n, W(f"bb.{i}.v"))])
        tq = q.view(G, hq, hd).transpose(0, 1)
        tk = k.view(-1, hkv, hd).transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
        tv = v.view(-1, hkv, hd).transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
        att = F.scaled_dot_product_attention(tq, tk, tv, is_causal=False).transpose(0, 1).reshape(G, hq * hd)
        h = h + F.linear(att, W(f"bb.{i}.o"))
        n2 = F.rms_norm(h, (d,), vec(f"bb.{i}.ff_norm"), eps)
        g = F.linear(n2, W(f"bb.{i}.gate"))
        act = F.gelu(g, approximate="tanh") if gelu else F.silu(g)
        h = h + F.linear(act * F.linear(n2, W(f"bb.{i}.up")), W(f"bb.{i}.down"))
    rows = h if all_rows else h[1:]
    hn = F.rms_norm(rows, (d,), vec("out_norm"), eps)
    if cfg.target_hidden != d:
        hn = F.linear(hn, W("out_proj"))
    logits = F.linear(hn, W("lm_head"))
    p = torch.softmax(logits, dim=-1)
    return logits.numpy(), p.argmax(dim=-1).numpy(), p.max(dim=-1).values.numpy()


@pytest.mark.parametrize("H,hq,hkv,window,n_ctx,ffn,all_rows", [
    (64, 4, 2, 0, 6, "swiglu", False),
    (128, 4, 2, 3, 7, "swiglu", False),
    (64, 4, 4, 0, 0, "gelu", False),
    (96, 4, 1, 4, 9, "swiglu", True),
    (64, 2, 2, 2, 5, "gelu", True),
])
def test_full_drafter_vs_torch_restatement(H, hq, hkv, window, n_ctx, ffn, all_rows):
    """Every weight live at once (jittered norms, two layers, context rows, windowed keys,
    d == H and d != H, both FFN gates, GQA and MHA, drafts from rows 1..gamma-1 or from all
    rows): the oracle's logits, tokens and confidences equal the torch restatement above.
    The other pins fix one piece each with the rest switched off; this one catches a mistake
    in how the pieces are chained (a norm weight of the wrong layer, the residual taken from
    the wrong stream, context keys normed with the wrong vector, the head fed unnormed rows)."""
    cfg = syn.with_overrides(tiny(H=H, hq=hq, hkv=hkv, window=window, gamma=5), ffn=ffn,
                             draft_all_rows=all_rows)
    m = model(cfg)
    for i in range(cfg.n_layers):
        m.mats[f"bb.{i}.q"].data[:] *= 6.0        # scores far from uniform
        m.mats[f"bb.{i}.k"].data[:] *= 6.0
    o = oracle.Oracle(m)
    t = taps(cfg, n_ctx)
    out = o.draft(13, *o.ctx_rows(t))
    logits, tok, conf = _torch_drafter(cfg, m, 13, t.reshape(n_ctx, cfg.n_taps * H), all_rows, ffn == "gelu")
    assert out["logits"].shape == logits.shape == (cfg.gamma if all_rows else cfg.gamma - 1, cfg.vocab)
    scale = float(np.abs(logits).max())
    assert scale > 1e-3
    assert np.allclose(out["logits"], logits, rtol=0, atol=1e-12 * max(1.0, scale))
    assert np.array_equal(out["tokens"], tok)
    assert np.allclose(out["conf"], conf, rtol=1e-11, atol=0)


def test_non_causal_block():
    """is_causal is false: block row 1 (draft 1) depends on block row gamma-1, which only
    mask_emb[gamma-2] feeds. A causal variant of the same oracle shows no such dependence."""
    cfg = tiny(gamma=5)
    m = model(cfg)
    kc, vc = oracle.Oracle(m).ctx_rows(taps(cfg, 4))
    base = oracle.Oracle(m).draft(9, kc, vc)["logits"]
    base_c = oracle.Oracle(m, causal=True).draft(9, kc, vc)["logits"]
    m.vecs["mask_emb"][cfg.gamma - 2] += 0.5
    pert = oracle.Oracle(m).draft(9, kc, vc)["logits"]
    pert_c = oracle.Oracle(m, causal=True).draft(9, kc, vc)["logits"]
    assert np.max(np.abs(pert[0] - base[0])) > 1e-6
    assert np.max(np.abs(pert_c[0] - base_c[0])) == 0.0
    assert np.max(np.abs(base_c[0] - base[0])) > 1e-6


def test_window_equivalences():
    """W >= P equals W = 0; rows outside the window never matter; rows inside do."""
    cfg0 = tiny(window=0)
    m = model(cfg0)
    kc, vc = oracle.Oracle(m).ctx_rows(taps(cfg0, 9))
    full = oracle.Oracle(m).draft(2, kc, vc)["logits"]
    m.cfg = syn.with_overrides(cfg0, window=9)
    assert np.array_equal(oracle.Oracle(m).draft(2, kc, vc)["logits"], full)
    m.cfg = syn.with_overrides(cfg0, window=4)
    o = oracle.Oracle(m)
    base = o.draft(2, kc, vc)["logits"]
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, :5] += 1.0
    vc2[:, :5] -= 1.0
    assert np.array_equal(o.draft(2, kc2, vc2)["logits"], base)
    kc2[:, 6] += 1.0
    assert np.max(np.abs(o.draft(2, kc2, vc2)["logits"] - base)) > 1e-9


def test_gqa_equals_mha_with_duplicated_kv_heads():
    """GQA with Hkv < Hq equals MHA whose K/V heads are the GQA heads repeated per group."""
    cg = tiny(hq=4, hkv=2)
    mg = model(cg)
    cm = syn.with_overrides(cg, n_kv_heads=4)
    mm = syn.HostModel(cm, dict(mg.mats), mg.vecs)
    hd = cg.head_dim
    for i in range(cg.n_layers):
        for w in ("k", "v"):
            src = mg.mats[f"bb.{i}.{w}"].data.reshape(2, hd, cg.d)
            dup = np.repeat(src, 2, axis=0).reshape(4 * hd, cg.d)
            mm.mats[f"bb.{i}.{w}"] = HostMatrix("f32", 4 * hd, cg.d, np.ascontiguousarray(dup))
    t = taps(cg, 6)
    og, om = oracle.Oracle(mg), oracle.Oracle(mm)
    lg = og.draft(4, *og.ctx_rows(t))["logits"]
    lm = om.draft(4, *om.ctx_rows(t))["logits"]
    assert np.allclose(lg, lm, rtol=0, atol=1e-13)


def test_ctx_rows_chunked_equal_whole():
    """Context rows are independent: projecting in chunks gives the same rows bit for bit."""
    cfg = tiny()
    o = oracle.Oracle(model(cfg))
    t = taps(cfg, 6)
    k, v = o.ctx_rows(t)
    parts = [o.ctx_rows(t[a:b]) for a, b in ((0, 1), (1, 3), (3, 6))]
    assert np.array_equal(np.concatenate([p[0] for p in parts], axis=1), k)
    assert np.array_equal(np.concatenate([p[1] for p in parts], axis=1), v)


def test_swiglu_ffn_vs_torch():
    """With W_o = 0 a layer adds W_down (SiLU(W_gate n) * W_up n), n = RMSNorm(H_d; ff_norm):
    pins gate vs up (SiLU on the gate only) against torch's SiLU."""
    cfg = tiny(L=1)
    m = model(cfg)
    m.mats["bb.0.o"].data[:] = 0
    o = oracle.Oracle(m)
    out = o.draft(1, *o.ctx_rows(taps(cfg, 2)), trace=True)
    h0 = torch.tensor(out["trace"][0])
    n = torch.tensor(np.stack([_rms(out["trace"][0][r], m.vecs["bb.0.ff_norm"], cfg.eps) for r in range(cfg.gamma)]))
    g = n @ torch.tensor(_raw(m.mats["bb.0.gate"])).T
    u = n @ torch.tensor(_raw(m.mats["bb.0.up"])).T
    ref = h0 + (torch.nn.functional.silu(g) * u) @ torch.tensor(_raw(m.mats["bb.0.down"])).T
    assert np.allclose(out["trace"][1], ref.numpy(), atol=1e-13)


def test_gelu_tanh_vs_torch():
    """The gated-GELU gate: GELU in its tanh approximation, against torch's
    gelu(approximate="tanh")."""
    x = np.linspace(-8, 8, 4001)
    ref = torch.nn.functional.gelu(torch.tensor(x, dtype=torch.float64), approximate="tanh").numpy()
    assert np.allclose(oracle.gelu_tanh(x), ref, rtol=0, atol=1e-14)


def test_gated_gelu_ffn_vs_torch():
    """The page's gated-GELU FFN: with W_o = 0 a layer adds W_down (gelu(W_gate n) * W_up n),
    n = RMSNorm(H_d; ff_norm), the gate through GELU's tanh form (torch's), the up path linear."""
    cfg = syn.with_overrides(tiny(L=1), ffn="gelu")
    m = model(cfg)
    m.mats["bb.0.o"].data[:] = 0
    o = oracle.Oracle(m)
    out = o.draft(1, *o.ctx_rows(taps(cfg, 2)), trace=True)
    h0 = torch.tensor(out["trace"][0])
    n = torch.tensor(np.stack([_rms(out["trace"][0][r], m.vecs["bb.0.ff_norm"], cfg.eps) for r in range(cfg.gamma)]))
    g = n @ torch.tensor(_raw(m.mats["bb.0.gate"])).T
    u = n @ torch.tensor(_raw(m.mats["bb.0.up"])).T
    ref = h0 + (torch.nn.functional.gelu(g, approximate="tanh") * u) @ torch.tensor(_raw(m.mats["bb.0.down"])).T
    assert np.allclose(out["trace"][1], ref.numpy(), atol=1e-13)
    silu = oracle.Oracle(syn.HostModel(syn.with_overrides(cfg, ffn="swiglu"), m.mats, m.vecs))
    assert not np.allclose(silu.draft(1, *silu.ctx_rows(taps(cfg, 2)))["logits"], out["logits"], atol=1e-9)


@pytest.mark.parametrize("wdtype", ["bf16", "q4"])
def test_stored_formats_equal_their_dense_f32_copy(wdtype):
    """A drafter stored as bf16 / 4-bit gives the same logits as the f32 drafter holding the
    dequantised values: the format only changes what the weights are, never the arithmetic."""
    cq = tiny(wdtype=wdtype)
    mq = model(cq)
    cf = syn.with_overrides(cq, wdtype="f32")
    mf = syn.HostModel(cf, {n: HostMatrix("f32", h.n_out, h.n_in, oracle.dense(h).astype(np.float32))
                            for n, h in mq.mats.items()}, mq.vecs)
    t = taps(cq, 5)
    oq, of = oracle.Oracle(mq), oracle.Oracle(mf)
    assert np.allclose(oq.draft(8, *oq.ctx_rows(t))["logits"], of.draft(8, *of.ctx_rows(t))["logits"],
                       rtol=0, atol=1e-12)


def test_session_window_trim_matches_full_history():
    """The multi-round helper that keeps only the last W rows gives the same block as the
    oracle run over the whole history."""
    cfg = tiny(window=4)
    m = model(cfg)
    o = oracle.Oracle(m)
    s = oracle.OracleSession(o)
    t = taps(cfg, 11)
    for a, b in ((0, 3), (3, 7), (7, 11)):
        s.project(0, t[a:b])
    kc, vc = o.ctx_rows(t)
    assert np.array_equal(s.draft(0, 6)["logits"], o.draft(6, kc, vc)["logits"])


# ------------------------------------------------------------------------------------------
# confidence-scheduled draft-length pruning (dflash.ts page: draft options, forwardRows loop)
# ------------------------------------------------------------------------------------------
def test_draft_length_page_rules():
    """Hand cases of the page's rule: position 0 is always drafted; the first later position
    whose confidence is below its threshold ends the block; a per-position list takes
    precedence over the uniform minConf; the comparison is strict."""
    L = oracle.draft_length
    assert L([0.0, 0.9, 0.9, 0.9], min_conf=0.5) == 4          # position 0 kept even at 0
    assert L([0.9, 0.9, 0.2, 0.9], min_conf=0.5) == 2          # truncated at the first low one
    assert L([0.9, 0.1, 0.9, 0.9], min_conf=0.5) == 1
    assert L([0.9, 0.5, 0.5, 0.5], min_conf=0.5) == 4          # equal is kept (strict <)
    assert L([0.9, 0.6, 0.3, 0.3], thresholds=[0.99, 0.7, 0.1, 0.1], min_conf=0.0) == 1
    assert L([0.9, 0.6, 0.3, 0.3], thresholds=[0.99, 0.5, 0.2, 0.4], min_conf=0.95) == 3
    assert L([0.9, 0.01, 0.0, 0.0], min_conf=0.0) == 4         # minConf 0 keeps everything
    assert L([0.9], min_conf=0.99) == 1                        # a one-draft block


def test_draft_length_invariants():
    """1 <= keep <= n; raising one threshold never lengthens the block; lowering every
    threshold to 0 keeps all n; keep is the first drop position of the brute-force scan."""
    rng = np.random.default_rng(5)
    for _ in range(2000):
        n = int(rng.integers(1, 16))
        conf = rng.random(n).astype(np.float32)
        th = rng.random(n).astype(np.float32) * 0.6
        k = oracle.draft_length(conf, th)
        assert 1 <= k <= n
        drops = [j for j in range(1, n) if conf[j] < th[j]]
        assert k == (drops[0] if drops else n)
        j = int(rng.integers(0, n))
        th2 = th.copy()
        th2[j] = min(1.0, th2[j] + 0.3)
        assert oracle.draft_length(conf, th2) <= k
        assert oracle.draft_length(conf, np.zeros(n, np.float32)) == n


def test_accept_kept_is_capped_acceptance():
    """Verifying only the first keep drafts: accepted = min(unpruned accepted, keep), and the
    bonus token is the target's token right after the accepted prefix (exhaustive, n <= 5)."""
    for n in range(1, 6):
        for d in itertools.product((0, 1), repeat=n):
            for t in itertools.product((0, 1), repeat=n + 1):
                a_full, _ = oracle.accept(np.array(d, dtype=np.int32), np.array(t, dtype=np.int32))
                for keep in range(1, n + 1):
                    a, nxt = oracle.accept_kept(np.array(d, dtype=np.int32), np.array(t, dtype=np.int32), keep)
                    assert a == min(a_full, keep) and nxt == t[a]


def test_draft_all_rows_adds_row0_draft():
    """Drafting from every block row (the page-3 forwardRows): the drafts of rows 1..gamma-1 are
    exactly the default mode's, and the extra first draft is the borrowed head applied to the
    output-normed final block row 0 (restated here with a dense head)."""
    cfg = tiny(gamma=5)
    m = model(cfg)
    o1 = oracle.Oracle(m)
    o2 = oracle.Oracle(syn.HostModel(syn.with_overrides(cfg, draft_all_rows=True), m.mats, m.vecs))
    k, v = o1.ctx_rows(taps(cfg, 3))
    a = o1.draft(4, k, v)
    b = o2.draft(4, k, v, trace=True)
    assert b["logits"].shape == (cfg.gamma, cfg.vocab) and a["logits"].shape == (cfg.gamma - 1, cfg.vocab)
    assert np.array_equal(b["logits"][1:], a["logits"]) and np.array_equal(b["tokens"][1:], a["tokens"])
    h0 = _rms(b["trace"][cfg.n_layers][0], m.vecs["out_norm"], cfg.eps)
    ref = oracle.dense(m.mats["lm_head"]) @ h0
    assert np.allclose(b["logits"][0], ref, rtol=0, atol=1e-12)
    assert b["tokens"][0] == int(np.argmax(ref))


# ------------------------------------------------------------------------------------------
# Markov sequential head (dflash.ts page, Eq 5: the markov branch of the drafting loop)
# ------------------------------------------------------------------------------------------
def _markov_cfg(**kw):
    return syn.with_overrides(tiny(gamma=5, vocab=97), markov_rank=64, **kw)


def test_markov_zero_w2_is_the_parallel_drafter():
    """W2 = 0 (the page's initialisation) leaves the drafts of the parallel head unchanged."""
    cfg = _markov_cfg()
    m = model(cfg)
    m.mats["markov.w2t"].data[:] = 0
    o = oracle.Oracle(m)
    k, v = o.ctx_rows(taps(cfg, 3))
    out = o.draft(5, k, v)
    assert np.array_equal(out["logits"], out["base_logits"])
    base = oracle.Oracle(syn.HostModel(syn.with_overrides(cfg, markov_rank=0), m.mats, m.vecs)).draft(5, k, v)
    assert np.array_equal(out["tokens"], base["tokens"])


def test_markov_bias_chain_and_linearity():
    """Row k's bias depends only on prev_k (the anchor for row 0, draft k-1 after): changing the
    anchor moves row 0 only, changing the token fed after row j moves row j+1 only; and the bias
    is linear in W2 (doubling W2 doubles logits - base)."""
    cfg = _markov_cfg()
    m = model(cfg)
    o = oracle.Oracle(m)
    rng = np.random.default_rng(3)
    n, V = cfg.n_draft, cfg.vocab
    base = rng.normal(size=(n, V))
    prev = np.array([11, 23, 37, 41], dtype=np.int32)
    a = o.markov(7, base, prev)["logits"]
    b = o.markov(8, base, prev)["logits"]
    assert not np.allclose(a[0], b[0]) and np.array_equal(a[1:], b[1:])
    for j in range(n - 1):
        p2 = prev.copy()
        p2[j] = (p2[j] + 5) % V
        c = o.markov(7, base, p2)["logits"]
        changed = [not np.array_equal(a[r], c[r]) for r in range(n)]
        assert changed == [r == j + 1 for r in range(n)]
    m2 = syn.HostModel(cfg, dict(m.mats), m.vecs)
    w2 = m.mats["markov.w2t"]
    m2.mats["markov.w2t"] = HostMatrix("f32", w2.n_out, w2.n_in, (w2.data * 2).astype(np.float32))
    d = oracle.Oracle(m2).markov(7, base, prev)["logits"]
    assert np.allclose(d - base, 2 * (a - base), rtol=0, atol=1e-12)
    own = o.markov(7, base)                         # its own greedy chain
    assert np.array_equal(o.markov(7, base, own["tokens"])["logits"], own["logits"])
    assert own["tokens"][0] == int(np.argmax(own["logits"][0]))
