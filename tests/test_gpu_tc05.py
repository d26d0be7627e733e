"""GPU parity of the many-row tcgen05 contraction (dflash_rows_matmul) against the oracle's
fp64 linear map, element by element, and of the draft round when it runs its projections on
that contraction (config large_batch_tc05).

Error model of the contraction (it reads each weight as the group-64 affine code
w = s q + b and computes, per group g of 64 inputs, v_g = sum (c + q_k) x_k on the tensor cores
with c = 128 or 64, then y += s v_g + (b - c s) sum x_k in fp32):
  * the products (c + q) x are exact in fp32 (8-bit integers times f16 values);
  * the group sums v_g and sum x_k carry fp32 accumulation error, at most 2^-23 per addition
    relative to the running magnitude (allowing truncating accumulation): over 64 inputs, or
    128 with the f16 remainder, at most 128 * 2^-23 * sum (c + q)|x|;
  * the fold's two fused multiply-adds and the ordered sum of the K slices add at most
    2^-23 relative to the running sum per step, over K/64 groups.
So |y - y_exact| <= (2^-16 + (K/64 + 2) 2^-22) * sum_g (|s| sum q|x| + (256|s| + |b|) sum |x|),
a deterministic bound that is loose because the offsets c make the intermediate terms large.
Two checks are tight: (1) with inputs on a 1/8 (remainder 1/64) grid every group sum is exact
in fp32, so only the fold's roundings remain (bounded by 2^-22 times the running magnitudes,
computed here from the exact group terms); (2) with N(0, 1) inputs the rms error stays below
1e-4 of the rms output (random rounding grows like sqrt(K) * 2^-24 times the terms)."""
import numpy as np
import pytest

import dflash_synth as syn
from dflash_synth import CONFIGS, DraftConfig

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _built():
    import speculative_block_draft_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.build()
    yield


def _mats(model, layer=0):
    """(DFLASH_MAT_*, natural-order list of the HostMatrix blocks it stacks)."""
    import speculative_block_draft_gb300 as pkg
    m = model.mats
    return {
        "ctx": (pkg.DFLASH_MAT_CTX, [m["W_c"]]),
        "qkv": (pkg.DFLASH_MAT_QKV, [m[f"bb.{layer}.q"], m[f"bb.{layer}.k"], m[f"bb.{layer}.v"]]),
        "o": (pkg.DFLASH_MAT_O, [m[f"bb.{layer}.o"]]),
        "gateup": (pkg.DFLASH_MAT_GATEUP, [m[f"bb.{layer}.gate"], m[f"bb.{layer}.up"]]),
        "down": (pkg.DFLASH_MAT_DOWN, [m[f"bb.{layer}.down"]]),
        "lm": (pkg.DFLASH_MAT_LM, [m["lm_head"]]),
    }


def _rows_of(blocks, sel):
    """The stacked matrix's natural rows `sel` as one q4 HostMatrix (sampled outputs)."""
    starts = np.cumsum([0] + [b.n_out for b in blocks])
    data, scale, bias = [], [], []
    for n in sel:
        j = int(np.searchsorted(starts, n, side="right") - 1)
        b, r = blocks[j], int(n - starts[j])
        data.append(b.data[r]), scale.append(b.scale[r]), bias.append(b.bias[r])
    k = blocks[0].n_in
    return syn.HostMatrix("q4", len(sel), k, np.ascontiguousarray(data), np.ascontiguousarray(scale),
                          np.ascontiguousarray(bias))


def _codes(hm):
    """q [n][G][64] float64, s, b [n][G] float64 of a q4 HostMatrix."""
    n, k = hm.n_out, hm.n_in
    shifts = (4 * np.arange(8, dtype=np.uint32))[None, None, :]
    q = ((hm.data[:, :, None] >> shifts) & 15).reshape(n, k // 64, 64).astype(np.float64)
    s = syn.bf16_bits_to_f32(hm.scale).astype(np.float64)
    b = syn.bf16_bits_to_f32(hm.bias).astype(np.float64)
    return q, s, b


def _bounds(hm, xh, xl, gps):
    """(deterministic bound, fold-only bound) per [row][output] for inputs x = xh + xl."""
    q, s, b = _codes(hm)
    G = q.shape[1]
    x = (xh + xl).reshape(xh.shape[0], G, 64)
    ax = (np.abs(xh) + np.abs(xl)).reshape(xh.shape[0], G, 64)
    X = ax.sum(axis=2)                                            # [r][G]
    P = np.matmul(ax.transpose(1, 0, 2), q.transpose(1, 2, 0)).transpose(1, 2, 0)   # sum q |x|, [r][n][G]
    inner = np.abs(s)[None] * P + (256 * np.abs(s) + np.abs(b))[None] * X[:, None, :]
    det = (2.0 ** -16 + (G + 2) * 2.0 ** -22) * inner.sum(axis=2)
    # fold only (exact group sums): running sums within each K slice, from the exact terms
    v = np.matmul(x.transpose(1, 0, 2), (q + 128.0).transpose(1, 2, 0)).transpose(1, 2, 0)
    xs = x.sum(axis=2)
    t_s = np.abs(s)[None] * np.abs(v)
    t_b = (np.abs(b) + 128 * np.abs(s))[None] * np.abs(xs)[:, None, :]
    contrib = s[None] * (v - 128.0 * xs[:, None, :]) + b[None] * xs[:, None, :]
    fold = np.zeros(det.shape)
    for g0 in range(0, G, gps):
        run = np.cumsum(contrib[:, :, g0:g0 + gps], axis=2)
        fold += (np.abs(run) + t_s[:, :, g0:g0 + gps] + t_b[:, :, g0:g0 + gps]).sum(axis=2)
    return det, 4 * U * (fold + np.abs(contrib).sum(axis=2))


def _check(h, which, blocks_map, rows, lo, exact, n_sample=None, seed=0):
    import oracle
    import speculative_block_draft_gb300 as pkg
    mat, blocks = blocks_map[which]
    n_out, k = sum(b.n_out for b in blocks), blocks[0].n_in
    rng = np.random.default_rng(seed + rows * 7 + lo)
    if exact:
        xh = rng.integers(-8, 9, size=(rows, k)) / 8.0
        xl = rng.integers(-8, 9, size=(rows, k)) / 64.0 if lo else np.zeros((rows, k))
    else:
        xf = rng.normal(size=(rows, k)).astype(np.float32)
        xh = xf.astype(np.float16).astype(np.float64)
        xl = (xf - xh).astype(np.float16).astype(np.float64) if lo else np.zeros((rows, k))
    x16 = torch.from_numpy(xh.astype(np.float16).view(np.int16)).cuda()
    xl16 = torch.from_numpy(xl.astype(np.float16).view(np.int16)).cuda() if lo else None
    plan = pkg.rows_matmul_plan(n_out, k, rows, lo, torch.cuda.get_device_properties(0).multi_processor_count)
    scratch = torch.empty(plan.scratch_bytes + 256, dtype=torch.uint8, device="cuda")
    scratch = scratch[(256 - scratch.data_ptr() % 256) % 256:]
    y = torch.full((rows, n_out), float("nan"), dtype=torch.float32, device="cuda")
    assert h.rows_matmul(mat, 0, x16, y, scratch, x_lo=xl16) == 0
    torch.cuda.synchronize()
    assert h.check_errors() == 0
    sel = np.arange(n_out) if n_sample is None else np.unique(
        np.concatenate([rng.choice(n_out, n_sample, replace=False), [0, n_out - 1]]))
    sub = _rows_of(blocks, sel)
    ref = oracle.linear(sub, xh + xl)                             # [rows][sel]
    got = y.cpu().numpy().astype(np.float64)[:, sel]
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    det, fold = _bounds(sub, xh, xl, plan.groups_per_slice)
    assert np.all(err <= det), f"{which}: max err {err.max()} above the deterministic bound"
    if exact:
        assert np.all(err <= fold), f"{which}: max err {err.max()}, fold bound {fold[err > fold].min()}"
    else:
        rms = np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(ref ** 2))
        assert rms <= 1e-4, f"{which}: relative rms error {rms}"
    return float(err.max())


SMALL = DraftConfig("tc05_small", n_layers=1, d=256, n_q_heads=4, n_kv_heads=2, head_dim=64, inter=1024, n_taps=4,
                    target_hidden=256, vocab=1000, gamma=5, window=0, ctx_len=16, wdtype="q4", adtype="bf16", seed=31)
TINY = DraftConfig("tc05_tiny", n_layers=1, d=64, n_q_heads=1, n_kv_heads=1, head_dim=64, inter=64, n_taps=10,
                   target_hidden=64, vocab=200, gamma=4, window=0, ctx_len=16, wdtype="q4", adtype="bf16", seed=32)


@pytest.fixture(scope="module")
def small_sessions():
    from speculative_block_draft_gb300.session import Session
    out = {}
    for cfg in (TINY, SMALL):
        m = syn.make_model(cfg)
        out[cfg.name] = (Session(m), _mats(m))
    yield out
    for s, _ in out.values():
        s.close()


@pytest.mark.parametrize("rows", [1, 16, 17, 100, 160])
@pytest.mark.parametrize("lo", [0, 1])
@pytest.mark.parametrize("exact", [True, False], ids=["grid", "normal"])
def test_rows_matmul_small_shapes(small_sessions, rows, lo, exact):
    """Every matrix of two small drafters: one 64-input group (TINY: 64x64, 192x64, 128x64),
    ten groups (TINY W_c 64x640), a ragged last 128-row tile and strip (vocab 200 and 1000),
    K split in slices (SMALL W_c 256x1024, down 256x1024), at 1-160 rows, with and without
    the remainder."""
    for name in ("tc05_tiny", "tc05_small"):
        s, mats = small_sessions[name]
        for which in mats:
            _check(s.h, which, mats, rows, lo, exact)


@pytest.mark.parametrize("which,lo", [("ctx", 0), ("qkv", 1), ("o", 0), ("gateup", 1), ("down", 0), ("lm", 0), ("lm", 1)])
def test_rows_matmul_full_shapes_160_rows(which, lo):
    """The 4-bit 5120-wide drafter's matrices at 160 rows (the batched workload's block rows),
    128 sampled outputs each (plus the first and last), N(0, 1) inputs and exact-grid inputs."""
    from parity_util import cached_model
    from speculative_block_draft_gb300.session import Session
    m = cached_model(CONFIGS["c3"], norm_jitter=0.1)
    s = _full_session(m)
    mats = _mats(m)
    e1 = _check(s.h, which, mats, 160, lo, exact=False, n_sample=128, seed=5)
    e2 = _check(s.h, which, mats, 160, lo, exact=True, n_sample=128, seed=6)
    print(f"\n{which} lo={lo}: max err normal {e1:.3g}, grid {e2:.3g}")


_FULL = {}


def _full_session(m):
    from speculative_block_draft_gb300.session import Session
    if "s" not in _FULL:
        _FULL["s"] = Session(m, max_batch=1, ctx_capacity=CONFIGS["c3"].window)
    return _FULL["s"]


def test_large_batch_round_small_ragged():
    """A draft round on the contraction: 8 requests x gamma 5 = 40 block rows (> 32, so every
    projection and the LM head run once over all rows), ragged prefills of 249 context rows in
    one call (W_c over 160-row chunks, crossing a chunk boundary), then U{1..8} appends; against
    the oracle at the benchmark spec's tolerances, error word clear."""
    from test_gpu_parity import run, small
    cfg = small("s_tc05", batch=8, ctx_len=50, ctx_min=12, window=40, append_min=1, append_max=8, agree=0.6,
                large_batch_tc05=True)
    assert int(syn.ctx_lengths(cfg).sum()) > 160
    run(cfg, rounds=3, ctx_capacity=64)


def test_large_batch_round_gelu_all_rows():
    """The same path with the page's gated-GELU FFN and drafts from every block row (the LM head
    epilogue reads every row), 5 requests x gamma 8 = 40 rows, hd 128."""
    from test_gpu_parity import run, small
    cfg = small("s_tc05_g", batch=5, ctx_len=60, ffn="gelu", draft_all_rows=True, gamma=8, head_dim=128,
                n_q_heads=4, n_kv_heads=2, d=512, target_hidden=512, inter=1024, agree=0.5, large_batch_tc05=True)
    run(cfg, rounds=2)
