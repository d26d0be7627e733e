"""GPU parity of the many-row tcgen05 contraction (dflash_rows_matmul) against the oracle's
fp64 linear map, element by element, and of the draft round when it runs its projections on
that contraction (config large_batch_tc05).

Error model of the contraction. It dequantises each stored weight, the group-64 affine code
w = s q + b, to f16 with one rounding (q made exact, then one fused f16 multiply-add), and
accumulates y = sum_k f16(w_k) (hi_k + lo_k) on the tensor cores in fp32 over a K slice, then sums
the slices in fp32:
  * |f16(w) - w| <= 2^-11 |w| + 2^-25 (round to nearest; the second term covers f16 subnormals);
  * f16 x f16 products are exact in fp32;
  * the accumulation of n = K (2K with the remainder) terms plus the slice sum adds at most
    (n + slices) 2^-22 times sum |f16(w) x| (a crude bound that allows truncating additions).
So |y - y_exact| <= (2^-11 + 1.001 (n + slices) 2^-22) sum_k |w_k| |x_k| + 2^-25 sum_k |x_k|, a
deterministic bound. The tight check is statistical: the rounding errors of the weights are
independent and at most 2^-11 relative (most synthetic weights, |w| < 1/16 on the 2^-15 grid that
bf16 scales and biases give them, are exact in f16), so the rms error stays below 2e-4 of the rms
output for both the N(0, 1) inputs and the inputs on an exact 1/8 (remainder 1/64) grid; an fp32
emulation of the same arithmetic gives about 2.5e-5."""
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


def _weights(hm):
    """The exact stored weights w = s q + b [n][k] (float64) of a q4 HostMatrix."""
    n, k = hm.n_out, hm.n_in
    shifts = (4 * np.arange(8, dtype=np.uint32))[None, None, :]
    q = ((hm.data[:, :, None] >> shifts) & 15).reshape(n, k // 64, 64).astype(np.float64)
    sc = syn.bf16_bits_to_f32(hm.scale).astype(np.float64)[:, :, None]
    bi = syn.bf16_bits_to_f32(hm.bias).astype(np.float64)[:, :, None]
    return (sc * q + bi).reshape(n, k)


def _bound(hm, xh, xl, slices):
    """Deterministic error bound per [row][output] for inputs x = xh + xl."""
    aw = np.abs(_weights(hm))
    ax = np.abs(xh) + np.abs(xl)
    n_terms = xh.shape[1] * (2 if np.any(xl) else 1)
    return (2.0 ** -11 + 1.001 * (n_terms + slices) * 2.0 ** -22) * (ax @ aw.T) + 2.0 ** -25 * ax.sum(axis=1)[:, None]


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
    det = _bound(sub, xh, xl, plan.k_slices)
    assert np.all(err <= det), f"{which}: max err {err.max()} above the deterministic bound"
    rms = np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(ref ** 2))
    assert rms <= 2e-4, f"{which}: relative rms error {rms}"
    return float(err.max()), float(rms)


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
    e1, r1 = _check(s.h, which, mats, 160, lo, exact=False, n_sample=128, seed=5)
    e2, r2 = _check(s.h, which, mats, 160, lo, exact=True, n_sample=128, seed=6)
    print(f"\n{which} lo={lo}: max err normal {e1:.3g} (rms {r1:.2g}), grid {e2:.3g} (rms {r2:.2g})")


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


def test_large_batch_round_ring_wraps_within_a_call():
    """Context calls on the contraction where one request appends more rows than its ring holds
    (window 40, ring of 64 slots, 100 prefill rows in one call): the later rows must overwrite the
    earlier ones in order, so the context K/V goes through the chunked path there; against the
    oracle, error word clear."""
    from test_gpu_parity import run, small
    cfg = small("s_tc05_wrap", batch=8, ctx_len=100, ctx_min=30, window=40, append_min=1, append_max=8, agree=0.6,
                large_batch_tc05=True)
    lengths = syn.ctx_lengths(cfg)
    assert int(lengths.sum()) > 160 and int(lengths.max()) > 64
    run(cfg, rounds=3, ctx_capacity=64, lengths=lengths)


def test_large_batch_round_gelu_all_rows():
    """The same path with the page's gated-GELU FFN and drafts from every block row (the LM head
    epilogue reads every row), 5 requests x gamma 8 = 40 rows, hd 128."""
    from test_gpu_parity import run, small
    cfg = small("s_tc05_g", batch=5, ctx_len=60, ffn="gelu", draft_all_rows=True, gamma=8, head_dim=128,
                n_q_heads=4, n_kv_heads=2, d=512, target_hidden=512, inter=1024, agree=0.5, large_batch_tc05=True)
    run(cfg, rounds=2)
