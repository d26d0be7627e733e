"""Host-side checks of the many-row tcgen05 contraction (dflash_rows_matmul): its launch plan's
invariants over the drafter's matrix shapes, and argument validation before any launch. No GPU."""
import ctypes

import pytest

import speculative_block_draft_gb300 as pkg

SMEM_MAX = 232448          # dynamic shared memory a CTA may opt into on sm_103a (227 KB)
TMEM_COLS = 512            # tensor-memory columns per SM

# (n_out, k_in) of the 5120-wide drafter's stored matrices: W_c, QKV, O, gate/up, down, LM head;
# plus a one-strip matrix, a matrix whose last 128-row tile is ragged, and one 64-input group
SHAPES = [(5120, 25600), (7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408), (151936, 5120),
          (16, 64), (200, 640), (48, 64)]


@pytest.fixture(scope="module")
def lib():
    pkg.build()
    return pkg.lib()


@pytest.mark.parametrize("n_out,k_in", SHAPES)
@pytest.mark.parametrize("rows", [1, 15, 16, 17, 100, 128, 160])
@pytest.mark.parametrize("x_lo", [0, 1])
def test_plan_invariants(lib, n_out, k_in, rows, x_lo):
    p = pkg.rows_matmul_plan(n_out, k_in, rows, x_lo, 152)
    groups = k_in // 64
    assert p.n_pad % 16 == 0 and rows <= p.n_pad < rows + 16            # the MMA's N
    assert 1 <= p.tiles_small <= p.tiles_big <= 3
    assert p.tiles_big * p.n_pad <= TMEM_COLS                            # one fp32 accumulator per tile
    assert p.m_tiles == -(-n_out // 128)
    # the tile groups cover every 128-row tile once: big groups first, the last group may be short
    assert 1 <= p.big_groups <= p.tile_groups and (p.big_groups - 1) * p.tiles_big < p.m_tiles
    covered = p.big_groups * p.tiles_big + (p.tile_groups - p.big_groups) * p.tiles_small
    last = p.tiles_big if p.tile_groups == p.big_groups else p.tiles_small
    assert covered - last < p.m_tiles <= covered
    assert p.tiles_big == 1 or p.tiles_big <= p.m_tiles
    assert p.grid == p.tile_groups * p.k_slices                            # CTAs: tile groups x K slices
    # the K slices cover every group once, none empty, each at least 4 groups where K allows
    assert (p.k_slices - 1) * p.groups_per_slice < groups <= p.k_slices * p.groups_per_slice
    assert p.groups_per_slice >= min(4, groups)
    # a K split never leaves CTAs for a second partial wave
    assert p.k_slices == 1 or p.grid <= 152
    assert 2 <= p.x_stages <= 4 and 1 <= p.w_stages <= 8 and 2 <= p.a_stages <= 6 and p.smem_bytes <= SMEM_MAX
    assert p.w_groups in (1, 2) and p.x_groups in (1, 2)
    # activation stage: x_groups tiles of n_pad rows x 128 B (twice with the remainder), each a
    # multiple of 1024 B
    stage = p.x_groups * p.n_pad * 128 * (2 if x_lo else 1)
    assert (p.n_pad * 128) % 1024 == 0
    # + the f16 A stages (one group) and the raw stages (w_groups groups), sized for the largest CTA
    assert p.smem_bytes >= (p.x_stages * stage + p.a_stages * p.tiles_big * 128 * 128 +
                            p.w_stages * p.w_groups * p.tiles_big * 4608)
    # scratch: one fp32 partial tile per (K slice, 128-row tile), then 8 chunks x 32 rows' norm scales
    assert p.scratch_bytes == p.k_slices * p.n_pad * p.m_tiles * 128 * 4 + 8 * 32 * 4


def test_plan_shapes_of_the_drafter(lib):
    """The cost model's choices on the 5120-wide drafter (152 SMs): no second partial wave."""
    lm = pkg.rows_matmul_plan(151936, 5120, 128, 0, 152)        # 1187 tiles in 594 CTAs of 2 (three f16 stages each)
    assert (lm.m_tiles, lm.k_slices, lm.tiles_big, lm.grid, lm.a_stages) == (1187, 1, 2, 594, 3)
    o = pkg.rows_matmul_plan(5120, 5120, 160, 0, 152)           # 40 tiles: 20 pairs x 5 K slices, one wave
    assert (o.tiles_big, o.k_slices, o.grid, o.a_stages) == (2, 5, 100, 3)
    gu = pkg.rows_matmul_plan(34816, 5120, 160, 1, 152)         # 272 tiles: 136 CTAs of 2, K whole
    assert (gu.k_slices, gu.tiles_big, gu.grid) == (1, 2, 136)
    down = pkg.rows_matmul_plan(5120, 17408, 160, 0, 152)       # 40 tiles over 272 groups: 20 pairs x 7 slices
    assert (down.tiles_big, down.k_slices, down.grid) == (2, 7, 140)
    tiny = pkg.rows_matmul_plan(16, 64, 1, 0, 152)              # one tile, one group
    assert (tiny.grid, tiny.k_slices, tiny.n_pad, tiny.tiles_big) == (1, 1, 16, 1)


def test_plan_rejects_bad_sizes(lib):
    p = pkg.dflash_rows_plan()
    L = lib
    assert L.dflash_rows_matmul_plan(5120, 5120, 161, 0, 152, ctypes.byref(p)) == pkg.DFLASH_ECAPACITY
    for args in ((5120, 5120, 0, 0, 152), (5120, 100, 16, 0, 152), (0, 5120, 16, 0, 152), (5120, 0, 16, 0, 152),
                 (5120, 5120, 16, 0, 0)):
        assert L.dflash_rows_matmul_plan(*args, ctypes.byref(p)) == pkg.DFLASH_EINVAL, args
    assert L.dflash_rows_matmul_plan(5120, 5120, 16, 0, 152, None) == pkg.DFLASH_EINVAL


def test_rows_matmul_validates_before_any_launch(lib):
    # a NULL handle is refused on the host; nothing reaches the device
    assert lib.dflash_rows_matmul(None, pkg.DFLASH_MAT_LM, 0, 16, None, None, 5120, None, 151936, None, 0,
                                  None) == pkg.DFLASH_EINVAL
    assert lib.dflash_rows_matmul(None, pkg.DFLASH_MAT_QKV, 0, 161, None, None, 5120, None, 7168, None, 0,
                                  None) == pkg.DFLASH_EINVAL


def test_large_batch_option_carves_the_contraction_scratch(lib):
    """large_batch_tc05 = 1 adds exactly the largest contraction scratch (the block projections and
    the head at 33 .. max_batch * gamma rows, capped at 160; W_c and the grouped context K/V at 33 .. 160
    context rows), the f16 copy of 160 context-tap rows, and room for 160 context rows in the per-layer input
    planes and their sums of squares to the workspace. It adds nothing where the option does not apply (one
    request of 8 rows, 16-bit weights, or a Markov head)."""
    import dflash_synth as syn
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("the workspace plan uses the device's SM count; checked here with the host default")
    cfg = syn.CONFIGS["c5"]
    off = pkg.make_config(cfg)
    on = pkg.make_config(syn.with_overrides(cfg, large_batch_tc05=True))
    rows = min(cfg.batch * cfg.gamma, pkg.DFLASH_ROWS_MATMUL_MAX)
    qkv = cfg.n_q_heads * cfg.head_dim + 2 * cfg.n_kv_heads * cfg.head_dim
    shapes = [(qkv, cfg.d), (cfg.d, cfg.n_q_heads * cfg.head_dim), (2 * cfg.inter, cfg.d), (cfg.d, cfg.inter),
              (cfg.vocab, cfg.d)]
    n_sm = 148   # the library's default when no device is present
    mh = cfg.n_taps * cfg.target_hidden
    # every many-row call size (33 rows up): the plan's K slices may grow as the rows shrink
    lo = {(qkv, cfg.d): 1, (2 * cfg.inter, cfg.d): 1, (cfg.vocab, cfg.d): 1}
    sizes = lambda top: [min(r, top) for r in range(33, top + 16, 16)]
    kvd = cfg.n_kv_heads * cfg.head_dim
    kv = [pkg.rows_matmul_plan(2 * kvd, cfg.d, r, 1, n_sm // cfg.n_layers) for r in sizes(pkg.DFLASH_ROWS_MATMUL_MAX)]
    want = max([pkg.rows_matmul_plan(n, k, r, lo.get((n, k), 0), n_sm).scratch_bytes for n, k in shapes
                for r in sizes(rows)] +
               [pkg.rows_matmul_plan(cfg.d, mh, r, 0, n_sm).scratch_bytes
                for r in sizes(pkg.DFLASH_ROWS_MATMUL_MAX)] +   # W_c
               # every layer's context K/V in one grouped launch: each layer's partial tiles, one row-scale area
               [cfg.n_layers * (p.scratch_bytes - 8 * 32 * 4) + 8 * 32 * 4 for p in kv])
    want = -(-want // 256) * 256
    want += -(-(pkg.DFLASH_ROWS_MATMUL_MAX * mh * 2) // 256) * 256   # context taps converted to f16
    # the head's vocab states: one slice per row chunk (up to 8) of n_sm CTAs x 32 rows x (max, sum, index)
    want += (8 - 1) * n_sm * 32 * 3 * 4
    # context rows of a call: 160 instead of 32 per input plane (f16 + remainder, one plane per layer),
    # and their sums of squares
    ssq_ld = -(-cfg.d // 16)
    want += cfg.n_layers * (160 - 32) * cfg.d * 2 * 2 + (160 - 32) * ssq_ld * 2 * 4
    diff = lib.dflash_workspace_bytes(ctypes.byref(on)) - lib.dflash_workspace_bytes(ctypes.byref(off))
    assert diff == want
    for over in (dict(batch=1, gamma=8), dict(wdtype="bf16"), dict(markov_rank=64)):
        a = pkg.make_config(syn.with_overrides(cfg, **over))
        b = pkg.make_config(syn.with_overrides(cfg, large_batch_tc05=True, **over))
        assert lib.dflash_workspace_bytes(ctypes.byref(b)) == lib.dflash_workspace_bytes(ctypes.byref(a)), over
