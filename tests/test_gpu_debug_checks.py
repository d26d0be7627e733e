"""The bounds-checking debug build (DFL_DEBUG_CHECKS), the stand-in for a memory checker: the same
kernels report out-of-range device-side values through the error word (DFLASH_EBOUNDS) instead
of only clamping or skipping them. A debug library is a process-wide choice (the environment
variable DFLASH_DEBUG_CHECKS=1 selects it when the binding loads), so these tests run a subset of
the parity suite and the reporting cases in a child process with it set; the release build's own
behaviour on the same out-of-range inputs (clamped, nothing reported) is checked here."""
import os
import subprocess
import sys

import numpy as np
import pytest

import dflash_synth as syn

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _debug() -> bool:
    return os.environ.get("DFLASH_DEBUG_CHECKS") == "1"


def _cfg():
    return syn.DraftConfig("s_dbg", n_layers=2, d=256, n_q_heads=4, n_kv_heads=2, head_dim=64, inter=512, n_taps=2,
                           target_hidden=256, vocab=1000, gamma=5, window=0, ctx_len=40, wdtype="q4",
                           adtype="bf16", seed=17)


def test_debug_build_runs_parity_subset_and_reports():
    """Child process on the debug library: parity cases that cover the GEMV (split K, clusters,
    grouped context K/V), attention, both tcgen05 kernels, the Markov head and acceptance finish
    with a clear error word and the oracle's results; the reporting cases below fail loudly."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if _debug():
        pytest.skip("already the child process")
    import speculative_block_draft_gb300 as pkg
    pkg.build(debug=True)
    mark = os.path.join(ROOT, "speculative_block_draft_gb300", "_build_debug", "reports.ok")
    if os.path.exists(mark):
        os.remove(mark)
    env = dict(os.environ, DFLASH_DEBUG_CHECKS="1", DFLASH_DEBUG_MARK=mark)
    sel = ("small_formats_and_head_dims and q4 or batch_ragged or sliding_window or markov_head_batched or "
           "accept_kernel or draft_lengths or small_skinny_tc05 or large_batch_round_small or "
           "rows_matmul_small_shapes or reports_out_of_range")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", sel,
                        "tests/test_gpu_parity.py", "tests/test_gpu_tc05.py", "tests/test_gpu_debug_checks.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    print(r.stdout[-3000:], r.stderr[-2000:])
    assert r.returncode == 0
    assert os.path.exists(mark), "the reporting cases did not run on the debug library"


def _session():
    from speculative_block_draft_gb300.session import Session
    cfg = _cfg()
    s = Session(syn.make_model(cfg, norm_jitter=0.1), max_batch=1, ctx_capacity=64)
    assert s.project([0], [cfg.ctx_len], syn.taps_rows(cfg, cfg.seed, 0, 0, cfg.ctx_len)) == 0
    return cfg, s


def test_reports_out_of_range_inputs():
    """Debug build only (it runs in the child process): an anchor outside the vocabulary and a
    kept-draft count above the block are clamped as in every build, and reported."""
    if not _debug():
        pytest.skip("needs the debug library (runs in the child process of the test above)")
    import speculative_block_draft_gb300 as pkg
    cfg, s = _session()
    g = s.draft([0], np.array([cfg.vocab + 3], dtype=np.int32), logits=False)
    assert g["rc"] == 0
    with pytest.raises(pkg.DFlashError) as e:
        s.check()
    assert e.value.status == pkg.DFLASH_EBOUNDS
    assert s.check() == 0
    n = cfg.n_draft
    d = np.zeros((1, n), dtype=np.int32)
    al, _ = s.accept_kept(d, np.array([n + 4], dtype=np.int32), np.zeros((1, n + 1), dtype=np.int32))
    assert al[0] == n
    with pytest.raises(pkg.DFlashError) as e:
        s.check()
    assert e.value.status == pkg.DFLASH_EBOUNDS
    g = s.draft([0], np.array([5], dtype=np.int32), logits=False)
    assert g["rc"] == 0 and s.check() == 0
    s.close()
    if os.environ.get("DFLASH_DEBUG_MARK"):
        with open(os.environ["DFLASH_DEBUG_MARK"], "w") as f:
            f.write("ok\n")


def test_release_build_clamps_silently():
    """Release build: the same out-of-range anchor drafts exactly what the last vocabulary entry
    drafts, and nothing is reported."""
    if _debug():
        pytest.skip("release behaviour")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_block_draft_gb300 as pkg
    pkg.build()
    cfg, s = _session()
    g1 = s.draft([0], np.array([cfg.vocab + 3], dtype=np.int32), logits=True)
    assert s.check() == 0
    g2 = s.draft([0], np.array([cfg.vocab - 1], dtype=np.int32), logits=True)
    assert s.check() == 0
    assert np.array_equal(g1["tokens"], g2["tokens"]) and np.array_equal(g1["logits"], g2["logits"])
    s.close()
