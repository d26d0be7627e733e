"""CPU-only checks of the C ABI: the library builds, loads and exports every entry point the
header declares; the ctypes mirrors have the C layout; host-side validation needs no GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import speculative_block_draft_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def lib():
    pkg.build()
    return pkg.lib()


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[a-z_0-9 ]+\*?\s*(dflash_[a-z_]+)\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (dflash_\w+)", out))
    assert set(names) <= exported
    assert set(pkg.SYMBOLS) == set(names)


def test_struct_layouts_match_c(tmp_path):
    src = tmp_path / "sz.c"
    src.write_text('#include "dflash.h"\n#include <stdio.h>\n#include <stddef.h>\nint main(){printf("%zu %zu %zu %zu %zu %zu %zu %zu",'
                   'sizeof(dflash_config), sizeof(dflash_matrix), sizeof(dflash_layer_weights), sizeof(dflash_weights),'
                   'sizeof(dflash_stats), offsetof(dflash_weights, layer), sizeof(dflash_rows_plan),'
                   'offsetof(dflash_rows_plan, smem_bytes));return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = list(map(int, subprocess.check_output([str(exe)]).split()))
    want = [ctypes.sizeof(pkg.dflash_config), ctypes.sizeof(pkg.dflash_matrix), ctypes.sizeof(pkg.dflash_layer_weights),
            ctypes.sizeof(pkg.dflash_weights), ctypes.sizeof(pkg.dflash_stats), pkg.dflash_weights.layer.offset,
            ctypes.sizeof(pkg.dflash_rows_plan), pkg.dflash_rows_plan.smem_bytes.offset]
    assert got == want


def test_host_validation_without_gpu(lib):
    bad = pkg.dflash_config()
    assert lib.dflash_workspace_bytes(ctypes.byref(bad)) == 0
    import dflash_synth as syn
    good = pkg.make_config(syn.CONFIGS["c3"])
    assert lib.dflash_workspace_bytes(ctypes.byref(good)) > 1_400_000_000   # repacked drafter + head
    for field, val in (("head_dim", 96), ("gamma", 1), ("gamma", 17), ("max_batch", 65), ("adtype", 7),
                       ("ffn_act", 2), ("draft_all_rows", 2), ("markov_rank", 96), ("markov_rank", 2048),
                       ("large_batch_tc05", 2), ("large_batch_tc05", -1)):
        c = pkg.make_config(syn.CONFIGS["c3"])
        setattr(c, field, val)
        assert lib.dflash_workspace_bytes(ctypes.byref(c)) == 0, field
    c = pkg.make_config(syn.CONFIGS["c3"], ctx_capacity=1000)        # ring smaller than the window
    assert lib.dflash_workspace_bytes(ctypes.byref(c)) == 0
    h = ctypes.c_void_p()
    assert lib.dflash_create(ctypes.byref(good), None, None, 0, None, ctypes.byref(h)) == pkg.DFLASH_EINVAL
    assert lib.dflash_draft_block(None, 1, None, None, 0.0, None, None, None, None) == pkg.DFLASH_EINVAL
    assert lib.dflash_ctx_len(None, 0) == -1
    assert lib.dflash_draft_lengths(None, 1, None, None, 0.0, None, None) == pkg.DFLASH_EINVAL
    assert lib.dflash_accept_kept(None, 1, None, None, None, None, None, None) == pkg.DFLASH_EINVAL
    assert lib.dflash_accept(None, 1, None, None, None, None, None) == pkg.DFLASH_EINVAL
    assert lib.dflash_set_wait_limit(None, 1000, None) == pkg.DFLASH_EINVAL
    assert lib.dflash_debug_stall(None, 0) == pkg.DFLASH_EINVAL
    assert lib.dflash_accept_histogram(None, None, 1, None) == pkg.DFLASH_EINVAL
    assert b"declined" in lib.dflash_status_str(pkg.DFLASH_DECLINED)


def test_debug_build_exports_the_same_symbols():
    """The bounds-checking build compiles for sm_103a and exports every declared entry point."""
    path = pkg.build(debug=True)
    assert path == pkg.LIB_PATH_DEBUG
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    assert set(declared()) <= set(re.findall(r" T (dflash_\w+)", out))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """With the compiled library absent the binding raises; there is no CPU fallback to take."""
    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "libdflash.so"))
    monkeypatch.setattr(pkg, "LIB_PATH_DEBUG", str(tmp_path / "libdflash_debug.so"))
    with pytest.raises(RuntimeError, match="not built"):
        pkg.lib()
