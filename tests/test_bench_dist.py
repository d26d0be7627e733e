"""The bench's host logic on CPU: the multi-GPU replicas (max elapsed over ranks, units summed;
gloo, world size 2), the oracle timing table and the reference arm's line."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    t, u = bench.reduce_over_ranks(1.5 + rank, 10.0 * (rank + 1))
    q.put((rank, t, u, bench.dist_env()[:2]))
    dist.destroy_process_group()


def test_reduce_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
    assert [r[1:3] for r in res] == [(2.5, 30.0), (2.5, 30.0)]
    assert [r[3] for r in res] == [(0, 2), (1, 2)]


def test_round_bytes_match_the_c3_budget():
    sys.path.insert(0, ROOT)
    import bench
    import dflash_synth as syn
    b = bench.round_bytes(syn.CONFIGS["c3"], [4096])
    assert abs(b["total"] / 1e6 - 1482.2) < 0.5          # layers 929.0 + head 437.6 + W_c 73.7 + KV 41.9
    assert abs(b["lm_head"] / 1e6 - 437.6) < 0.1


def test_round_flops_c5_hand_count():
    """The batched workload's algorithmic FLOP per round, counted by hand: 160 block rows through
    five layers of (Q/K/V 5120x7168, O 5120x5120, gate/up/down 3x5120x17408), 128 drafting rows
    through the 151936x5120 head, 144 new context rows through W_c (5120x25600) and each layer's
    context K/V (2x1024x5120), and the block attention over a 2048-key window plus the 5 block keys."""
    sys.path.insert(0, ROOT)
    import bench
    import dflash_synth as syn
    cfg = syn.CONFIGS["c5"]
    f = bench.round_flops(cfg, [4096] * 32, 144.0)
    layer = 5120 * 7168 + 5120 * 5120 + 3 * 5120 * 17408
    assert f["layers"] == 2 * 160 * 5 * layer
    assert f["lm_head"] == 2 * 128 * 151936 * 5120
    assert f["W_c"] == 2 * 144 * 5120 * 25600
    assert f["ctx_kv"] == 2 * 144 * 5 * 2048 * 5120
    assert f["attention"] == 4 * 5 * 40 * 5 * (32 * (2048 + 5)) * 128
    assert abs(f["total"] - sum(v for k, v in f.items() if k != "total")) < 1


def test_probe_classes_cover_the_round_bytes():
    """The live per-kernel roofline classes: the layer classes (x L) add up to the round's layer
    bytes, the head and W_c to theirs, attention to the window's K/V bytes; the context K/V launch
    re-streams W_k and W_v of every layer."""
    sys.path.insert(0, ROOT)
    import bench
    import dflash_synth as syn
    cfg = syn.CONFIGS["c3"]
    rb = bench.round_bytes(cfg, [4096])
    cls = {name: (kind, n, b) for name, kind, n, b in bench.probe_classes(cfg, [4096], 8.0)}
    assert sorted(k for k, _, _ in cls.values()) == list(range(8))
    layer = sum(n * b for name, (_, n, b) in cls.items() if name in ("qkv", "o", "gate_up", "down"))
    assert abs(layer - rb["layers"]) < 1 and abs(cls["lm_head"][2] - rb["lm_head"]) < 1
    assert abs(cls["w_c"][2] - rb["W_c"]) < 1 and abs(cls["attention"][1] * cls["attention"][2] - rb["kv"]) < 1
    assert abs(cls["ctx_kv"][2] - 5 * 2 * 1024 * 5120 * bench.Q4_BYTES_PER_PARAM) < 1


def test_probe_classes_count_context_blocks_on_the_tcgen05_path():
    """Context calls of more than 32 rows on the tcgen05 path run W_c and every layer's K/V once per
    block of up to 160 rows; the GEMV path once per 32-row chunk."""
    sys.path.insert(0, ROOT)
    import bench
    import dflash_synth as syn
    cfg = syn.CONFIGS["c5"]
    tc = syn.with_overrides(cfg, large_batch_tc05=True)
    for rows, gemv_n, tc_n in ((144.0, 5, 1), (200.0, 7, 2), (20.0, 1, 1)):
        g = {name: n for name, _, n, _ in bench.probe_classes(cfg, [4096] * 32, rows)}
        t = {name: n for name, _, n, _ in bench.probe_classes(tc, [4096] * 32, rows)}
        assert g["w_c"] == g["ctx_kv"] == gemv_n, rows
        assert t["w_c"] == t["ctx_kv"] == tc_n, rows


def test_oracle_table_one_core_and_all_cores():
    """The oracle timing table (1 core and all cores per workload) on the tiny fp32 drafter."""
    import bench
    t = bench.oracle_table(("c1",))
    rows = t["oracle_table"]
    assert {r["threads"] for r in rows} == {1, t["cores"]}
    for r in rows:
        assert r["config"] == "c1" and r["round_s"] > 0 and abs(r["blocks_per_s"] * r["round_s"] - 1) < 1e-9


def _run_bench(args, env_extra):
    import json
    import subprocess
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       env=env, cwd=ROOT, timeout=600)
    lines = [json.loads(s) for s in r.stdout.splitlines() if s.startswith("{")]
    return r.returncode, lines, r.stderr


def test_reference_arm_line_on_the_small_drafter():
    """`bench.py --impl reference` times the oracle on the host and prints one JSON line with the
    contract's keys: impl, metric/unit/value, the cpu_baseline that describes this run (its value is
    the line's), and an e2e object with no host-device copies."""
    rc, lines, err = _run_bench(["--impl", "reference", "--config", "c1", "--steps", "2", "--warmup", "3"],
                                {"RANK": "0", "WORLD_SIZE": "1"})
    assert rc == 0, err
    assert len(lines) == 1
    ln = lines[0]
    assert ln["impl"] == "reference" and ln["unit"] == "blocks/s" and ln["higher_is_better"] is True
    assert ln["steps"] == 2 and ln["warmup"] == 3 and ln["dtype"] == "f64" and ln["value"] > 0
    assert ln["config"]["workload"].startswith("c1")
    cb = ln["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == ln["value"] and cb["cores"] >= 1 and cb["sample"]
    assert ln["e2e"] == {"value": ln["value"], "unit": "blocks/s", "h2d_bytes_per_step": 0,
                         "d2h_bytes_per_step": 0}
    assert abs(ln["ms_per_step"] - 1e3 / ln["value"]) < 1e-6 * ln["ms_per_step"]


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs the reference arm and prints; the other ranks exit 0 silently."""
    rc, lines, err = _run_bench(["--impl", "reference", "--config", "c1", "--steps", "2", "--warmup", "3"],
                                {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert rc == 0, err
    assert lines == []


def _classes_and_times(cfg, lengths, ctx_rows, dominant):
    import bench
    classes = bench.probe_classes(cfg, lengths, ctx_rows)
    ms = {name: 0.01 for name, _, _, _ in classes}
    ms[dominant] = 0.1
    return classes, ms


@pytest.mark.parametrize("name,tc", [("c3", False), ("c5", False), ("c5", True)])
def test_class_flops_add_up_to_the_round(name, tc):
    """Per-launch FLOP of the probed classes times their launches per round equal the round's
    algorithmic FLOP, on either projection path."""
    sys.path.insert(0, ROOT)
    import bench
    import dflash_synth as syn
    cfg = syn.with_overrides(syn.CONFIGS[name], large_batch_tc05=tc)
    lengths = [4096] * cfg.batch
    ctx_rows = 144.0 if cfg.batch > 1 else 8.0
    fl = bench.class_flops(cfg, lengths, ctx_rows)
    total = sum(fl[n] * per_round for n, _, per_round, _ in bench.probe_classes(cfg, lengths, ctx_rows))
    assert abs(total - bench.round_flops(cfg, lengths, ctx_rows)["total"]) <= 1e-9 * total


def test_rooflines_gemv_round_is_hbm_bound():
    """The 8-row round (one request): every class on the GEMV, the dominant one reported in GB/s
    against the copy bandwidth, with its ncu traffic lookup."""
    sys.path.insert(0, ROOT)
    import bench
    import dflash_synth as syn
    cfg = syn.CONFIGS["c3"]
    classes, ms = _classes_and_times(cfg, [4096], 8.0, "gate_up")
    peaks = {"hbm_gbs": 6660.3, "bf16_tflops": 1884.6, "bf16_tflops_sustained": 1723.8, "source": "measured"}
    by, roof = bench.class_rooflines(cfg, classes, ms, 0.58, peaks, [4096], 8.0)
    assert all(v["path"] in ("gemv", "attention") and v["bound"] == "hbm" for v in by.values())
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["kernel"].startswith("gate_up: 4-bit GEMV")
    nbytes = 2 * cfg.inter * cfg.d * 0.5625
    assert abs(roof["achieved"] - nbytes / 1e-4 / 1e9) < 1e-6 * roof["achieved"]
    assert abs(roof["frac"] - roof["achieved"] / 6660.3) < 1e-12
    assert "traffic" in roof and abs(by["gate_up"]["share_of_round"] - 0.1 * 5 / 0.58) < 1e-12


def test_rooflines_batched_tcgen05_round_is_tensor_bound():
    """The batched round on the tcgen05 path (160 block rows, 144 context rows per round): the
    block projections, the head and the context classes are contractions above the ridge, reported
    in TFLOP/s against the burst tensor peak; attention stays HBM-bound; without the option the same
    round is all GEMV."""
    sys.path.insert(0, ROOT)
    import bench
    import dflash_synth as syn
    peaks = {"hbm_gbs": 6660.3, "bf16_tflops": 1884.6, "bf16_tflops_sustained": 1723.8, "source": "measured"}
    cfg = syn.with_overrides(syn.CONFIGS["c5"], large_batch_tc05=True)
    lengths = [4096] * 32
    assert bench.tc05_classes(cfg, 144.0) == {"qkv", "o", "gate_up", "down", "lm_head", "w_c", "ctx_kv"}
    assert bench.tc05_classes(cfg, 20.0) == {"qkv", "o", "gate_up", "down", "lm_head"}
    classes, ms = _classes_and_times(cfg, lengths, 144.0, "gate_up")
    by, roof = bench.class_rooflines(cfg, classes, ms, 2.0, peaks, lengths, 144.0)
    assert by["attention"]["bound"] == "hbm" and by["attention"]["path"] == "attention"
    assert all(by[n]["bound"] == "tensor" and by[n]["path"] == "tcgen05" for n in ("qkv", "o", "gate_up", "down", "lm_head"))
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["traffic"] is None
    assert roof["kernel"].startswith("gate_up: tcgen05 contraction")
    flop = 2.0 * 160 * 2 * cfg.inter * cfg.d
    assert abs(roof["achieved"] - flop / 1e-4 / 1e12) < 1e-9 * roof["achieved"]
    assert abs(roof["frac"] - roof["achieved"] / 1884.6) < 1e-12 and roof["peak"] == 1884.6
    off = syn.CONFIGS["c5"]
    assert bench.tc05_classes(off, 144.0) == set()
    by_off, roof_off = bench.class_rooflines(off, *_classes_and_times(off, lengths, 144.0, "gate_up"), 2.0, peaks,
                                             lengths, 144.0)
    assert roof_off["bound"] == "hbm" and all(v["path"] != "tcgen05" for v in by_off.values())
