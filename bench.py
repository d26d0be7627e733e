"""Draft-round benchmark: draft blocks/s and achieved HBM GB/s on one GB300 (replicas for N > 1).

A step is one speculative round for every request of the workload: dflash_project_ctx (the
round's new context rows), dflash_draft_block, dflash_accept. Default workload: the page-1 DFlash2
geometry, 4-bit (config c3). Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c3] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dflash_synth as syn  # noqa: E402

Q4_BYTES_PER_PARAM = 0.5 + 4.0 / 64.0   # 4-bit code + bf16 scale and bias per 64 inputs
BYTES_PER_PARAM = {"q4": Q4_BYTES_PER_PARAM, "bf16": 2.0, "f32": 4.0}


# ---------------------------------------------------------------------------------------------
# algorithmic work of one round
# ---------------------------------------------------------------------------------------------
def round_params(cfg) -> dict:
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    layer = cfg.d * (qd + 2 * kvd) + qd * cfg.d + 3 * cfg.d * cfg.inter
    p = {"W_c": cfg.d * cfg.n_taps * cfg.target_hidden, "layers": cfg.n_layers * layer,
         "lm_head": cfg.vocab * cfg.target_hidden}
    if cfg.d != cfg.target_hidden:
        p["tok_out_proj"] = 2 * cfg.d * cfg.target_hidden
    return p


def round_bytes(cfg, ctx_lens) -> dict:
    bpp = BYTES_PER_PARAM[cfg.wdtype]
    b = {k: v * bpp for k, v in round_params(cfg).items()}
    kvd = cfg.n_kv_heads * cfg.head_dim
    act = 4 if cfg.adtype == "f32" else 2
    keys = sum(min(int(P), cfg.window) if cfg.window else int(P) for P in ctx_lens)
    b["kv"] = cfg.n_layers * keys * kvd * 2 * act
    if cfg.markov_rank:   # W2 of the Markov head streamed once per draft, plus the W1 rows
        b["markov"] = cfg.n_draft * cfg.vocab * cfg.markov_rank * bpp + cfg.batch * cfg.n_draft * cfg.markov_rank * bpp
    b["total"] = sum(b.values())
    return b


def round_flops(cfg, ctx_lens, ctx_rows: float) -> dict:
    """Algorithmic multiply-add work of one round (2 FLOP per weight and activation row):
    projections of every block row, the head over the drafting rows, W_c and each layer's context
    K/V over the round's new context rows, and the block attention (QK^T and PV)."""
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    p = round_params(cfg)
    rows_b, rows_d = cfg.batch * cfg.gamma, cfg.batch * cfg.n_draft
    f = {"layers": 2.0 * rows_b * p["layers"], "lm_head": 2.0 * rows_d * p["lm_head"],
         "W_c": 2.0 * ctx_rows * p["W_c"], "ctx_kv": 2.0 * ctx_rows * cfg.n_layers * 2 * kvd * cfg.d}
    if "tok_out_proj" in p:
        f["tok_out_proj"] = 2.0 * (cfg.batch + rows_d) * p["tok_out_proj"] / 2
    keys = sum((min(int(P), cfg.window) if cfg.window else int(P)) + cfg.gamma for P in ctx_lens)
    f["attention"] = 4.0 * cfg.n_layers * cfg.n_q_heads * cfg.gamma * keys * cfg.head_dim
    f["total"] = sum(f.values())
    return f


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1900.0)),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d.get("bf16_tflops", 1700.0))),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def load_traffic(kernel: str):
    """ncu DRAM bytes per launch of `kernel` (a PROBES name), if captured on the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d[kernel]
        if ent.get("source_hash") != kernel_source_hash(tuple(ent.get("sources", LM_HEAD_SOURCES))):
            return None
        return float(ent["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# The sources the projection launches are compiled from: the GEMV kernel and its epilogues, the
# vocab merge, and the constants and helpers they include. A change to any of them voids a record.
LM_HEAD_SOURCES = ("common.cuh", "gemv_f32.cu", "gemv_impl.cuh", "gemv_q4.cu", "internal.h")
ATTN_SOURCES = ("attn.cu", "common.cuh", "internal.h")

def on_tc05(cfg) -> bool:
    """Whether the library's many-row option applies to this drafter (4-bit weights, d == H, no
    Markov head): calls of more than 32 rows then run on the tcgen05 contraction."""
    return (bool(getattr(cfg, "large_batch_tc05", False)) and cfg.wdtype == "q4" and cfg.d == cfg.target_hidden
            and not getattr(cfg, "markov_rank", 0))


def ctx_calls(cfg, ctx_rows_per_round):
    """(launches per round, rows per launch) of the context classes: one per block of up to 160
    rows on the tcgen05 path (calls of more than 32 rows), else one per 32-row chunk."""
    rows = int(round(ctx_rows_per_round))
    tc = on_tc05(cfg) and rows > 32
    chunks = max(1, -(-rows // (160 if tc else 32)))
    return chunks, ctx_rows_per_round / chunks, tc


def tc05_classes(cfg, ctx_rows_per_round) -> set:
    """The probed classes that run on the tcgen05 contraction: every block projection and the head
    when a draft call carries 33-160 block rows, the context classes when a context call carries
    more than 32 rows."""
    if not on_tc05(cfg):
        return set()
    out = set()
    if 32 < cfg.batch * cfg.gamma <= 160:
        out |= {"qkv", "o", "gate_up", "down", "lm_head"}
    if ctx_calls(cfg, ctx_rows_per_round)[2]:
        out |= {"w_c", "ctx_kv"}
    return out


# Kernel classes of a round that bench.py times live (dflash_set_probe kinds): name, probe kind,
# launches per round, algorithmic bytes per launch (weights at their stored size; attention: the
# window's context K and V rows of one layer).
def probe_classes(cfg, ctx_lens, ctx_rows_per_round):
    bpp = BYTES_PER_PARAM[cfg.wdtype]
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    act = 4 if cfg.adtype == "f32" else 2
    keys = sum(min(int(P), cfg.window) if cfg.window else int(P) for P in ctx_lens)
    L, d, I = cfg.n_layers, cfg.d, cfg.inter
    # context calls of more than 32 rows on the tcgen05 path: W_c and every layer's K/V once per
    # block of up to 160 rows (the probes bracket a whole block); otherwise once per 32-row chunk
    chunks = ctx_calls(cfg, ctx_rows_per_round)[0]
    return [("lm_head", 0, 1, cfg.vocab * cfg.target_hidden * bpp),
            ("qkv", 1, L, (qd + 2 * kvd) * d * bpp),
            ("attention", 2, L, keys * kvd * 2 * act),
            ("o", 3, L, d * qd * bpp),
            ("gate_up", 4, L, 2 * I * d * bpp),
            ("down", 5, L, d * I * bpp),
            ("w_c", 6, chunks, d * cfg.n_taps * cfg.target_hidden * bpp),
            ("ctx_kv", 7, chunks, L * 2 * kvd * d * bpp)]


def class_flops(cfg, ctx_lens, ctx_rows_per_round) -> dict:
    """Algorithmic FLOP per launch of each probed class (2 per weight and activation row; attention:
    QK^T and PV over the window's keys plus the block's own). Summed with the launches per round of
    probe_classes they give round_flops' total (d == H)."""
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    L, d, I = cfg.n_layers, cfg.d, cfg.inter
    rows_b, rows_d = cfg.batch * cfg.gamma, cfg.batch * cfg.n_draft
    keys = sum((min(int(P), cfg.window) if cfg.window else int(P)) + cfg.gamma for P in ctx_lens)
    rows_c = ctx_calls(cfg, ctx_rows_per_round)[1]
    return {"lm_head": 2.0 * rows_d * cfg.vocab * cfg.target_hidden,
            "qkv": 2.0 * rows_b * (qd + 2 * kvd) * d,
            "attention": 4.0 * cfg.n_q_heads * cfg.gamma * keys * cfg.head_dim,
            "o": 2.0 * rows_b * d * qd,
            "gate_up": 2.0 * rows_b * 2 * I * d,
            "down": 2.0 * rows_b * d * I,
            "w_c": 2.0 * rows_c * d * cfg.n_taps * cfg.target_hidden,
            "ctx_kv": 2.0 * rows_c * L * 2 * kvd * d}


GEMV_LABELS = {"lm_head": "4-bit GEMV + fused argmax/softmax confidence, then the vocab merge",
               "attention": "block attention over the window (+ split merge)",
               "w_c": "4-bit GEMV, context projection (Eq 2) + ctx norm sums",
               "ctx_kv": "4-bit GEMV, context K/V of every layer, one grouped launch"}
TC05_LABELS = {"lm_head": "tcgen05 contraction over every drafting row + vocab-state epilogue, then the vocab merge",
               "w_c": "tcgen05 contraction, context projection (Eq 2) of a block of up to 160 rows + chunk epilogues",
               "ctx_kv": "tcgen05 contraction, context K/V of every layer in one grouped launch + epilogue"}


def class_rooflines(cfg, classes, class_ms, t_round_ms, peaks, ctx_lens, ctx_rows_per_round):
    """Per probed class: live time, share of the round, algorithmic bytes and FLOP per launch and
    both fractions; and the roofline object of the class with the largest share. A class on the
    tcgen05 contraction whose FLOP per byte is above the ridge (tensor peak / HBM peak) is reported
    against the tensor peak (the burst bf16 figure: f16 operands run at the bf16 rate), every other
    class against the HBM copy bandwidth."""
    flops = class_flops(cfg, ctx_lens, ctx_rows_per_round)
    tc = tc05_classes(cfg, ctx_rows_per_round)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    by_kernel = {}
    for name, kind, per_round, nbytes in classes:
        ms = class_ms[name]
        gbs = nbytes / (ms / 1e3) / 1e9
        tfs = flops[name] / (ms / 1e3) / 1e12
        bound = "tensor" if name in tc and flops[name] / nbytes > ridge else "hbm"
        by_kernel[name] = {"avg_launch_us": 1e3 * ms, "launches_per_round": per_round,
                           "share_of_round": ms * per_round / t_round_ms, "algorithmic_bytes_per_launch": nbytes,
                           "achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
                           "algorithmic_flop_per_launch": flops[name], "achieved_tflops": tfs,
                           "tensor_frac": tfs / peaks["bf16_tflops"],
                           "path": "tcgen05" if name in tc else ("attention" if name == "attention" else "gemv"),
                           "bound": bound}
    dom = max(by_kernel, key=lambda k: by_kernel[k]["share_of_round"])
    dk = by_kernel[dom]
    labels = TC05_LABELS if dom in tc else GEMV_LABELS
    default = ("tcgen05 contraction over every block row + fused epilogue, layer 0 (the layers are identical)"
               if dom in tc else "4-bit GEMV with fused epilogue, layer 0 (the layers are identical)")
    roof = {"kernel": f"{dom}: " + labels.get(dom, default), "bound": dk["bound"]}
    if dk["bound"] == "tensor":
        roof.update({"achieved": dk["achieved_tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": dk["tensor_frac"], "traffic": None,
                     "algorithmic_flop_per_launch": dk["algorithmic_flop_per_launch"],
                     "hbm_frac": dk["frac"],
                     "peak_source": f"{peaks['source']} (cuBLAS bf16 burst, MEASURED_PEAKS.json bf16_tflops)"})
    else:
        roof.update({"achieved": dk["achieved_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": dk["frac"], "traffic": None if dom in tc else load_traffic(dom),
                     "algorithmic_bytes_per_launch": dk["algorithmic_bytes_per_launch"],
                     "peak_source": f"{peaks['source']} (burst copy, MEASURED_PEAKS.json hbm_gbs)"})
    roof.update({"avg_launch_ms": dk["avg_launch_us"] / 1e3, "share_of_round": dk["share_of_round"]})
    return by_kernel, roof


def kernel_source_hash(names=LM_HEAD_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_block_draft_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        ids = [x.strip() for x in vis.split(",")] if vis else []
        self.dev = ids[device_index] if device_index < len(ids) else str(device_index)
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.dev, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# distributed helpers (replicas: no data-path collective; timing max over ranks)
# ---------------------------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def reduce_over_ranks(elapsed_s: float, units: float, group=None):
    """(max elapsed over ranks, sum of units over ranks); identity when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------------------------
def oracle_round_seconds(cfg, model, rounds: int = 1, scale_rows: int = 1):
    """Wall time of the oracle for one round of request 0 (ctx rows projected, block drafted over
    a full window, accept). The context window's K/V are drawn from the generator (the oracle's
    cost does not depend on their values), so no multi-minute prefill is needed.
    scale_rows > 1 times only 1/scale_rows of every matrix's output rows and scales up."""
    import oracle
    n_new = cfg.appends()[0]
    P = cfg.ctx_len
    nwin = min(P, cfg.window) if cfg.window else P
    kvd = cfg.n_kv_heads * cfg.head_dim
    k = syn.normal(cfg.seed, "bench.kctx", (cfg.n_layers, nwin, kvd), 1.0).astype(np.float64)
    v = syn.normal(cfg.seed, "bench.vctx", (cfg.n_layers, nwin, kvd), 1.0).astype(np.float64)
    taps = syn.taps_to_f32(cfg, syn.taps_rows(cfg, cfg.seed, 0, P, n_new)).astype(np.float64)
    if scale_rows == 1:
        o = oracle.Oracle(model)
        times = []
        for r in range(rounds):
            t0 = time.perf_counter()
            kn, vn = o.ctx_rows(taps)
            kk = np.concatenate([k, kn], axis=1)[:, -nwin:] if cfg.window else np.concatenate([k, kn], axis=1)
            vv = np.concatenate([v, vn], axis=1)[:, -nwin:] if cfg.window else np.concatenate([v, vn], axis=1)
            out = o.draft(int(syn.anchors(cfg.seed, 1, r, cfg.vocab)[0]), np.ascontiguousarray(kk),
                          np.ascontiguousarray(vv))
            t = syn.target_tokens(cfg.seed, 0, r, out["tokens"], cfg.agree or 0.0, cfg.vocab)
            oracle.accept(out["tokens"], t)
            times.append(time.perf_counter() - t0)
        return times
    # sampled step: the oracle's projections on a row slice of every matrix of the round
    import dflash_synth
    G = cfg.gamma
    xs = {}
    t0 = time.perf_counter()
    for name, hm in model.mats.items():
        if name == "embed":
            continue
        rows = max(16, hm.n_out // scale_rows)
        part = dflash_synth.HostMatrix(hm.fmt, rows, hm.n_in, hm.data[:rows],
                                       None if hm.scale is None else hm.scale[:rows],
                                       None if hm.bias is None else hm.bias[:rows])
        nrow = n_new if name == "W_c" else (cfg.n_draft if name in ("lm_head", "out_proj") else G)
        if name not in xs or xs[name].shape != (nrow, hm.n_in):
            xs[name] = syn.normal(cfg.seed, "bench.x", (nrow, hm.n_in), 1.0).astype(np.float64)
        oracle.linear(part, xs[name])
        if name.endswith((".k", ".v")):
            oracle.linear(part, xs[name][:1].repeat(n_new, axis=0))
    return [(time.perf_counter() - t0) * scale_rows]


def set_oracle_threads(n: int):
    """OpenMP threads of the oracle's shared library (the process's one OpenMP runtime)."""
    import ctypes
    import ctypes.util
    import oracle
    oracle._load()
    gomp = ctypes.CDLL(ctypes.util.find_library("gomp") or "libgomp.so.1")
    gomp.omp_set_num_threads(int(n))


def rows_matmul_bench(which: str, rows_list, iters: int = 5) -> dict:
    """Time dflash_rows_matmul (the many-row tcgen05 contraction) on one stored matrix of the
    4-bit 5120-wide drafter (a one-layer drafter with the full head, so the model stays small):
    per row count, the call's time (contraction + slice reduction) and its algorithmic rates."""
    import torch

    import speculative_block_draft_gb300 as pkg
    from speculative_block_draft_gb300.session import Session
    pkg.build()
    c3 = syn.CONFIGS["c3"]
    cfg = syn.with_overrides(c3, name="rows_matmul_l1", n_layers=1, window=0, ctx_len=16)
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    shapes = {"lm": (pkg.DFLASH_MAT_LM, cfg.vocab, cfg.target_hidden), "ctx": (pkg.DFLASH_MAT_CTX, cfg.d, cfg.n_taps * cfg.target_hidden),
              "qkv": (pkg.DFLASH_MAT_QKV, qd + 2 * kvd, cfg.d), "o": (pkg.DFLASH_MAT_O, cfg.d, qd),
              "gateup": (pkg.DFLASH_MAT_GATEUP, 2 * cfg.inter, cfg.d), "down": (pkg.DFLASH_MAT_DOWN, cfg.d, cfg.inter)}
    mat, n_out, k = shapes[which]
    s = Session(syn.make_model(cfg), max_batch=1, ctx_capacity=64)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    peaks = load_peaks()
    out = []
    for rows in rows_list:
        plan = pkg.rows_matmul_plan(n_out, k, rows, 0, nsm)
        sc = torch.empty(plan.scratch_bytes + 256, dtype=torch.uint8, device="cuda")
        sc = sc[(256 - sc.data_ptr() % 256) % 256:]
        x = torch.randn(rows, k, device="cuda").half().view(torch.int16)
        y = torch.empty(rows, n_out, dtype=torch.float32, device="cuda")
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ms = []
        for _ in range(iters):
            ev[0].record()
            s.h.rows_matmul(mat, 0, x, y, sc)
            ev[1].record()
            torch.cuda.synchronize()
            ms.append(ev[0].elapsed_time(ev[1]))
        t = float(np.median(ms)) / 1e3
        wbytes = n_out * k * Q4_BYTES_PER_PARAM
        out.append({"rows": rows, "us": 1e6 * t, "grid": plan.grid, "k_slices": plan.k_slices,
                    "weights_gbs": wbytes / t / 1e9, "hbm_frac": wbytes / t / 1e9 / peaks["hbm_gbs"],
                    "tflops": 2 * rows * n_out * k / t / 1e12,
                    "tensor_frac": 2 * rows * n_out * k / t / 1e12 / peaks["bf16_tflops_sustained"]})
    assert s.check() == 0
    s.close()
    return {"rows_matmul": which, "shape": [n_out, k], "results": out}


def oracle_table(names=("c1", "c2", "c3", "c5")):
    """Oracle blocks/s for one round on 1 core and on all cores, per workload. A round of a
    batched workload is its requests' rounds in sequence (requests are independent, and with the
    window every request attends to the same number of keys), timed as request 0's round x B.
    Large drafters on 1 core time a 1/16 row sample of every matrix (attention, <1% of the work,
    left out), scaled back up."""
    import platform
    cores = os.cpu_count() or 1
    out = []
    for name in names:
        cfg = syn.CONFIGS[name]
        model = syn.make_model(cfg)
        big = cfg.d * cfg.inter >= 4096 * 4096
        for threads in sorted({1, cores}):
            set_oracle_threads(threads)
            scale = 16 if (big and threads == 1) else 1
            t_req = oracle_round_seconds(cfg, model, rounds=1, scale_rows=scale)[0]
            out.append({"config": name, "threads": threads, "round_s": t_req * cfg.batch,
                        "blocks_per_s": 1.0 / t_req,
                        "sample": ("full round of request 0" if scale == 1 else
                                   f"projections on 1/{scale} of every matrix's rows, x{scale}")
                                  + (f", round = {cfg.batch} x request 0" if cfg.batch > 1 else "")})
    set_oracle_threads(cores)
    return {"oracle_table": out, "cores": cores, "host": platform.machine()}


def run_reference(args, cfg):
    """The CPU oracle as the reference arm, on this arm's workload and metric."""
    rank, ws, _ = dist_env()
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    os.environ.setdefault("OMP_NUM_THREADS", str(threads))
    model = syn.make_model(cfg)
    est = oracle_round_seconds(cfg, model, rounds=1)[0]
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    scale = max(1, int(np.ceil(est / per_step)))
    for _ in range(args.warmup):
        oracle_round_seconds(cfg, model, rounds=1, scale_rows=scale)
    times = []
    for _ in range(args.steps):
        times.extend(oracle_round_seconds(cfg, model, rounds=1, scale_rows=scale))
    total = sum(times)
    value = len(times) / total     # blocks of one request per second
    sample = ("one full round of request 0 per step" if scale == 1 else
              f"per step the round's projections on 1/{scale} of every matrix's rows, time x{scale}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg),
            "cpu_baseline": {"value": value, "unit": "blocks/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "draft blocks/s (4-bit 5120-wide DFlash2 drafter round: context projection + block draft + accept)"


def workload_config(cfg) -> dict:
    return {"workload": (f"{cfg.name}: L{cfg.n_layers} d{cfg.d} {cfg.n_q_heads}/{cfg.n_kv_heads}x{cfg.head_dim} "
                         f"I{cfg.inter} taps {cfg.n_taps}xH{cfg.target_hidden} V{cfg.vocab} gamma{cfg.gamma} "
                         f"window{cfg.window} ctx{cfg.ctx_len} batch{cfg.batch} weights {cfg.wdtype}"),
            "requests": cfg.batch, "gamma": cfg.gamma, "ctx_len": cfg.ctx_len, "window": cfg.window,
            "new_ctx_rows_per_round": list(cfg.appends()),
            **({"large_batch_tc05": True} if getattr(cfg, "large_batch_tc05", False) else {}),
            **({"skinny_tc05": True} if getattr(cfg, "skinny_tc05", False) else {}),
            "l2": "no flush: every round streams >1.4 GB of weights, far above the 129 MB L2"}


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="c3")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--lat-steps", type=int, default=20,
                    help="rounds timed one by one after the timed region, for the p10/p50/p90 round latency")
    ap.add_argument("--markov-rank", type=int, default=0,
                    help="add the Markov sequential head of this rank (not part of the headline workload)")
    ap.add_argument("--oracle-table", default="",
                    help="comma-separated workloads: print the oracle's 1-core / all-core round times and exit")
    ap.add_argument("--large-batch-tc05", action="store_true",
                    help="library option: draft calls of more than 32 block rows on the tcgen05 contraction")
    ap.add_argument("--rows-matmul", default="", choices=["", "lm", "ctx", "qkv", "o", "gateup", "down"],
                    help="time dflash_rows_matmul on one matrix of the 4-bit drafter instead of the round")
    ap.add_argument("--rows", default="16,32,64,160", help="activation row counts for --rows-matmul")
    ap.add_argument("--probe-rounds", type=int, default=5,
                    help="rounds per kernel class timed live after the timed region (one launch each)")
    ap.add_argument("--skinny-tc05", action="store_true",
                    help="draft calls of at most 32 block rows run their projections on the tcgen05 projection kernel")
    ap.add_argument("--profile-ctx", type=int, default=0,
                    help="prefill only this many context rows (for short profiler captures; not a bench value)")
    args = ap.parse_args()
    if args.oracle_table:
        print(json.dumps(oracle_table(tuple(args.oracle_table.split(",")))), flush=True)
        return 0
    if args.rows_matmul:
        print(json.dumps(rows_matmul_bench(args.rows_matmul, [int(v) for v in args.rows.split(",")], args.steps)),
              flush=True)
        return 0
    cfg = syn.CONFIGS[args.config]
    if args.markov_rank:
        cfg = syn.with_overrides(cfg, markov_rank=args.markov_rank)
    if args.large_batch_tc05:
        cfg = syn.with_overrides(cfg, large_batch_tc05=True)
    if args.skinny_tc05:
        cfg = syn.with_overrides(cfg, skinny_tc05=True)
    if args.impl == "reference":
        return run_reference(args, cfg)

    import torch
    import torch.distributed as dist

    import speculative_block_draft_gb300 as pkg
    from speculative_block_draft_gb300.session import Session

    rank, ws, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.build()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    # ---- drafter, context, per-step inputs resident in HBM -----------------------------------
    model = syn.make_model(cfg)
    B, G, n = cfg.batch, cfg.gamma, cfg.n_draft
    sess = Session(model, max_batch=B, ctx_capacity=(cfg.window if cfg.window else
                                                      cfg.ctx_len + 8 * (args.steps + args.warmup + args.e2e_steps + args.lat_steps + 8 * args.probe_rounds + 8)))
    h, stream = sess.h, sess.stream
    lengths = syn.ctx_lengths(cfg)
    if args.profile_ctx:
        lengths = np.minimum(lengths, args.profile_ctx)
    width = cfg.n_taps * cfg.target_hidden
    for b in range(B):
        done = 0
        while done < int(lengths[b]):
            m = min(4096, int(lengths[b]) - done)
            rows = syn.taps_rows(cfg, cfg.seed + rank, b, done, m)
            assert sess.project([b], [m], rows) == 0
            done += m
    total_steps = args.warmup + args.steps
    counts = [syn.append_counts(cfg, s) for s in range(total_steps + args.e2e_steps)]
    pos = lengths.astype(np.int64).copy()
    step_taps, step_anchor, step_target = [], [], []
    for s in range(total_steps + args.e2e_steps):
        rows = [syn.taps_rows(cfg, cfg.seed + rank, b, int(pos[b]), int(counts[s][b])) for b in range(B)]
        pos += counts[s]
        step_taps.append(np.concatenate(rows))
        step_anchor.append(syn.anchors(cfg.seed + rank, B, s, cfg.vocab))
        step_target.append(syn.tokens(cfg.seed + rank, "bench.target", B * G, cfg.vocab, offset=s * B * G)
                           .reshape(B, G))
    dev_taps = [sess.upload(t) for t in step_taps[:total_steps]]
    dev_anchor = [sess.upload(a) for a in step_anchor[:total_steps]]
    dev_target = [sess.upload(t) for t in step_target[:total_steps]]
    draft = torch.empty((B, n), dtype=torch.int32, device=dev)
    conf = torch.empty((B, n), dtype=torch.float32, device=dev)
    acc_len = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    req = list(range(B))

    def step(s, probe=None):
        c = [int(x) for x in counts[s]]
        h.project_ctx(req, c, dev_taps[s], stream=stream)
        if probe is not None:
            h.set_probe(*probe, kernel=0)
        rc = h.draft_block(req, dev_anchor[s], draft, conf, None, stream=stream)
        assert rc == 0
        h.accept(draft, dev_target[s], acc_len, nxt, stream=stream)

    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            step(s)
    stream.synchronize()
    assert h.check_errors(stream) == 0

    # ---- timed region: K rounds, inputs resident ---------------------------------------------
    probes = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in probes:           # torch creates the CUDA events on first record; the library re-records them
        a.record(stream)
        b.record(stream)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = h.launch_count()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        torch.cuda.nvtx.range_push("timed")
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(args.steps):
                step(args.warmup + i, probe=probes[i])
            ev1.record(stream)
        stream.synchronize()
        torch.cuda.nvtx.range_pop()
    barrier()
    torch.cuda.synchronize()
    launches = h.launch_count() - launches0
    elapsed = ev0.elapsed_time(ev1) / 1e3
    assert h.check_errors(stream) == 0
    lm_ms = float(np.mean([a.elapsed_time(b) for a, b in probes]))
    t_max, blocks = reduce_over_ranks(elapsed, float(B * args.steps))
    value = blocks / t_max

    # ---- every kernel class of the round timed live: events around one launch per probe round ----
    ctx_rows = float(np.mean([np.sum(counts[args.warmup + i]) for i in range(args.steps)]))
    classes = probe_classes(cfg, lengths, ctx_rows)
    class_ms = {}
    for name, kind, _, _ in classes:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.probe_rounds)]
        with torch.cuda.stream(stream):
            for j, (a0, a1) in enumerate(evs):
                a0.record(stream)   # torch creates the events on first record; the library re-records them
                a1.record(stream)
                h.set_probe(a0, a1, kernel=kind)
                step(args.warmup + j % args.steps)
        stream.synchronize()
        class_ms[name] = float(np.mean([a0.elapsed_time(a1) for a0, a1 in evs]))
    assert h.check_errors(stream) == 0

    # ---- end to end through the C ABI with host buffers --------------------------------------
    pin_taps = [torch.from_numpy(t.view(np.int16) if t.dtype == np.uint16 else t).pin_memory()
                for t in step_taps[total_steps:]]
    pin_anchor = [torch.from_numpy(a).pin_memory() for a in step_anchor[total_steps:]]
    pin_target = [torch.from_numpy(t).pin_memory() for t in step_target[total_steps:]]
    out_draft = torch.empty((B, n), dtype=torch.int32).pin_memory()
    out_len = torch.empty(B, dtype=torch.int32).pin_memory()
    out_nxt = torch.empty(B, dtype=torch.int32).pin_memory()
    d_taps = torch.empty((max(t.shape[0] for t in pin_taps), width), dtype=pin_taps[0].dtype, device=dev)
    d_anchor = torch.empty(B, dtype=torch.int32, device=dev)
    d_target = torch.empty((B, G), dtype=torch.int32, device=dev)
    h2d = d2h = 0
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.e2e_steps):
            s = total_steps + i
            nt = pin_taps[i].shape[0]
            d_taps[:nt].copy_(pin_taps[i], non_blocking=True)
            d_anchor.copy_(pin_anchor[i], non_blocking=True)
            d_target.copy_(pin_target[i], non_blocking=True)
            h.project_ctx(req, [int(x) for x in counts[s]], d_taps, stream=stream)
            assert h.draft_block(req, d_anchor, draft, conf, None, stream=stream) == 0
            h.accept(draft, d_target, acc_len, nxt, stream=stream)
            out_draft.copy_(draft, non_blocking=True)
            out_len.copy_(acc_len, non_blocking=True)
            out_nxt.copy_(nxt, non_blocking=True)
            stream.synchronize()          # the host needs the accepted length before the next round
            h2d += pin_taps[i][:nt].numel() * pin_taps[i].element_size() + 4 * B + 4 * B * G
            d2h += 4 * B * n + 8 * B
        e1.record(stream)
    stream.synchronize()
    e2e_t, e2e_blocks = reduce_over_ranks(e0.elapsed_time(e1) / 1e3, float(B * args.e2e_steps))
    e2e_value = e2e_blocks / e2e_t

    # ---- round latency distribution: rounds bracketed one by one (after the timed region, so the
    # headline is untouched; a bracketed round cannot overlap its neighbours) -------------------
    latency = None
    if args.lat_steps > 0:
        try:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.lat_steps)]
            with torch.cuda.stream(stream):
                for i, (a0, a1) in enumerate(evs):
                    a0.record(stream)
                    step(args.warmup + i % args.steps)
                    a1.record(stream)
            stream.synchronize()
            assert h.check_errors(stream) == 0
            ms = np.array([a0.elapsed_time(a1) for a0, a1 in evs])
            latency = {"rounds": int(ms.size), "p10_ms": float(np.percentile(ms, 10)),
                       "p50_ms": float(np.percentile(ms, 50)), "p90_ms": float(np.percentile(ms, 90)),
                       "how": "each round between its own CUDA events on the library's stream, after the "
                              "timed region; no overlap with neighbouring rounds"}
        except Exception as exc:   # the distribution is extra; it never costs the headline line
            latency = {"error": f"{type(exc).__name__}: {exc}"[:200]}

    if rank != 0:
        sess.close()
        if ws > 1:
            dist.destroy_process_group()
        return 0

    peaks = load_peaks()
    rb = round_bytes(cfg, lengths)
    rf = round_flops(cfg, lengths, ctx_rows)
    t_round = t_max / args.steps
    # per kernel class: live achieved GB/s against its algorithmic bytes; the roofline object is
    # the class that takes the largest share of the round (launch time x launches per round)
    class_ms["lm_head"] = lm_ms
    t_round_ms = 1e3 * t_max / args.steps
    by_kernel, roof = class_rooflines(cfg, classes, class_ms, t_round_ms, peaks, lengths, ctx_rows)
    line = {
        "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {**workload_config(cfg), **({"profile_ctx": args.profile_ctx} if args.profile_ctx else {})},
        "round_hbm": {"algorithmic_bytes": rb["total"], "breakdown_mb": {k: round(v / 1e6, 1) for k, v in rb.items()},
                      "achieved_gbs": rb["total"] / (t_max / args.steps) / 1e9,
                      "peak_gbs": peaks["hbm_gbs"],
                      "frac": rb["total"] / (t_max / args.steps) / 1e9 / peaks["hbm_gbs"],
                      "peak_source": peaks["source"]},
        "round_tensor": {"algorithmic_flop": rf["total"],
                         "breakdown_gflop": {k: round(v / 1e9, 2) for k, v in rf.items()},
                         "achieved_tflops": rf["total"] / t_round / 1e12,
                         "peak_tflops": peaks["bf16_tflops_sustained"],
                         "frac": rf["total"] / t_round / 1e12 / peaks["bf16_tflops_sustained"],
                         "peak_source": f"{peaks['source']} (cuBLAS bf16, sustained; the projections run f16 "
                                        f"operands on the same tensor-core rate)"},
        "roofline": roof,
        "roofline_by_kernel": by_kernel,
        "e2e": {"value": e2e_value, "unit": "blocks/s", "h2d_bytes_per_step": h2d // max(1, args.e2e_steps),
                "d2h_bytes_per_step": d2h // max(1, args.e2e_steps), "steps": args.e2e_steps},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    if latency is not None:
        line["round_latency"] = latency
    if not args.no_cpu_baseline and ws >= 1:
        threads = os.cpu_count() or 1
        times = oracle_round_seconds(cfg, model, rounds=2)
        cpu_v = 1.0 / (sum(times) / len(times))
        line["cpu_baseline"] = {"value": cpu_v, "unit": "blocks/s", "cores": threads, "kind": "oracle",
                                "sample": f"{len(times)} rounds of request 0 (project {cfg.appends()[0]} ctx rows, "
                                          f"draft one block over the full window, accept); window K/V drawn "
                                          f"from the generator"}
    print(json.dumps(line), flush=True)
    sess.close()
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
