"""The five synthetic workloads of the DFlash drafter round, as plain data.

Shapes come from the page-1 DFlash2 geometry ("Inco Hacks Native: DFlash 2 Speculation",
section 1: 5 layers, taps [5,19,33,47,61], hidden 5120, intermediate 17408, head_dim 128,
block 8, 4-bit) and from the page-3 ``DEFAULT_DFLASH_CONFIG`` (gamma 5, dDraft 1024,
5 layers, 8 heads, ffMult 2, 4 taps).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class DraftConfig:
    name: str
    n_layers: int
    d: int                # draft width
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    inter: int            # SwiGLU inner width
    n_taps: int           # m tapped target layers
    target_hidden: int    # H
    vocab: int            # V
    gamma: int            # block size; gamma-1 drafts per block
    window: int           # sliding window over context rows (0 = full context)
    ctx_len: int          # committed context length P before the first round
    batch: int = 1
    wdtype: str = "bf16"  # 'f32' | 'bf16' | 'q4'  (storage of every projection matrix)
    adtype: str = "bf16"  # 'f32' | 'bf16'        (taps, context K/V cache, activations)
    eps: float = 1e-6
    agree: float | None = None    # synthetic target agreement rate (None: uniform tokens)
    ffn: str = "swiglu"           # gated FFN: "swiglu" silu(g)*u, or "gelu" (tanh-form GELU)*u
    draft_all_rows: bool = False  # draft from all gamma block rows (gamma tokens), not rows 1..gamma-1
    markov_rank: int = 0          # Markov sequential head rank r (0: none), a multiple of 64
    large_batch_tc05: bool = False  # many-row draft calls on the tcgen05 contraction (library option)
    skinny_tc05: bool = False     # draft calls of <= 32 rows on the tcgen05 projection kernel (library option)
    append_min: int = 0           # new context rows per request per round (0,0: gamma rows)
    append_max: int = 0
    ctx_min: int = 0              # ragged contexts: P uniform in [ctx_min, ctx_len] (0: fixed)
    seed: int = 20261202

    @property
    def n_draft(self) -> int:
        return self.gamma if self.draft_all_rows else self.gamma - 1

    def appends(self) -> tuple[int, int]:
        if self.append_max:
            return self.append_min, self.append_max
        return self.gamma, self.gamma


C1 = DraftConfig("c1_tiny_f32", n_layers=2, d=256, n_q_heads=4, n_kv_heads=4, head_dim=64, inter=512,
                 n_taps=2, target_hidden=512, vocab=4096, gamma=4, window=0, ctx_len=64,
                 wdtype="f32", adtype="f32", seed=20261203)
C2 = DraftConfig("c2_p3default_bf16", n_layers=5, d=1024, n_q_heads=8, n_kv_heads=8, head_dim=128,
                 inter=2048, n_taps=4, target_hidden=2560, vocab=32768, gamma=5, window=0, ctx_len=1024,
                 wdtype="bf16", adtype="bf16", seed=20261204)
C3 = DraftConfig("c3_dflash2_q4_5120", n_layers=5, d=5120, n_q_heads=40, n_kv_heads=8, head_dim=128,
                 inter=17408, n_taps=5, target_hidden=5120, vocab=151936, gamma=8, window=2048,
                 ctx_len=4096, wdtype="q4", adtype="bf16", seed=20261205)


def c4_point(gamma: int, head_dim: int, window: int = 2048) -> DraftConfig:
    """Block/head sweep on the config-3 weights: width 5120 kept, heads rescaled."""
    hq, hkv = (40, 8) if head_dim == 128 else (20, 4)
    return DraftConfig(f"c4_g{gamma}_hd{head_dim}_w{window}", n_layers=5, d=5120, n_q_heads=hq,
                       n_kv_heads=hkv, head_dim=head_dim, inter=17408, n_taps=5, target_hidden=5120,
                       vocab=151936, gamma=gamma, window=window, ctx_len=8192, wdtype="q4",
                       adtype="bf16", agree=0.7, seed=C3.seed)


C4 = [c4_point(g, hd) for g in (4, 5, 8) for hd in (128, 256)] + [c4_point(8, 128, window=0)]

C5 = DraftConfig("c5_batched_32x_g5", n_layers=5, d=5120, n_q_heads=40, n_kv_heads=8, head_dim=128,
                 inter=17408, n_taps=5, target_hidden=5120, vocab=151936, gamma=5, window=2048,
                 ctx_len=16384, ctx_min=512, batch=32, wdtype="q4", adtype="bf16", agree=0.6,
                 append_min=1, append_max=8, seed=C3.seed)

CONFIGS = {"c1": C1, "c2": C2, "c3": C3, "c5": C5}
for _c in C4:
    CONFIGS[_c.name] = _c
