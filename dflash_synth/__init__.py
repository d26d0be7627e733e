"""Seeded synthetic inputs shared by the oracle's tests, the CUDA path's tests and the bench.

Holds none of the drafter's arithmetic: it draws weights (N(0, 0.02), norm weights 1),
context taps (N(0, 1)), anchor tokens and synthetic target tokens, and packs weights into
the storage formats both sides read (fp32, bf16 bits, group-64 affine 4-bit).
The generator itself is C (``synth.c``) so multi-gigabyte drafters are drawn in seconds.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import zlib
from dataclasses import dataclass, field, replace

import numpy as np

from .configs import CONFIGS, DraftConfig  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdflash_synth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator with gcc (plain C, OpenMP; no architecture flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, i32, f32, f64 = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32,
                                   ctypes.c_float, ctypes.c_double)
        vp = ctypes.c_void_p
        lib.syn_key.restype = u64
        lib.syn_key.argtypes = [u64, u64]
        lib.syn_normal_f32.argtypes = [u64, u64, i64, f32, vp]
        lib.syn_uniform_f64.argtypes = [u64, u64, i64, vp]
        lib.syn_tokens.argtypes = [u64, u64, i64, i32, vp]
        lib.syn_to_bf16.argtypes = [vp, i64, vp]
        lib.syn_quantize_q4g64.argtypes = [vp, i64, i64, vp, vp, vp]
        lib.syn_target_tokens.argtypes = [u64, u64, i32, vp, f64, i32, vp]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def tensor_key(seed: int, name: str) -> int:
    """Stream key for a named tensor (the name is hashed with CRC-32 into a tensor id)."""
    return int(_load().syn_key(seed & (2**64 - 1), zlib.crc32(name.encode())))


def normal(seed: int, name: str, shape, std: float = 1.0, offset: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    _load().syn_normal_f32(tensor_key(seed, name), offset, n, std, _ptr(out))
    return out.reshape(shape)


def uniform(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().syn_uniform_f64(tensor_key(seed, name), offset, n, _ptr(out))
    return out


def tokens(seed: int, name: str, n: int, vocab: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().syn_tokens(tensor_key(seed, name), offset, n, vocab, _ptr(out))
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().syn_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h).astype(np.uint32) << 16).view(np.float32)


def quantize_q4g64(w: np.ndarray):
    """fp32 [rows][cols] -> (packed u32 [rows][cols/8], scale bf16-bits, bias bf16-bits)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert cols % 64 == 0, cols
    packed = np.empty((rows, cols // 8), dtype=np.uint32)
    scale = np.empty((rows, cols // 64), dtype=np.uint16)
    bias = np.empty((rows, cols // 64), dtype=np.uint16)
    _load().syn_quantize_q4g64(_ptr(w), rows, cols, _ptr(packed), _ptr(scale), _ptr(bias))
    return packed, scale, bias


def target_tokens(seed: int, req: int, round_idx: int, draft: np.ndarray, p: float, vocab: int) -> np.ndarray:
    """Synthetic target greedy tokens t[0..n] for one block of n drafts: t[k] equals draft[k]
    with probability p (independently per position), the bonus t[n] is uniform."""
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    n = draft.shape[0]
    out = np.empty(n + 1, dtype=np.int32)
    _load().syn_target_tokens(tensor_key(seed, f"target.req{req}"), round_idx * 4096, n,
                              _ptr(draft), float(p), vocab, _ptr(out))
    return out


# ----------------------------------------------------------------------------------------
# Weight containers in the storage formats both sides read.
# ----------------------------------------------------------------------------------------
@dataclass
class HostMatrix:
    """A projection matrix [n_out][n_in] in one storage format.

    fmt 'f32'  : data float32 [n_out][n_in]
    fmt 'bf16' : data uint16 (bf16 bits) [n_out][n_in]
    fmt 'q4'   : data uint32 [n_out][n_in/8] (nibble i of word j = input 8j+i), scale and
                 bias uint16 (bf16 bits) [n_out][n_in/64]; element = scale*q + bias
    """
    fmt: str
    n_out: int
    n_in: int
    data: np.ndarray
    scale: np.ndarray | None = None
    bias: np.ndarray | None = None

    def nbytes(self) -> int:
        n = self.data.nbytes
        if self.scale is not None:
            n += self.scale.nbytes + self.bias.nbytes
        return n


def make_matrix(seed: int, name: str, n_out: int, n_in: int, fmt: str, std: float = 0.02) -> HostMatrix:
    """Draw N(0, std) [n_out][n_in] in row chunks (about 32 M elements each) and store it in ``fmt``."""
    chunk_rows = max(1, (1 << 25) // n_in)
    if fmt == "f32":
        return HostMatrix(fmt, n_out, n_in, normal(seed, name, (n_out, n_in), std))
    if fmt == "bf16":
        data = np.empty((n_out, n_in), dtype=np.uint16)
        for r0 in range(0, n_out, chunk_rows):
            r1 = min(n_out, r0 + chunk_rows)
            w = normal(seed, name, (r1 - r0, n_in), std, offset=r0 * n_in)
            data[r0:r1] = to_bf16_bits(w)
        return HostMatrix(fmt, n_out, n_in, data)
    if fmt == "q4":
        packed = np.empty((n_out, n_in // 8), dtype=np.uint32)
        scale = np.empty((n_out, n_in // 64), dtype=np.uint16)
        bias = np.empty((n_out, n_in // 64), dtype=np.uint16)
        for r0 in range(0, n_out, chunk_rows):
            r1 = min(n_out, r0 + chunk_rows)
            w = normal(seed, name, (r1 - r0, n_in), std, offset=r0 * n_in)
            packed[r0:r1], scale[r0:r1], bias[r0:r1] = quantize_q4g64(w)
        return HostMatrix(fmt, n_out, n_in, packed, scale, bias)
    raise ValueError(fmt)


@dataclass
class HostModel:
    cfg: DraftConfig
    mats: dict = field(default_factory=dict)   # name -> HostMatrix
    vecs: dict = field(default_factory=dict)   # name -> float32 array

    def nbytes(self) -> int:
        return sum(m.nbytes() for m in self.mats.values()) + sum(v.nbytes for v in self.vecs.values())


def make_model(cfg: DraftConfig, seed: int | None = None, norm_jitter: float = 0.0, skip=()) -> HostModel:
    """Synthetic drafter in the spirit of the page-3 seeded init: every projection N(0, 0.02),
    mask_emb / block_pos N(0, 0.02), norm weights 1 (plus optional N(0, norm_jitter) so tests
    can tell the norms apart). Borrowed target tables ``embed`` and ``lm_head`` are drawn the
    same way. Names not wanted can be listed in ``skip``."""
    c = cfg
    seed = c.seed if seed is None else seed
    m = HostModel(cfg)
    fmt = c.wdtype
    qd, kvd = c.n_q_heads * c.head_dim, c.n_kv_heads * c.head_dim

    def mat(name, n_out, n_in):
        if name not in skip:
            m.mats[name] = make_matrix(seed, name, n_out, n_in, fmt)

    def norm_vec(name):
        v = np.ones(c.d, dtype=np.float32)
        if norm_jitter:
            v = v + normal(seed, name, (c.d,), norm_jitter)
        m.vecs[name] = v.astype(np.float32)

    for i in range(c.n_layers):
        norm_vec(f"bb.{i}.attn_norm")
        mat(f"bb.{i}.q", qd, c.d)
        mat(f"bb.{i}.k", kvd, c.d)
        mat(f"bb.{i}.v", kvd, c.d)
        mat(f"bb.{i}.o", c.d, qd)
        norm_vec(f"bb.{i}.ff_norm")
        mat(f"bb.{i}.gate", c.inter, c.d)
        mat(f"bb.{i}.up", c.inter, c.d)
        mat(f"bb.{i}.down", c.d, c.inter)
    mat("W_c", c.d, c.n_taps * c.target_hidden)
    norm_vec("ctx_norm")
    if c.d != c.target_hidden:
        mat("tok_proj", c.d, c.target_hidden)
        mat("out_proj", c.target_hidden, c.d)
    # drawn at a fixed 32 rows so a smaller gamma sees a prefix of the same rows
    m.vecs["mask_emb"] = np.ascontiguousarray(normal(seed, "mask_emb", (32, c.d), 0.02)[: c.gamma - 1])
    m.vecs["block_pos"] = np.ascontiguousarray(normal(seed, "block_pos", (32, c.d), 0.02)[: c.gamma])
    norm_vec("out_norm")
    mat("embed", c.vocab, c.target_hidden)
    mat("lm_head", c.vocab, c.target_hidden)
    if c.markov_rank:
        # Markov sequential head: W1 [V][r] N(0, 0.02) as on the page; W2 (stored transposed,
        # [V][r]) drawn N(0, 0.5) instead of the page's zero init, so the bias moves the drafts
        if "markov.w1" not in skip:
            m.mats["markov.w1"] = make_matrix(seed, "markov.w1", c.vocab, c.markov_rank, fmt)
        if "markov.w2t" not in skip:
            m.mats["markov.w2t"] = make_matrix(seed, "markov.w2t", c.vocab, c.markov_rank, fmt, std=0.5)
    return m


def taps_rows(cfg: DraftConfig, seed: int, req: int, pos0: int, n: int) -> np.ndarray:
    """Context taps for positions [pos0, pos0+n) of request ``req``: [n][n_taps*H] N(0,1),
    fp32 or bf16 bits per the config's activation type. Row p is the same whatever chunk it
    is drawn in."""
    width = cfg.n_taps * cfg.target_hidden
    x = normal(seed, f"taps.req{req}", (n, width), 1.0, offset=pos0 * width)
    return x if cfg.adtype == "f32" else to_bf16_bits(x)


def taps_to_f32(cfg: DraftConfig, taps: np.ndarray) -> np.ndarray:
    return taps if cfg.adtype == "f32" else bf16_bits_to_f32(taps)


def anchors(seed: int, n_req: int, round_idx: int, vocab: int) -> np.ndarray:
    return np.array([tokens(seed, f"anchor.req{b}", 1, vocab, offset=round_idx)[0] for b in range(n_req)],
                    dtype=np.int32)


def ctx_lengths(cfg: DraftConfig) -> np.ndarray:
    """Committed context length per request: fixed, or uniform in [ctx_min, ctx_len]."""
    if not cfg.ctx_min:
        return np.full(cfg.batch, cfg.ctx_len, dtype=np.int64)
    u = uniform(cfg.seed, "ctx_len", cfg.batch)
    return (cfg.ctx_min + np.floor(u * (cfg.ctx_len - cfg.ctx_min + 1))).astype(np.int64)


def append_counts(cfg: DraftConfig, round_idx: int) -> np.ndarray:
    """New context rows per request for one round: fixed, or uniform in {append_min..append_max}."""
    lo, hi = cfg.appends()
    if lo == hi:
        return np.full(cfg.batch, lo, dtype=np.int64)
    u = uniform(cfg.seed, "append", cfg.batch, offset=round_idx * cfg.batch)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)


def with_overrides(cfg: DraftConfig, **kw) -> DraftConfig:
    return replace(cfg, **kw)
