"""CPU oracle for one DFlash drafting round -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``dflash_oracle.c`` (plain C, fp64). This module compiles it with gcc and
marshals numpy arrays in and out. Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's
CPU-baseline arm may import it; the CUDA library never links, calls or imports anything here.

Pinned functions: dequantisation, RMSNorm, attention (torch SDPA), SiLU (torch), acceptance
(exhaustive brute force and the page-1 worked examples), argmax/confidence (closed forms),
context projection (one-hot taps), block construction + output head (identity layers),
the key set and GQA map (uniform attention), non-causality. The end-to-end logits of a full
random drafter are pinned only through those pieces: the pages print no forward-pass values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dflash_oracle.c")
_HDR = os.path.join(_HERE, "dflash_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdflash_oracle.so")
_lib = None

F32, BF16, Q4G64 = 0, 1, 2
_FMT = {"f32": F32, "bf16": BF16, "q4": Q4G64}
MAX_LAYERS = 16


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, OpenMP over independent outputs, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "d", "n_q_heads", "n_kv_heads", "head_dim", "inter",
                                             "n_taps", "target_hidden", "vocab", "gamma", "window")] + \
               [("eps", ctypes.c_double), ("causal", ctypes.c_int), ("ffn_act", ctypes.c_int),
                ("draft_all_rows", ctypes.c_int)]


class Mat(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("n_out", ctypes.c_int), ("n_in", ctypes.c_int),
                ("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class Layer(ctypes.Structure):
    _fields_ = [(n, Mat) for n in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")] + \
               [("attn_norm", ctypes.c_void_p), ("ff_norm", ctypes.c_void_p)]


class Weights(ctypes.Structure):
    _fields_ = [(n, Mat) for n in ("w_c", "tok_proj", "out_proj", "embed", "lm_head")] + \
               [(n, ctypes.c_void_p) for n in ("ctx_norm", "mask_emb", "block_pos", "out_norm")] + \
               [("layer", Layer * MAX_LAYERS)]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.orc_weight.restype = f64
        lib.orc_weight.argtypes = [ctypes.POINTER(Mat), i32, i32]
        lib.orc_linear.argtypes = [ctypes.POINTER(Mat), i32, vp, vp]
        lib.orc_rmsnorm.argtypes = [vp, vp, i32, f64, vp]
        lib.orc_silu.restype = f64
        lib.orc_silu.argtypes = [f64]
        lib.orc_attention.argtypes = [i32, i32, i32, i32, vp, i32, vp, vp, i32, vp]
        lib.orc_ctx_rows.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Weights), i32, vp, vp, vp]
        lib.orc_draft.restype = i32
        lib.orc_draft.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Weights), i32, i32, vp, vp,
                                  vp, vp, vp, vp, vp]
        lib.orc_argmax_conf.argtypes = [vp, i32, vp, vp, vp]
        lib.orc_accept.restype = i32
        lib.orc_accept.argtypes = [i32, vp, vp, vp]
        lib.orc_markov.restype = None
        lib.orc_markov.argtypes = [ctypes.POINTER(Mat), ctypes.POINTER(Mat), i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.orc_gelu_tanh.restype = ctypes.c_double
        lib.orc_gelu_tanh.argtypes = [ctypes.c_double]
        lib.orc_draft_length.restype = i32
        lib.orc_draft_length.argtypes = [i32, vp, vp, ctypes.c_float]
        lib.orc_accept_kept.restype = i32
        lib.orc_accept_kept.argtypes = [i32, i32, vp, vp, vp]
        _lib = lib
    return _lib


def _p(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _mat(hm) -> Mat:
    if hm is None:
        return Mat(0, 0, 0, None, None, None)
    return Mat(_FMT[hm.fmt], hm.n_out, hm.n_in, _p(hm.data), _p(hm.scale), _p(hm.bias))


# ---------------------------------------------------------------------------------------------
# small pieces (exposed for the pins)
# ---------------------------------------------------------------------------------------------
def weight(hm, n: int, k: int) -> float:
    m = _mat(hm)
    return _load().orc_weight(ctypes.byref(m), n, k)


def dense(hm) -> np.ndarray:
    """The whole matrix dequantised (small matrices only)."""
    x = np.eye(hm.n_in, dtype=np.float64)
    return linear(hm, x).T.copy()


def linear(hm, x: np.ndarray) -> np.ndarray:
    x = _f64(x)
    rows = x.shape[0]
    y = np.empty((rows, hm.n_out), dtype=np.float64)
    m = _mat(hm)
    _load().orc_linear(ctypes.byref(m), rows, _p(x), _p(y))
    return y


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = _f64(x)
    w = np.ascontiguousarray(w, dtype=np.float32)
    y = np.empty_like(x)
    _load().orc_rmsnorm(_p(x), _p(w), x.shape[-1], eps, _p(y))
    return y


def silu(x: float) -> float:
    return _load().orc_silu(float(x))


def gelu_tanh(x):
    """GELU in its tanh approximation, elementwise, fp64."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    return np.array([_load().orc_gelu_tanh(float(v)) for v in a.ravel()]).reshape(a.shape)


def attention(q, k, v, n_q_heads: int, n_kv_heads: int, head_dim: int, causal_block_start: int = -1):
    q, k, v = _f64(q), _f64(k), _f64(v)
    out = np.empty_like(q)
    _load().orc_attention(q.shape[0], n_q_heads, n_kv_heads, head_dim, _p(q), k.shape[0], _p(k), _p(v),
                          causal_block_start, _p(out))
    return out


def argmax_conf(logits: np.ndarray):
    logits = _f64(logits)
    tok, conf, margin = ctypes.c_int(), ctypes.c_double(), ctypes.c_double()
    _load().orc_argmax_conf(_p(logits), logits.shape[0], ctypes.byref(tok), ctypes.byref(conf),
                            ctypes.byref(margin))
    return tok.value, conf.value, margin.value


def accept(draft, target):
    """(accepted length a, next anchor target[a]) for drafts d[0..n-1] and target t[0..n]."""
    d = np.ascontiguousarray(draft, dtype=np.int32)
    t = np.ascontiguousarray(target, dtype=np.int32)
    assert t.shape[0] == d.shape[0] + 1
    nxt = ctypes.c_int()
    a = _load().orc_accept(d.shape[0], _p(d), _p(t), ctypes.byref(nxt))
    return a, nxt.value


def draft_length(conf, thresholds=None, min_conf=0.0):
    """Drafts kept by confidence-scheduled pruning (position 0 always; the first k >= 1 with
    conf[k] < threshold ends the block). conf and thresholds are fp32, as the library takes them."""
    c = np.ascontiguousarray(conf, dtype=np.float32)
    th = None if thresholds is None else np.ascontiguousarray(thresholds, dtype=np.float32)
    return _load().orc_draft_length(c.shape[0], _p(c), _p(th) if th is not None else None, float(min_conf))


def accept_kept(draft, target, keep):
    """(accepted length, next anchor) when only the first `keep` drafts are verified."""
    d = np.ascontiguousarray(draft, dtype=np.int32)
    t = np.ascontiguousarray(target, dtype=np.int32)
    assert t.shape[0] == d.shape[0] + 1
    nxt = ctypes.c_int()
    a = _load().orc_accept_kept(d.shape[0], int(keep), _p(d), _p(t), ctypes.byref(nxt))
    return a, nxt.value


# ---------------------------------------------------------------------------------------------
# the drafter
# ---------------------------------------------------------------------------------------------
class Oracle:
    """Holds ctypes views of a HostModel (dflash_synth) and runs the oracle on it."""

    def __init__(self, model, causal: bool = False):
        c = model.cfg
        assert c.n_layers <= MAX_LAYERS
        self.cfg = c
        self.model = model
        self._vecs = {k: np.ascontiguousarray(v, dtype=np.float32) for k, v in model.vecs.items()}
        self.c = Cfg(c.n_layers, c.d, c.n_q_heads, c.n_kv_heads, c.head_dim, c.inter, c.n_taps,
                     c.target_hidden, c.vocab, c.gamma, c.window, c.eps, 1 if causal else 0,
                     1 if getattr(c, "ffn", "swiglu") == "gelu" else 0, 1 if getattr(c, "draft_all_rows", False) else 0)
        w = Weights()
        mats = model.mats
        w.w_c = _mat(mats["W_c"])
        w.tok_proj = _mat(mats.get("tok_proj"))
        w.out_proj = _mat(mats.get("out_proj"))
        w.embed = _mat(mats["embed"])
        w.lm_head = _mat(mats["lm_head"])
        w.ctx_norm = _p(self._vecs["ctx_norm"])
        w.mask_emb = _p(self._vecs["mask_emb"]) if self._vecs["mask_emb"].size else None
        w.block_pos = _p(self._vecs["block_pos"])
        w.out_norm = _p(self._vecs["out_norm"])
        for i in range(c.n_layers):
            L = w.layer[i]
            L.wq, L.wk, L.wv, L.wo = (_mat(mats[f"bb.{i}.{n}"]) for n in ("q", "k", "v", "o"))
            L.w_gate, L.w_up, L.w_down = (_mat(mats[f"bb.{i}.{n}"]) for n in ("gate", "up", "down"))
            L.attn_norm = _p(self._vecs[f"bb.{i}.attn_norm"])
            L.ff_norm = _p(self._vecs[f"bb.{i}.ff_norm"])
        self.w = w

    def markov(self, anchor: int, base_logits: np.ndarray, prev_tokens=None):
        """The Markov head's serial drafts over base logits [n][V]; prev_tokens (n ints) fixes the
        chain's previous tokens after the first (used to follow another implementation's chain)."""
        c = self.cfg
        n, V = base_logits.shape
        m1, m2 = _mat(self.model.mats["markov.w1"]), _mat(self.model.mats["markov.w2t"])
        logits = np.empty((n, V), dtype=np.float64)
        toks = np.empty(n, dtype=np.int32)
        conf = np.empty(n, dtype=np.float64)
        margin = np.empty(n, dtype=np.float64)
        prev = None if prev_tokens is None else np.ascontiguousarray(prev_tokens, dtype=np.int32)
        base = np.ascontiguousarray(base_logits, dtype=np.float64)
        _load().orc_markov(ctypes.byref(m1), ctypes.byref(m2), c.markov_rank, V, n, int(anchor), _p(base),
                           _p(prev) if prev is not None else None, _p(logits), _p(toks), _p(conf), _p(margin))
        return {"logits": logits, "tokens": toks, "conf": conf, "margin": margin}

    @property
    def kvd(self) -> int:
        return self.cfg.n_kv_heads * self.cfg.head_dim

    def ctx_rows(self, taps_f64: np.ndarray):
        """Per-layer context K/V rows [L][rows][Hkv*hd] for taps rows [rows][m*H]."""
        taps = _f64(taps_f64)
        rows = taps.shape[0]
        L = self.cfg.n_layers
        k = np.empty((L, rows, self.kvd), dtype=np.float64)
        v = np.empty_like(k)
        if rows:
            _load().orc_ctx_rows(ctypes.byref(self.c), ctypes.byref(self.w), rows, _p(taps), _p(k), _p(v))
        return k, v

    def draft(self, anchor: int, k_ctx: np.ndarray, v_ctx: np.ndarray, trace: bool = False, prev_tokens=None):
        """One block: logits [n_draft][V], tokens, conf, margin (top1 - top2), optional trace."""
        c = self.cfg
        n_ctx = k_ctx.shape[1]
        k_ctx, v_ctx = _f64(k_ctx), _f64(v_ctx)
        n = c.n_draft
        logits = np.empty((n, c.vocab), dtype=np.float64)
        toks = np.empty(n, dtype=np.int32)
        conf = np.empty(n, dtype=np.float64)
        margin = np.empty(n, dtype=np.float64)
        tr = np.empty((c.n_layers + 1, c.gamma, c.d), dtype=np.float64) if trace else None
        rc = _load().orc_draft(ctypes.byref(self.c), ctypes.byref(self.w), int(anchor), n_ctx,
                               _p(k_ctx), _p(v_ctx), _p(logits), _p(toks), _p(conf), _p(margin), _p(tr))
        if rc != 0:
            raise ValueError(f"orc_draft rejected its inputs (rc={rc})")
        out = {"logits": logits, "tokens": toks, "conf": conf, "margin": margin}
        if getattr(c, "markov_rank", 0):
            out = dict(self.markov(anchor, logits, prev_tokens), base_logits=logits)
        if trace:
            out["trace"] = tr
        return out


class OracleSession:
    """Per-request context K/V as the oracle computes it (fp64), for multi-round tests.

    ``skip(req, n)`` advances a request's position count without rows; it is valid only when the
    skipped positions fall outside the sliding window of every later draft (they then never
    enter the attention), which ``draft`` checks.
    """

    def __init__(self, oracle: Oracle):
        self.o = oracle
        L, kvd = oracle.cfg.n_layers, oracle.kvd
        self._empty = np.zeros((L, 0, kvd), dtype=np.float64)
        self.k, self.v, self.n_pos, self.first = {}, {}, {}, {}

    def skip(self, req: int, n: int):
        assert self.k.get(req, self._empty).shape[1] == 0, "skip only before the first stored row"
        self.n_pos[req] = self.n_pos.get(req, 0) + n
        self.first[req] = self.n_pos[req]

    def project(self, req: int, taps_f64: np.ndarray):
        k, v = self.o.ctx_rows(taps_f64)
        self.k[req] = np.concatenate([self.k.get(req, self._empty), k], axis=1)
        self.v[req] = np.concatenate([self.v.get(req, self._empty), v], axis=1)
        self.n_pos[req] = self.n_pos.get(req, 0) + k.shape[1]
        self.first.setdefault(req, 0)
        c = self.o.cfg
        if c.window > 0 and self.k[req].shape[1] > c.window:   # rows outside any later window
            self.k[req] = np.ascontiguousarray(self.k[req][:, -c.window:])
            self.v[req] = np.ascontiguousarray(self.v[req][:, -c.window:])
            self.first[req] = max(self.first[req], 1)

    def draft(self, req: int, anchor: int, trace: bool = False, prev_tokens=None):
        c = self.o.cfg
        n_pos = self.n_pos.get(req, 0)
        k = self.k.get(req, self._empty)
        v = self.v.get(req, self._empty)
        if self.first.get(req, 0):
            assert c.window > 0 and k.shape[1] >= min(c.window, n_pos), "skipped rows would enter the window"
        if c.window > 0 and k.shape[1] > c.window:
            k, v = k[:, -c.window:], v[:, -c.window:]
        return self.o.draft(anchor, np.ascontiguousarray(k), np.ascontiguousarray(v), trace=trace,
                            prev_tokens=prev_tokens)
