"""Python binding of the GB300 DFlash draft-round library (include/dflash.h).

Argument marshalling only: every step of the round runs in the CUDA kernels of ``libdflash.so``
(built in-tree from ``csrc/`` for sm_103a). PyTorch provides device memory and streams. There is
no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(os.path.dirname(_HERE), "include")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "libdflash.so")
# Debug build (DFLASH_DEBUG_CHECKS=1 in the environment selects it): the same kernels compiled with
# device bounds checks that report through dflash_check_errors (DFLASH_EBOUNDS) instead of silently
# clamping or skipping; a stand-in for a memory checker.
_BUILD_DEBUG = os.path.join(_HERE, "_build_debug")
LIB_PATH_DEBUG = os.path.join(_BUILD_DEBUG, "libdflash.so")


def _debug_selected() -> bool:
    return os.environ.get("DFLASH_DEBUG_CHECKS") == "1"
_SOURCES = ["abi.cu", "gemv_q4.cu", "gemv_bf16.cu", "gemv_f32.cu", "attn.cu", "misc.cu", "noalloc.cu", "gemm_tc05.cu", "tc05_epi.cu",
            "proj_tc05.cu"]
_HEADERS = ["internal.h", "common.cuh", "gemv_impl.cuh", "gemm_tc05.h", "tc05.cuh"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-gencode", "arch=compute_103a,code=sm_103a",
              "-Xcompiler", "-fPIC"]

DFLASH_OK, DFLASH_DECLINED, DFLASH_EINVAL, DFLASH_ECAPACITY, DFLASH_ECUDA, DFLASH_ETIMEOUT = 0, 1, -1, -2, -3, -4
DFLASH_EBOUNDS = -5
DFLASH_F32, DFLASH_BF16, DFLASH_Q4G64 = 0, 1, 2
DFLASH_MAX_LAYERS = 8
DFLASH_MAX_BATCH = 64
DFLASH_NOALLOC_MAX_ROWS = 64
DTYPE = {"f32": DFLASH_F32, "bf16": DFLASH_BF16, "q4": DFLASH_Q4G64}


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    """Compile csrc/*.cu for sm_103a (one -gencode) into _build/libdflash.so, in parallel; with
    debug (default: DFLASH_DEBUG_CHECKS=1 in the environment) the bounds-checking build into
    _build_debug/libdflash.so."""
    if debug is None:
        debug = _debug_selected()
    out_dir, lib_path = (_BUILD_DEBUG, LIB_PATH_DEBUG) if debug else (_BUILD, LIB_PATH)
    flags = NVCC_FLAGS + (["-DDFL_DEBUG_CHECKS"] if debug else [])
    os.makedirs(out_dir, exist_ok=True)
    deps = [os.path.join(_CSRC, f) for f in _SOURCES + _HEADERS] + [os.path.join(_INCLUDE, "dflash.h")]
    newest = max(os.path.getmtime(p) for p in deps)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= newest:
        return lib_path
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(_CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(_SOURCES)) as ex:
        objs = list(ex.map(compile_one, _SOURCES))
    tmp = lib_path + f".{os.getpid()}.tmp"
    r = subprocess.run([nvcc, "-shared", "-cudart", "shared", *objs, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


# ---------------------------------------------------------------------------------------------
# ctypes mirrors of include/dflash.h
# ---------------------------------------------------------------------------------------------
class dflash_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "d", "n_q_heads", "n_kv_heads", "head_dim", "inter", "n_taps", "target_hidden", "vocab",
        "gamma", "window", "max_batch", "ctx_capacity")] + \
        [("eps", ctypes.c_float), ("wdtype", ctypes.c_int), ("adtype", ctypes.c_int), ("ffn_act", ctypes.c_int),
         ("draft_all_rows", ctypes.c_int), ("markov_rank", ctypes.c_int), ("large_batch_tc05", ctypes.c_int),
         ("skinny_tc05", ctypes.c_int)]


class dflash_matrix(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class dflash_layer_weights(ctypes.Structure):
    _fields_ = [(n, dflash_matrix) for n in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")] + \
               [("attn_norm", ctypes.c_void_p), ("ff_norm", ctypes.c_void_p)]


class dflash_weights(ctypes.Structure):
    _fields_ = [(n, dflash_matrix) for n in ("w_c", "tok_proj", "out_proj", "embed", "lm_head")] + \
               [(n, ctypes.c_void_p) for n in ("ctx_norm", "mask_emb", "block_pos", "out_norm")] + \
               [("layer", dflash_layer_weights * DFLASH_MAX_LAYERS)] + \
               [(n, dflash_matrix) for n in ("markov_w1", "markov_w2t")]


class dflash_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("rounds", "blocks", "declined", "ctx_rows", "accept_calls")]


class dflash_rows_plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_pad", "m_tiles", "k_slices", "groups_per_slice", "grid",
                                            "x_stages", "tile_groups", "tiles_big", "big_groups", "tiles_small",
                                            "w_stages", "w_groups", "a_stages", "x_groups")] + [("smem_bytes", ctypes.c_size_t),
                                                            ("scratch_bytes", ctypes.c_size_t)]


DFLASH_ROWS_MATMUL_MAX = 160
DFLASH_MAT_CTX, DFLASH_MAT_QKV, DFLASH_MAT_O, DFLASH_MAT_GATEUP, DFLASH_MAT_DOWN, DFLASH_MAT_LM = range(6)


_lib = None
SYMBOLS = ["dflash_workspace_bytes", "dflash_create", "dflash_project_ctx", "dflash_draft_block",
           "dflash_accept", "dflash_reset_request", "dflash_ctx_len", "dflash_check_errors",
           "dflash_get_stats", "dflash_set_probe", "dflash_launch_count", "dflash_destroy",
           "dflash_status_str", "dflash_greedy_from_logits_noalloc", "dflash_draft_lengths",
           "dflash_accept_kept", "dflash_rows_matmul_plan", "dflash_rows_matmul", "dflash_set_wait_limit",
           "dflash_debug_stall", "dflash_accept_histogram"]


def lib():
    """Load libdflash.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = LIB_PATH_DEBUG if _debug_selected() else LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"libdflash.so is not built ({path}); run speculative_block_draft_gb300.build()")
        L = ctypes.CDLL(path)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        P = ctypes.POINTER
        L.dflash_workspace_bytes.restype = ctypes.c_size_t
        L.dflash_workspace_bytes.argtypes = [P(dflash_config)]
        L.dflash_create.restype = i32
        L.dflash_create.argtypes = [P(dflash_config), P(dflash_weights), vp, ctypes.c_size_t, vp, P(vp)]
        L.dflash_project_ctx.restype = i32
        L.dflash_project_ctx.argtypes = [vp, i32, vp, vp, vp, vp]
        L.dflash_draft_block.restype = i32
        L.dflash_draft_block.argtypes = [vp, i32, vp, vp, f32, vp, vp, vp, vp]
        L.dflash_accept.restype = i32
        L.dflash_accept.argtypes = [vp, i32, vp, vp, vp, vp, vp]
        L.dflash_reset_request.restype = i32
        L.dflash_reset_request.argtypes = [vp, i32]
        L.dflash_ctx_len.restype = ctypes.c_int64
        L.dflash_ctx_len.argtypes = [vp, i32]
        L.dflash_check_errors.restype = i32
        L.dflash_check_errors.argtypes = [vp, vp]
        L.dflash_get_stats.restype = i32
        L.dflash_get_stats.argtypes = [vp, P(dflash_stats)]
        L.dflash_set_probe.restype = i32
        L.dflash_set_probe.argtypes = [vp, i32, vp, vp]
        L.dflash_launch_count.restype = ctypes.c_uint64
        L.dflash_launch_count.argtypes = [vp]
        L.dflash_destroy.restype = None
        L.dflash_destroy.argtypes = [vp]
        L.dflash_status_str.restype = ctypes.c_char_p
        L.dflash_status_str.argtypes = [i32]
        L.dflash_greedy_from_logits_noalloc.restype = i32
        L.dflash_greedy_from_logits_noalloc.argtypes = [vp, i32, i32, vp, vp, vp]
        L.dflash_draft_lengths.restype = i32
        L.dflash_draft_lengths.argtypes = [vp, i32, vp, vp, f32, vp, vp]
        L.dflash_accept_kept.restype = i32
        L.dflash_accept_kept.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
        L.dflash_rows_matmul_plan.restype = i32
        L.dflash_rows_matmul_plan.argtypes = [i32, i32, i32, i32, i32, P(dflash_rows_plan)]
        L.dflash_rows_matmul.restype = i32
        L.dflash_rows_matmul.argtypes = [vp, i32, i32, i32, vp, vp, i32, vp, i32, vp, ctypes.c_size_t, vp]
        L.dflash_set_wait_limit.restype = i32
        L.dflash_set_wait_limit.argtypes = [vp, ctypes.c_uint, vp]
        L.dflash_debug_stall.restype = i32
        L.dflash_debug_stall.argtypes = [vp, i32]
        L.dflash_accept_histogram.restype = i32
        L.dflash_accept_histogram.argtypes = [vp, P(ctypes.c_uint64), i32, vp]
        _lib = L
    return _lib


def greedy_from_logits_noalloc(logits, token, conf=None, stream=None) -> int:
    """dflash_greedy_from_logits_noalloc on device tensors: logits fp32 [rows][vocab] ->
    token int32 [rows], conf fp32 [rows] (optional). Allocates nothing on the device."""
    rows, vocab = logits.shape
    return _check(lib().dflash_greedy_from_logits_noalloc(logits.data_ptr(), rows, vocab, token.data_ptr(),
                                                          conf.data_ptr() if conf is not None else None,
                                                          _stream_ptr(stream)), "dflash_greedy_from_logits_noalloc")


def rows_matmul_plan(n_out: int, k_in: int, n_rows: int, x_lo: bool, n_sm: int) -> dflash_rows_plan:
    """dflash_rows_matmul_plan: launch geometry and scratch of a many-row contraction (host only)."""
    p = dflash_rows_plan()
    _check(lib().dflash_rows_matmul_plan(n_out, k_in, n_rows, int(bool(x_lo)), n_sm, ctypes.byref(p)),
           "dflash_rows_matmul_plan")
    return p


class DFlashError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib().dflash_status_str(status).decode()} ({status})")


def _check(status: int, what: str) -> int:
    if status < 0:
        raise DFlashError(status, what)
    return status


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _int_array(xs):
    arr = (ctypes.c_int32 * len(xs))(*[int(x) for x in xs])
    return arr


FFN = {"swiglu": 0, "gelu": 1}


def make_config(cfg, max_batch: int | None = None, ctx_capacity: int | None = None) -> dflash_config:
    """dflash_config for a dflash_synth.DraftConfig."""
    mb = max_batch or cfg.batch
    if ctx_capacity is None:
        ctx_capacity = cfg.window if cfg.window > 0 else cfg.ctx_len + 64 * cfg.gamma
    return dflash_config(cfg.n_layers, cfg.d, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.inter, cfg.n_taps,
                         cfg.target_hidden, cfg.vocab, cfg.gamma, cfg.window, mb, ctx_capacity, cfg.eps,
                         DTYPE[cfg.wdtype], DTYPE[cfg.adtype], FFN[cfg.ffn], 1 if cfg.draft_all_rows else 0,
                         cfg.markov_rank, 1 if getattr(cfg, "large_batch_tc05", False) else 0,
                         1 if getattr(cfg, "skinny_tc05", False) else 0)


class DeviceModel:
    """A dflash_synth.HostModel uploaded to device tensors, plus the dflash_weights pointing at them."""

    def __init__(self, host_model, device="cuda"):
        import torch
        self.cfg = host_model.cfg
        self.tensors = {}

        def t(name, a):
            x = torch.from_numpy(a).to(device)
            self.tensors.setdefault(name, []).append(x)
            return x.data_ptr()

        def m(name):
            hm = host_model.mats.get(name)
            if hm is None:
                return dflash_matrix(None, None, None)
            view = {"uint32": "int32", "uint16": "int16"}.get(hm.data.dtype.name)
            data = hm.data.view(view) if view else hm.data
            if hm.scale is None:
                return dflash_matrix(t(name, data), None, None)
            return dflash_matrix(t(name, data), t(name, hm.scale.view("int16")), t(name, hm.bias.view("int16")))

        w = dflash_weights()
        w.w_c, w.tok_proj, w.out_proj = m("W_c"), m("tok_proj"), m("out_proj")
        w.embed, w.lm_head = m("embed"), m("lm_head")
        w.markov_w1, w.markov_w2t = m("markov.w1"), m("markov.w2t")
        v = host_model.vecs
        w.ctx_norm, w.block_pos, w.out_norm = t("ctx_norm", v["ctx_norm"]), t("block_pos", v["block_pos"]), \
            t("out_norm", v["out_norm"])
        w.mask_emb = t("mask_emb", v["mask_emb"]) if v["mask_emb"].size else None
        for i in range(self.cfg.n_layers):
            L = w.layer[i]
            L.wq, L.wk, L.wv, L.wo = (m(f"bb.{i}.{n}") for n in ("q", "k", "v", "o"))
            L.w_gate, L.w_up, L.w_down = (m(f"bb.{i}.{n}") for n in ("gate", "up", "down"))
            L.attn_norm = t(f"bb.{i}.attn_norm", v[f"bb.{i}.attn_norm"])
            L.ff_norm = t(f"bb.{i}.ff_norm", v[f"bb.{i}.ff_norm"])
        self.weights = w

    def free(self, keep=("embed", "markov.w1")):
        """Drop the device copies the handle no longer needs after dflash_create (the embedding
        table and the Markov head's W1 are borrowed by the handle and must be kept)."""
        self.tensors = {k: v for k, v in self.tensors.items() if k in keep}


class Handle:
    """Owns a workspace tensor and a dflash_handle. Methods map 1:1 onto the C calls."""

    def __init__(self, cfg: dflash_config, weights: dflash_weights, stream=None, device="cuda"):
        import torch
        self.cfg = cfg
        nbytes = lib().dflash_workspace_bytes(ctypes.byref(cfg))
        if nbytes == 0:
            raise DFlashError(DFLASH_EINVAL, "dflash_workspace_bytes")
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        base = (self.workspace.data_ptr() + 255) // 256 * 256
        self.workspace_bytes = nbytes
        h = ctypes.c_void_p()
        _check(lib().dflash_create(ctypes.byref(cfg), ctypes.byref(weights), base, nbytes, _stream_ptr(stream),
                                   ctypes.byref(h)), "dflash_create")
        self.h = h

    def project_ctx(self, req_ids, n_new, taps, stream=None) -> int:
        return _check(lib().dflash_project_ctx(self.h, len(req_ids), _int_array(req_ids), _int_array(n_new),
                                               taps.data_ptr() if taps is not None else None, _stream_ptr(stream)),
                      "dflash_project_ctx")

    def draft_block(self, req_ids, anchor, draft, conf=None, logits=None, temperature=0.0, stream=None) -> int:
        return _check(lib().dflash_draft_block(self.h, len(req_ids), _int_array(req_ids), anchor.data_ptr(),
                                               float(temperature), draft.data_ptr(),
                                               conf.data_ptr() if conf is not None else None,
                                               logits.data_ptr() if logits is not None else None,
                                               _stream_ptr(stream)), "dflash_draft_block")

    def accept(self, draft, target, accept_len, next_anchor, stream=None) -> int:
        return _check(lib().dflash_accept(self.h, draft.shape[0], draft.data_ptr(), target.data_ptr(),
                                          accept_len.data_ptr(), next_anchor.data_ptr(), _stream_ptr(stream)),
                      "dflash_accept")

    def rows_matmul(self, matrix, layer, x, y, scratch, x_lo=None, stream=None) -> int:
        """y[r][n] = sum_k x[r][k] W[n][k] for a stored 4-bit matrix (DFLASH_MAT_*): x f16 [rows][ldx]
        (int16 bits), x_lo its f16 remainder or None, y fp32 [rows][ldy], scratch a uint8 device
        tensor of at least the plan's scratch_bytes (256-byte aligned)."""
        return _check(lib().dflash_rows_matmul(self.h, matrix, layer, x.shape[0], x.data_ptr(),
                                               x_lo.data_ptr() if x_lo is not None else None, x.stride(0),
                                               y.data_ptr(), y.stride(0), scratch.data_ptr(), scratch.numel(),
                                               _stream_ptr(stream)), "dflash_rows_matmul")

    def draft_lengths(self, conf, keep, thresholds=None, min_conf=0.0, stream=None) -> int:
        """Confidence-scheduled pruning: keep[i] = drafts of request i the target verifies."""
        return _check(lib().dflash_draft_lengths(self.h, conf.shape[0], conf.data_ptr(),
                                                 thresholds.data_ptr() if thresholds is not None else None,
                                                 float(min_conf), keep.data_ptr(), _stream_ptr(stream)),
                      "dflash_draft_lengths")

    def accept_kept(self, draft, keep, target, accept_len, next_anchor, stream=None) -> int:
        return _check(lib().dflash_accept_kept(self.h, draft.shape[0], draft.data_ptr(), keep.data_ptr(),
                                               target.data_ptr(), accept_len.data_ptr(), next_anchor.data_ptr(),
                                               _stream_ptr(stream)), "dflash_accept_kept")

    def reset_request(self, req_id: int) -> int:
        return _check(lib().dflash_reset_request(self.h, req_id), "dflash_reset_request")

    def ctx_len(self, req_id: int) -> int:
        return lib().dflash_ctx_len(self.h, req_id)

    def check_errors(self, stream=None) -> int:
        return _check(lib().dflash_check_errors(self.h, _stream_ptr(stream)), "dflash_check_errors")

    def stats(self) -> dict:
        s = dflash_stats()
        _check(lib().dflash_get_stats(self.h, ctypes.byref(s)), "dflash_get_stats")
        return {n: getattr(s, n) for n, _ in dflash_stats._fields_}

    def set_probe(self, start_event, stop_event, kernel: int = 0) -> int:
        return _check(lib().dflash_set_probe(self.h, kernel, start_event.cuda_event, stop_event.cuda_event),
                      "dflash_set_probe")

    def launch_count(self) -> int:
        return lib().dflash_launch_count(self.h)

    def accept_histogram(self, stream=None) -> list:
        """counts[a] = accepted blocks whose accepted length was a, for a = 0 .. n_draft."""
        n = self.cfg.gamma - 1 + self.cfg.draft_all_rows + 1
        buf = (ctypes.c_uint64 * n)()
        _check(lib().dflash_accept_histogram(self.h, buf, n, _stream_ptr(stream)), "dflash_accept_histogram")
        return list(buf)

    def set_wait_limit(self, limit_us: int, stream=None) -> int:
        """Test hook: limit of the kernels' bounded waits in microseconds (0: the 1 s default)."""
        return _check(lib().dflash_set_wait_limit(self.h, limit_us, _stream_ptr(stream)), "dflash_set_wait_limit")

    def debug_stall(self, cta: int) -> int:
        """Test hook: CTA `cta` of every projection launch of the next draft call waits on a barrier
        nothing completes (cta < 0 disarms)."""
        return _check(lib().dflash_debug_stall(self.h, cta), "dflash_debug_stall")

    def close(self):
        if getattr(self, "h", None):
            lib().dflash_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
