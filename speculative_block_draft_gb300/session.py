"""Host-array convenience layer over the C ABI: uploads inputs, calls the library, downloads
outputs. Marshalling only; the round itself runs in libdflash.so."""
from __future__ import annotations

import numpy as np
import torch

from . import DeviceModel, Handle, make_config


def _act_dtype(cfg):
    return torch.float32 if cfg.adtype == "f32" else torch.int16   # bf16 bits travel as int16


class Session:
    """One drafter (a dflash_synth.HostModel) on one device, with its own stream."""

    def __init__(self, host_model, max_batch: int | None = None, ctx_capacity: int | None = None,
                 device: str = "cuda:0"):
        self.cfg = host_model.cfg
        self.device = torch.device(device)
        self.stream = torch.cuda.Stream(device=self.device)
        self.dm = DeviceModel(host_model, device=self.device)
        self.ccfg = make_config(self.cfg, max_batch=max_batch, ctx_capacity=ctx_capacity)
        with torch.cuda.stream(self.stream):
            self.h = Handle(self.ccfg, self.dm.weights, stream=self.stream, device=self.device)
        self.stream.synchronize()
        self.dm.free(keep=("embed", "markov.w1"))   # borrowed by the handle; the rest was copied

    def upload(self, arr: np.ndarray, dtype=None) -> torch.Tensor:
        a = np.ascontiguousarray(arr)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        elif a.dtype == np.uint32:
            a = a.view(np.int32)
        return torch.from_numpy(a).to(self.device, non_blocking=False)

    def project(self, req_ids, n_new, taps: np.ndarray | None):
        t = self.upload(taps) if taps is not None and taps.size else None
        with torch.cuda.stream(self.stream):
            rc = self.h.project_ctx(list(req_ids), list(n_new), t, stream=self.stream)
        self.stream.synchronize()
        return rc

    def draft(self, req_ids, anchors: np.ndarray, logits: bool = True, temperature: float = 0.0):
        n = self.cfg.n_draft
        nr = len(req_ids)
        a = self.upload(np.asarray(anchors, dtype=np.int32))
        d = torch.empty((nr, n), dtype=torch.int32, device=self.device)
        c = torch.empty((nr, n), dtype=torch.float32, device=self.device)
        lg = torch.empty((nr, n, self.cfg.vocab), dtype=torch.float32, device=self.device) if logits else None
        with torch.cuda.stream(self.stream):
            rc = self.h.draft_block(list(req_ids), a, d, c, lg, temperature=temperature, stream=self.stream)
        self.stream.synchronize()
        out = {"rc": rc, "tokens": d.cpu().numpy(), "conf": c.cpu().numpy()}
        if logits:
            out["logits"] = lg.cpu().numpy()
        return out

    def accept(self, draft: np.ndarray, target: np.ndarray):
        d = self.upload(np.asarray(draft, dtype=np.int32))
        t = self.upload(np.asarray(target, dtype=np.int32))
        nr = d.shape[0]
        al = torch.empty(nr, dtype=torch.int32, device=self.device)
        na = torch.empty(nr, dtype=torch.int32, device=self.device)
        with torch.cuda.stream(self.stream):
            self.h.accept(d, t, al, na, stream=self.stream)
        self.stream.synchronize()
        return al.cpu().numpy(), na.cpu().numpy()

    def draft_lengths(self, conf: np.ndarray, thresholds: np.ndarray | None = None, min_conf: float = 0.0):
        c = self.upload(np.asarray(conf, dtype=np.float32))
        th = self.upload(np.asarray(thresholds, dtype=np.float32)) if thresholds is not None else None
        keep = torch.empty(c.shape[0], dtype=torch.int32, device=self.device)
        with torch.cuda.stream(self.stream):
            self.h.draft_lengths(c, keep, thresholds=th, min_conf=min_conf, stream=self.stream)
        self.stream.synchronize()
        return keep.cpu().numpy()

    def accept_kept(self, draft: np.ndarray, keep: np.ndarray, target: np.ndarray):
        d = self.upload(np.asarray(draft, dtype=np.int32))
        k = self.upload(np.asarray(keep, dtype=np.int32))
        t = self.upload(np.asarray(target, dtype=np.int32))
        nr = d.shape[0]
        al = torch.empty(nr, dtype=torch.int32, device=self.device)
        na = torch.empty(nr, dtype=torch.int32, device=self.device)
        with torch.cuda.stream(self.stream):
            self.h.accept_kept(d, k, t, al, na, stream=self.stream)
        self.stream.synchronize()
        return al.cpu().numpy(), na.cpu().numpy()

    def check(self):
        return self.h.check_errors(stream=self.stream)

    def close(self):
        self.h.close()
