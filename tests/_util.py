"""Shared helpers of the GPU parity tests: run the CUDA path step by step
through the C ABI and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from moe_inputs import make_inputs

# Tolerances.  bf16: the stated bar for layer outputs (relative Frobenius 1e-2,
# max-abs 3e-2).  fp32: fp32 accumulation over at most a few thousand terms,
# relative error ~1e-6; 1e-4 leaves margin.  Gates: fp32 scores, 1e-5 abs.
TOL = {"bf16": (1e-2, 3e-2), "f32": (1e-4, 1e-4)}
GATE_ATOL = 1e-5
MARGIN_EXCLUDE = 1e-5


def gpu_inputs(cfg, seed=None):
    """Inputs on the GPU plus CPU views for the oracle (small configs are drawn
    on the CPU and copied, large ones drawn on the GPU)."""
    big = cfg.T * cfg.d > 4_000_000 or cfg.E * cfg.I * cfg.d > 50_000_000
    if big:
        g = make_inputs(cfg, "cuda", seed)
        return g, g
    c = make_inputs(cfg, "cpu", seed)
    g = {k: v.cuda() for k, v in c.items()}
    return g, c


def rel_frob(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_close(got, want, dtype, what=""):
    rf, ma = TOL[dtype]
    r = rel_frob(got, want)
    m = float(np.max(np.abs(np.asarray(got, np.float64) - want))) if np.size(want) else 0.0
    assert r <= rf, f"{what}: relative Frobenius {r:.3e} > {rf}"
    assert m <= ma, f"{what}: max-abs {m:.3e} > {ma}"
    return r, m


class GpuRun:
    """Buffers and step-by-step calls of the CUDA path for one config."""

    def __init__(self, m, cfg, inp_gpu, add_residual=None):
        self.m = m
        self.lc = cfg
        self.cfg = m.cfg_from_layer(cfg)
        if add_residual is not None:
            self.cfg.add_residual = add_residual
        self.inp = inp_gpu
        T, K, E, S, d, I = cfg.T, cfg.K, cfg.E, cfg.S, cfg.d, cfg.I
        dev = "cuda"
        adt = inp_gpu["x"].dtype
        self.idx = torch.full((T, K), -1, dtype=torch.int32, device=dev)
        self.gates = torch.full((T, K), float("nan"), dtype=torch.float32, device=dev)
        self.counts = torch.full((E,), -1, dtype=torch.int32, device=dev)
        self.offsets = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
        self.xp = torch.zeros((T * K, d), dtype=adt, device=dev)
        self.perm = torch.full((T * K,), -1, dtype=torch.int32, device=dev)
        self.pos = torch.full((T, K), -1, dtype=torch.int32, device=dev)
        R = T * K + S * T
        self.act = torch.zeros((R, I), dtype=adt, device=dev)
        self.y = torch.zeros((R, d), dtype=adt, device=dev)
        self.out = torch.zeros((T, d), dtype=adt, device=dev)
        self.ws = {w: m.alloc_workspace(self.cfg, w) for w in
                   (m.MOE_WS_ROUTE, m.MOE_WS_DISPATCH, m.MOE_WS_EXPERTS, m.MOE_WS_FORWARD)}

    def route(self):
        g = self.inp
        self.m.route(self.cfg, g["x"], g["centroids"], g["bias"], self.idx, self.gates,
                     self.ws[self.m.MOE_WS_ROUTE])

    def dispatch(self, idx=None):
        self.m.dispatch(self.cfg, self.inp["x"], self.idx if idx is None else idx, self.counts,
                        self.offsets, self.xp, self.perm, self.pos,
                        self.ws[self.m.MOE_WS_DISPATCH])

    def experts(self):
        g = self.inp
        self.m.experts(self.cfg, self.xp, g["x"], self.offsets, g["w13"], g["w2"],
                       g["ws13"] if self.lc.S else None, g["ws2"] if self.lc.S else None,
                       self.act, self.y, self.ws[self.m.MOE_WS_EXPERTS])

    def combine(self, gates=None, pos=None):
        self.m.combine(self.cfg, self.y, self.gates if gates is None else gates,
                       self.pos if pos is None else pos, self.inp["x"], self.out)

    def forward(self):
        g = self.inp
        self.m.forward(self.cfg, g["x"], g["centroids"], g["bias"], g["w13"], g["w2"],
                       g["ws13"] if self.lc.S else None, g["ws2"] if self.lc.S else None,
                       self.idx, self.gates, self.counts, self.out,
                       self.ws[self.m.MOE_WS_FORWARD])

    def status(self):
        return self.m.get_status()


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()
