"""MoeLayer: owns one layer's weights, bias and workspace on one GPU and calls
moe_forward / moe_update_bias through the C ABI."""
from __future__ import annotations

import torch

from . import _lib


class MoeLayer:
    """One DeepSeekMoE layer resident on a CUDA device.

    weights: dict with centroids [E,d], bias [E] fp32, w13 [E,2I,d], w2 [E,d,I],
    ws13 [S,2I,d], ws2 [S,d,I] (device tensors, layouts of include/moe.h).
    """

    def __init__(self, cfg: _lib.MoeCfg, weights: dict, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        self.w = weights
        self.bias = weights["bias"]
        self._ws = None
        self._T = None

    def _buffers(self, T: int):
        if self._T != T:
            self.cfg.T = T
            self._ws = _lib.alloc_workspace(self.cfg, _lib.MOE_WS_FORWARD, self.device)
            K, E = self.cfg.K, self.cfg.E
            self.idx = torch.empty((T, K), dtype=torch.int32, device=self.device)
            self.gates = torch.empty((T, K), dtype=torch.float32, device=self.device)
            self.counts = torch.empty((E,), dtype=torch.int32, device=self.device)
            self.load_stats = torch.empty((2,), dtype=torch.float32, device=self.device)
            self._T = T

    def forward(self, x: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
        """out = layer(x); also leaves idx, gates, counts on the layer."""
        T = x.shape[0]
        self._buffers(T)
        if out is None:
            out = torch.empty_like(x)
        w = self.w
        _lib.forward(self.cfg, x, w["centroids"], self.bias, w["w13"], w["w2"], w.get("ws13"),
                     w.get("ws2"), self.idx, self.gates, self.counts, out, self._ws, stream)
        return out

    def update_bias(self, stream=None) -> torch.Tensor:
        """Sign update of the balancing bias from the last forward's counts."""
        _lib.update_bias(self.cfg, self.counts, self.bias, self.load_stats, stream)
        return self.load_stats

    def step(self, x: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
        """One batch of the layer: forward, then the bias update for the next batch."""
        out = self.forward(x, out, stream)
        self.update_bias(stream)
        return out

    def step_host(self, x_host: torch.Tensor, out_host: torch.Tensor, x_dev: torch.Tensor,
                  out_dev: torch.Tensor, stream=None) -> torch.Tensor:
        """Host-to-host step: copies x (pinned host) in, runs the layer and the
        bias update, copies out back to pinned host memory."""
        x_dev.copy_(x_host, non_blocking=True)
        self.step(x_dev, out_dev, stream)
        out_host.copy_(out_dev, non_blocking=True)
        return out_host
