"""MoeLayer: owns one layer's weights, bias and workspace on one GPU and calls
moe_forward (or its FP8 / pre-normed forms) and moe_update_bias through the C ABI."""
from __future__ import annotations

import torch

from . import _lib, parallel


class MoeLayer:
    """One DeepSeekMoE layer resident on a CUDA device.

    weights: dict with centroids [E,d], bias [E] fp32, w13 [E,2I,d], w2 [E,d,I],
    ws13 [S,2I,d], ws2 [S,d,I] (device tensors, layouts of include/moe.h).  FP8
    layers (cfg.wgt_dtype == MOE_E4M3) also carry w13_scale, w2_scale,
    ws13_scale, ws2_scale and run through moe_forward_fp8.

    norm_w ([d] fp32) puts the layer behind its RMSNorm: h = x + MoE(RMSNorm(x))
    through moe_forward_prenorm / moe_forward_fp8_prenorm, with eps norm_eps.

    fp8_path picks the GEMMs of an FP8 layer: "e4m3" (moe_forward_fp8: tokens
    and activations quantised to e4m3 1x128 tiles, e4m3 tensor cores, fp32
    promotion every 128 K; the faster) or "w8a16" (moe_forward_w8a16: e4m3
    weights dequantised to bf16 on the fly, bf16 tokens and activations; the
    more accurate).
    """

    def __init__(self, cfg: _lib.MoeCfg, weights: dict, device="cuda", norm_w=None,
                 norm_eps: float = 1e-6, fp8_path: str = "e4m3"):
        self.cfg = cfg
        self.device = torch.device(device)
        self.w = weights
        self.bias = weights["bias"]
        self.fp8 = cfg.wgt_dtype == _lib.MOE_E4M3
        self._fp8w = _lib.fp8_weights(weights) if self.fp8 else None
        self.norm_w = norm_w
        self.norm_eps = norm_eps
        if fp8_path not in ("w8a16", "e4m3"):
            raise ValueError(f"fp8_path {fp8_path!r}")
        self.w8a16 = self.fp8 and fp8_path == "w8a16" and norm_w is None
        self._ws = None
        self._T = None
        # tokens of the whole data-parallel batch, when every rank's batch size
        # is known up front (saves the host read that summing them costs)
        self.T_global = None

    def _buffers(self, T: int):
        if self._T != T:
            self.cfg.T = T
            kind = (_lib.MOE_WS_FORWARD_W8A16 if self.w8a16 else
                    _lib.MOE_WS_FORWARD if self.norm_w is None else _lib.MOE_WS_FORWARD_PRENORM)
            self._ws = _lib.alloc_workspace(self.cfg, kind, self.device)
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
        if self.w8a16:
            _lib.forward_w8a16(self.cfg, x, w["centroids"], self.bias, self._fp8w, self.idx,
                               self.gates, self.counts, out, self._ws, stream)
        elif self.norm_w is not None and self.fp8:
            _lib.forward_fp8_prenorm(self.cfg, x, self.norm_w, self.norm_eps, w["centroids"],
                                     self.bias, self._fp8w, self.idx, self.gates, self.counts,
                                     out, self._ws, stream)
        elif self.norm_w is not None:
            _lib.forward_prenorm(self.cfg, x, self.norm_w, self.norm_eps, w["centroids"],
                                 self.bias, w["w13"], w["w2"], w.get("ws13"), w.get("ws2"),
                                 self.idx, self.gates, self.counts, out, self._ws, stream)
        elif self.fp8:
            _lib.forward_fp8(self.cfg, x, w["centroids"], self.bias, self._fp8w, self.idx,
                             self.gates, self.counts, out, self._ws, stream)
        else:
            _lib.forward(self.cfg, x, w["centroids"], self.bias, w["w13"], w["w2"],
                         w.get("ws13"), w.get("ws2"), self.idx, self.gates, self.counts, out,
                         self._ws, stream)
        return out

    def update_bias(self, stream=None, group=None) -> torch.Tensor:
        """Sign update of the balancing bias from the last forward's counts.
        Under torch.distributed with more than one rank the counts are first
        summed over `group` (data-parallel replicas balance on the global
        batch; see parallel.py), against the tokens of all ranks
        (self.T_global if set, else summed over the ranks)."""
        def upd(cfg, counts, bias):
            _lib.update_bias(cfg, counts, bias, self.load_stats, stream)
            return self.load_stats
        return parallel.balance_step(self.cfg, self.counts, self.bias, upd, group,
                                     T_global=self.T_global)

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


class HostPipeline:
    """Runs a layer over a sequence of batches that live in pinned host memory.

    Step i copies its tokens host->device on one copy stream, runs the layer
    (forward + bias update) on the compute stream, and copies its output
    device->host on a second copy stream.  Two device buffers alternate, so
    the copies of step i+1 (in) and step i-1 (out) overlap the compute of
    step i; the compute of step i still sees the bias left by step i-1.
    """

    def __init__(self, layer: MoeLayer, like: torch.Tensor):
        self.layer = layer
        dev = layer.device
        self.x_dev = [torch.empty_like(like, device=dev) for _ in range(2)]
        self.out_dev = [torch.empty_like(like, device=dev) for _ in range(2)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
        self.x_ready, self.done, self.out_free = ev(), ev(), ev()
        self._used = [False, False]

    def run(self, x_hosts, out_hosts, stream=None):
        """Processes batch i = x_hosts[i] into out_hosts[i] for every i;
        returns once all work is queued (synchronise the streams to wait)."""
        comp = stream or torch.cuda.current_stream(self.layer.device)
        for i, (xh, oh) in enumerate(zip(x_hosts, out_hosts)):
            b = i & 1
            with torch.cuda.stream(self.h2d):
                if self._used[b]:
                    self.h2d.wait_event(self.done[b])      # compute of step i-2 read x[b]
                self.x_dev[b].copy_(xh, non_blocking=True)
                self.x_ready[b].record(self.h2d)
            comp.wait_event(self.x_ready[b])
            if self._used[b]:
                comp.wait_event(self.out_free[b])           # step i-2's output copied out
            self.layer.step(self.x_dev[b], self.out_dev[b], comp)
            self.done[b].record(comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.done[b])
                oh.copy_(self.out_dev[b], non_blocking=True)
                self.out_free[b].record(self.d2h)
            self._used[b] = True
        return out_hosts

    def synchronize(self):
        self.d2h.synchronize()
