"""Seeded random inputs for a DeepSeekMoE layer.

Every tensor j of a layer is drawn from its own torch generator seeded with
``seed * 1000 + j`` on the requested device, in fp32, then rounded (RNE) to the
layer's dtype.  Large tensors are drawn on the GPU in per-expert slabs so that
no fp32 copy of a whole weight tensor is ever materialised.

Layout (row-major, K-contiguous, as the C ABI expects):
    x          [T, d]            tokens u_t
    centroids  [E, d]            expert centroids e_i
    bias       [E]     fp32      load-balancing bias b_i
    w13        [E, 2I, d]        rows 0..I-1 = gate projection, I..2I-1 = up
    w2         [E, d, I]         down projection
    ws13       [S, 2I, d]        shared experts, same layout
    ws2        [S, d, I]
    norm_w     [d]     fp32      weight of the RMSNorm in front of the layer

FP8 (e4m3) layers store every expert weight as e4m3 values plus one fp32 scale
per 128 x 128 block ("block-wise" quantisation of the V3 walk-through,
section 4.3): w13_scale [E, 2I/128, d/128], w2_scale [E, d/128, I/128], and
ws13_scale, ws2_scale alike.  Quantisation belongs to the generator: each
block is drawn in fp32, scale = max|w| / 448, q = e4m3(w / scale) rounded to
nearest even and clamped to +-448.  The layer then computes with q * scale.

Zipf-skewed layers (zipf_s > 0) make expert popularity follow rank^-zipf_s:
x[:, 0] = 1 in every token and centroid column 0 holds a per-expert offset
delta_i, fitted once on a seed-1 calibration batch so that the unbiased
top-K frequency of expert i (rank i + 1) approaches the target (see
``zipf_offsets``).
"""
from __future__ import annotations

import torch

import math

from .configs import LayerCfg, F32, BF16, E4M3

_TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16}
E4M3_MAX = 448.0
BLOCK = 128


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, dtype, device, seed, slab_rows=None):
    """N(0, std) drawn in fp32 then rounded to ``dtype``; drawn slab by slab
    along dim 0 when ``slab_rows`` is given (bounded fp32 temporaries)."""
    out = torch.empty(shape, dtype=dtype, device=device)
    g = _gen(device, seed)
    n0 = shape[0]
    step = n0 if slab_rows is None else max(1, slab_rows)
    for a in range(0, n0, step):
        b = min(n0, a + step)
        t = torch.randn((b - a,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        t.mul_(std)
        out[a:b].copy_(t)
    return out


def make_tokens(cfg: LayerCfg, device="cpu", seed=None, step: int = 0) -> torch.Tensor:
    """Token batch x ~ N(0, x_std) in the activation dtype.  ``step`` selects a
    fresh batch (used by multi-step balancing runs).  Zipf layers set x[:, 0] = 1."""
    s = cfg.seed if seed is None else seed
    dt = _TORCH_DT[cfg.act]
    x = _normal((cfg.T, cfg.d), cfg.x_std, dt, device, s * 1000 + 0 + 17 * step,
                slab_rows=4096)
    if cfg.zipf_s > 0:
        x[:, 0] = 1.0
    return x


def _quantize_blocks(w: torch.Tensor):
    """fp32 [n, R, C] -> (e4m3 [n, R, C], fp32 scales [n, R/128, C/128])."""
    n, R, C = w.shape
    blk = w.reshape(n, R // BLOCK, BLOCK, C // BLOCK, BLOCK)
    amax = blk.abs().amax(dim=(2, 4))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (blk / scale[:, :, None, :, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    q = q.reshape(n, R, C).to(torch.float8_e4m3fn)
    return q, scale.to(torch.float32)


def _normal_e4m3(shape, std, device, seed, slab_rows=8):
    """N(0, std) weights drawn in fp32 slab by slab, stored block-scaled e4m3."""
    n, R, C = shape
    if R % BLOCK or C % BLOCK:
        raise ValueError("FP8 weights need both dims to be multiples of 128")
    q = torch.empty(shape, dtype=torch.float8_e4m3fn, device=device)
    sc = torch.empty((n, R // BLOCK, C // BLOCK), dtype=torch.float32, device=device)
    g = _gen(device, seed)
    for a in range(0, n, slab_rows):
        b = min(n, a + slab_rows)
        t = torch.randn((b - a, R, C), generator=g, device=device, dtype=torch.float32)
        t.mul_(std)
        q[a:b], sc[a:b] = _quantize_blocks(t)
    return q, sc


def zipf_targets(E: int, K: int, s: float) -> torch.Tensor:
    """Per-token top-K frequency of the expert of rank r = i + 1: proportional
    to r^-s, capped at 1 (an expert is chosen at most once per token), and
    summing to K.  The cap is met by water-filling: capped experts are fixed at
    1 and the rest rescaled until no other exceeds 1."""
    w = torch.arange(1, E + 1, dtype=torch.float64) ** (-s)
    f = torch.zeros(E, dtype=torch.float64)
    capped = torch.zeros(E, dtype=torch.bool)
    for _ in range(E):
        free = ~capped
        f[free] = w[free] * (K - capped.sum().item()) / w[free].sum()
        f[capped] = 1.0
        over = free & (f > 1.0)
        if not over.any():
            break
        capped |= over
    return f


def zipf_offsets(cfg: LayerCfg, centroids: torch.Tensor, calib_tokens: int = 4096,
                 iters: int = 50) -> torch.Tensor:
    """Centroid offsets delta_i (added to logit i through x[:, 0] = 1) fitted so
    the unbiased top-K frequencies on a seed-1 batch of ``calib_tokens`` tokens
    approach ``zipf_targets``: delta_i += 0.5 (ln target_i - ln freq_i), at most
    ``iters`` times.  Sigmoid is monotone, so top-K of the scores is top-K of
    the logits and the fit works on logits."""
    dev = centroids.device
    xc = make_tokens(cfg.with_(T=calib_tokens), dev, seed=1).float()
    base = xc[:, 1:] @ centroids[:, 1:].float().T              # logits without column 0
    tgt = zipf_targets(cfg.E, cfg.K, cfg.zipf_s).to(dev)
    delta = torch.zeros(cfg.E, dtype=torch.float64, device=dev)
    floor = 0.5 / calib_tokens
    for _ in range(iters):
        top = torch.topk(base + delta.float()[None, :], cfg.K, dim=1).indices
        freq = torch.bincount(top.reshape(-1), minlength=cfg.E).double() / calib_tokens
        delta += 0.5 * (torch.log(tgt.clamp_min(floor)) - torch.log(freq.clamp_min(floor)))
    return delta


def make_inputs(cfg: LayerCfg, device="cpu", seed=None) -> dict:
    """All layer inputs for ``cfg`` on ``device`` (see module docstring)."""
    s = cfg.seed if seed is None else seed
    fp8 = cfg.wgt == E4M3
    wdt = torch.bfloat16 if fp8 else _TORCH_DT[cfg.wgt]   # centroid dtype
    T, d, E, S, I = cfg.T, cfg.d, cfg.E, cfg.S, cfg.I
    out = {"x": make_tokens(cfg, device, s)}
    out["centroids"] = _normal((E, d), cfg.w_std, wdt, device, s * 1000 + 1)
    if cfg.zipf_s > 0:
        out["centroids"][:, 0] = zipf_offsets(cfg, out["centroids"]).to(wdt)
    if cfg.bias_range > 0:
        g = _gen(device, s * 1000 + 2)
        b = torch.rand((E,), generator=g, device=device, dtype=torch.float32)
        out["bias"] = (b * 2.0 - 1.0) * cfg.bias_range
    else:
        out["bias"] = torch.zeros((E,), dtype=torch.float32, device=device)
    shapes = {"w13": (E, 2 * I, d), "w2": (E, d, I), "ws13": (S, 2 * I, d), "ws2": (S, d, I)}
    for j, (k, shp) in enumerate(shapes.items()):
        if fp8:
            out[k], out[k + "_scale"] = _normal_e4m3(shp, cfg.w_std, device, s * 1000 + 3 + j)
        else:
            out[k] = _normal(shp, cfg.w_std, wdt, device, s * 1000 + 3 + j, slab_rows=8)
    out["norm_w"] = make_norm_weight(cfg, device, s)
    return out


def make_norm_weight(cfg: LayerCfg, device="cpu", seed=None) -> torch.Tensor:
    """Per-channel weight of the RMSNorm in front of the layer, fp32 [d]:
    U(0.5, 1.5), a spread around the initial value 1 so that a dropped or
    misplaced weight changes the result."""
    s = cfg.seed if seed is None else seed
    g = _gen(device, s * 1000 + 7)
    return 0.5 + torch.rand((cfg.d,), generator=g, device=device, dtype=torch.float32)


def make_dout(cfg: LayerCfg, device="cpu", seed=None) -> torch.Tensor:
    """Gradient of a scalar loss with respect to the layer output, for the
    backward pass: N(0, 1) per element in the activation dtype [T, d], drawn
    slab by slab like the tokens."""
    s = cfg.seed if seed is None else seed
    return _normal((cfg.T, cfg.d), 1.0, _TORCH_DT[cfg.act], device, s * 1000 + 8,
                   slab_rows=4096)
