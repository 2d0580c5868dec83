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
"""
from __future__ import annotations

import torch

from .configs import LayerCfg, F32, BF16

_TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16}


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
    fresh batch (used by multi-step balancing runs)."""
    s = cfg.seed if seed is None else seed
    dt = _TORCH_DT[cfg.act]
    return _normal((cfg.T, cfg.d), cfg.x_std, dt, device, s * 1000 + 0 + 17 * step,
                   slab_rows=4096)


def make_inputs(cfg: LayerCfg, device="cpu", seed=None) -> dict:
    """All layer inputs for ``cfg`` on ``device`` (see module docstring)."""
    if cfg.wgt not in _TORCH_DT:
        raise NotImplementedError(f"weight dtype {cfg.wgt} has no generator yet")
    s = cfg.seed if seed is None else seed
    wdt = _TORCH_DT[cfg.wgt]
    T, d, E, S, I = cfg.T, cfg.d, cfg.E, cfg.S, cfg.I
    out = {"x": make_tokens(cfg, device, s)}
    out["centroids"] = _normal((E, d), cfg.w_std, wdt, device, s * 1000 + 1)
    if cfg.bias_range > 0:
        g = _gen(device, s * 1000 + 2)
        b = torch.rand((E,), generator=g, device=device, dtype=torch.float32)
        out["bias"] = (b * 2.0 - 1.0) * cfg.bias_range
    else:
        out["bias"] = torch.zeros((E,), dtype=torch.float32, device=device)
    out["w13"] = _normal((E, 2 * I, d), cfg.w_std, wdt, device, s * 1000 + 3, slab_rows=8)
    out["w2"] = _normal((E, d, I), cfg.w_std, wdt, device, s * 1000 + 4, slab_rows=8)
    out["ws13"] = _normal((S, 2 * I, d), cfg.w_std, wdt, device, s * 1000 + 5, slab_rows=8)
    out["ws2"] = _normal((S, d, I), cfg.w_std, wdt, device, s * 1000 + 6, slab_rows=8)
    return out
