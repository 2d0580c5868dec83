"""GPU parity of the RMSNorm in front of the layer (V3 walk-through, section
4.1: an RMSNorm before and after the MoE layer, eps 1e-6) and of the layer
behind it, h = x + MoE(RMSNorm(x)), through the C ABI.

moe_rmsnorm computes the norm in fp32 and rounds once to the activation type;
the oracle computes it in fp64 and rounds once.  The two can land on
neighbouring bf16 values where the exact result lies within fp32 error of a
rounding boundary (about one element in 10^4), so the norm is compared
element-wise within one unit in the last place with at most 1e-3 of the
elements off.

The layer's router reads no normalised token: its logit is
inv_rms * (x . (w * e_i)) with the weighted centroids w * e_i held in the
weight type, on both sides.  The strict routing checks (sets bit-exact,
gates within 1e-5) therefore apply to every token whose K-th vs (K+1)-th
margin is >= 1e-5; a token below that margin must hold a valid top-K of the
oracle's keys and its gates, and its output is compared with the oracle's
layer on that choice.  The experts read the normalised rows.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from moe_inputs import small_cases, get_config
from oracle import moe_oracle as O
from tests._util import (GpuRun, gpu_inputs, assert_close, to_np, rel_frob, check_near_ties,
                         with_gpu_choice)

pytestmark = pytest.mark.gpu

m = pytest.importorskip("mixture_experts_layer_88_b300")

EPS = 1e-6
SMALL = ["tiny", "small_bf16", "ragged_bf16", "softmax_norenorm"]


def _cfg(name):
    return small_cases()[name] if name in small_cases() else get_config(name)


def _ulp(v, act):
    """Spacing of the activation type at each value of v (normal range)."""
    _, e = np.frexp(np.asarray(v, np.float64))
    bits = 8 if act == "bf16" else 24
    return np.ldexp(1.0, e - bits)


def _norm_gpu(cfg, g):
    mc = m.cfg_from_layer(cfg)
    xn = torch.empty_like(g["x"])
    inv = torch.empty((cfg.T,), dtype=torch.float32, device="cuda")
    m.rmsnorm(mc, g["x"], g["norm_w"], EPS, xn, inv)
    torch.cuda.synchronize()
    assert m.get_status() == 0
    return xn, inv


def _rows_agree(cfg, xn_gpu, c, rows=None):
    """Per token row: does the kernel's normalised row equal the oracle's?"""
    x = c["x"] if rows is None else c["x"][torch.as_tensor(rows, device=c["x"].device)]
    want = O.round_act(O.rmsnorm(x, c["norm_w"], EPS)[0], cfg.act)
    got = to_np(xn_gpu if rows is None else xn_gpu[torch.as_tensor(rows, device="cuda")])
    return np.all(got == want, axis=1), got, want


@pytest.mark.parametrize("name", SMALL + ["v3_prefill"])
def test_rmsnorm_parity(name):
    cfg = _cfg(name)
    g, c = gpu_inputs(cfg)
    xn, inv = _norm_gpu(cfg, g)
    rows = None
    if cfg.T > 4096:
        rng = np.random.default_rng(11)
        rows = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, 254, replace=False)]))
    same, got, want = _rows_agree(cfg, xn, c, rows)
    x = c["x"] if rows is None else c["x"][torch.as_tensor(rows, device=c["x"].device)]
    _, winv = O.rmsnorm(x, c["norm_w"], EPS)
    ginv = inv.cpu().numpy().astype(np.float64)
    if rows is not None:
        ginv = ginv[rows]
    np.testing.assert_allclose(ginv, winv, rtol=2e-6, atol=0)   # fp32 sum of d squares
    diff = np.abs(got - want)
    if cfg.act == "bf16":
        assert np.all(diff <= _ulp(want, "bf16")), "normalised value off by more than one ulp"
        assert np.mean(diff > 0) <= 1e-3, f"{np.mean(diff > 0):.2e} of the elements off"
    else:
        np.testing.assert_allclose(got, O.rmsnorm(x, c["norm_w"], EPS)[0], rtol=1e-6, atol=0)


def test_rmsnorm_in_place_and_constant_rows():
    cfg = small_cases()["small_bf16"]
    g, c = gpu_inputs(cfg)
    xn, _ = _norm_gpu(cfg, g)
    x2 = g["x"].clone()
    mc = m.cfg_from_layer(cfg)
    m.rmsnorm(mc, x2, g["norm_w"], EPS, x2)            # xn may be x itself
    torch.cuda.synchronize()
    assert torch.equal(x2, xn)
    # constant rows: closed form c * w / sqrt(c^2 + eps), rounded once
    xc = torch.full((4, cfg.d), 0.0, dtype=torch.bfloat16, device="cuda")
    for i, v in enumerate((0.5, -3.0, 1e-3, 7.0)):
        xc[i] = v
    mc4 = m.cfg_from_layer(cfg.with_(T=4))
    out = torch.empty_like(xc)
    m.rmsnorm(mc4, xc, g["norm_w"], EPS, out)
    torch.cuda.synchronize()
    w = O._f64(c["norm_w"])
    for i, v in enumerate((0.5, -3.0, 1e-3, 7.0)):
        cv = float(torch.tensor(v, dtype=torch.bfloat16))
        want = O.round_bf16(cv * w / np.sqrt(cv * cv + EPS))
        got = to_np(out[i])
        assert np.all(np.abs(got - want) <= _ulp(want, "bf16"))


class PrenormRun(GpuRun):
    def forward_prenorm(self):
        g = self.inp
        ws = m.alloc_workspace(self.cfg, m.MOE_WS_FORWARD_PRENORM)
        m.forward_prenorm(self.cfg, g["x"], g["norm_w"], EPS, g["centroids"], g["bias"],
                          g["w13"], g["w2"], g["ws13"] if self.lc.S else None,
                          g["ws2"] if self.lc.S else None, self.idx, self.gates, self.counts,
                          self.out, ws)


def _oracle_prenorm(cfg, c, **kw):
    return O.moe_layer(c, cfg.K, cfg.normalize, cfg.score_func, n_groups=cfg.n_groups,
                       topk_groups=cfg.topk_groups, norm_w=c["norm_w"], norm_eps=EPS,
                       act=cfg.act, wgt="bf16" if cfg.wgt == "e4m3" else cfg.wgt, **kw)


def _checked(cfg, c, idx_g, gates_g, add_residual, tokens=None, **kw):
    """The oracle's pre-normed layer (on `tokens`, default all) with routing
    checked against the GPU's: chosen sets bit-exact where the K-th vs
    (K+1)-th margin is >= 1e-5, a valid top-K within 1e-5 and its gates
    elsewhere (those rows recomputed on the GPU's choice).  The router reads
    the raw tokens and the weighted centroids on both sides, so no token's
    routing depends on the rounding of its normalised row."""
    ref = _oracle_prenorm(cfg, c, add_residual=add_residual, tokens=tokens, **kw)
    keep, n_excl = check_near_ties(cfg, idx_g, ref["margin"], ref["scores"], c["bias"], gates_g)
    if cfg.zipf_s == 0:
        assert n_excl <= max(2, len(keep) // 50)
    np.testing.assert_array_equal(np.sort(idx_g, 1)[keep], np.sort(ref["idx"], 1)[keep])
    tok = np.arange(len(keep)) if tokens is None else np.asarray(tokens)
    return with_gpu_choice(ref, idx_g, keep, lambda rows, ix: _oracle_prenorm(
        cfg, c, add_residual=add_residual, tokens=tok[rows], idx=ix, **kw))


# bf16 small layers take the fused router (logits from the raw tokens and the
# weighted centroids, 1/rms from its own sums of squares, rows normalised in
# the dispatch); the fp32 layer ("tiny") and E > 256 ("wide_e") take the
# RMSNorm kernel and the two-kernel router with its logits scaled by inv_rms
PRE = SMALL + ["wide_e", "grouped_bf16"]


@pytest.mark.parametrize("name", PRE)
def test_forward_prenorm_vs_oracle(name):
    cfg = _cfg(name)
    ar = 1 if name in ("tiny", "small_bf16") else 0
    g, c = gpu_inputs(cfg)
    run = PrenormRun(m, cfg, g, add_residual=ar)
    run.forward_prenorm()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    idx_g = run.idx.cpu().numpy()
    ref = _checked(cfg, c, idx_g, run.gates.cpu().numpy(), ar)
    # with add_residual the oracle's residual is x itself: adding the
    # normalised tokens instead would be off by O(1)
    assert_close(to_np(run.out), ref["out"] if ar else ref["delta"], cfg.act,
                 f"{name} pre-normed layer")
    np.testing.assert_array_equal(run.counts.cpu().numpy(),
                                  np.bincount(idx_g.reshape(-1), minlength=cfg.E))
    # against the oracle that also rounds act, y and the output where the
    # kernels store them (its normalised rows are rounded to the activation
    # type in either form)
    refr = _checked(cfg, c, idx_g, run.gates.cpu().numpy(), ar, stored_rounding=True)
    r = rel_frob(to_np(run.out), refr["out"] if ar else refr["delta"])
    assert r <= {"bf16": 1e-3, "f32": 1e-5}[cfg.act], f"{name}: stored rounding {r:.3e}"


@pytest.mark.parametrize("name", ["small_bf16", "ragged_bf16", "softmax_norenorm"])
def test_forward_prenorm_matches_layer_on_normalised_tokens(name):
    """moe_forward_prenorm(x) and moe_forward(moe_rmsnorm(x)) compute the same
    layer with the router's one rounding in different places (w * e_i held
    in bf16 against xn held in bf16: ~2^-9 relative per product, so logits
    and gates differ by ~1e-3).  They must pick the same experts for nearly
    every token and, on those tokens, agree within the layer bar."""
    cfg = _cfg(name)
    g, _ = gpu_inputs(cfg)
    a = PrenormRun(m, cfg, g, add_residual=0)
    a.forward_prenorm()
    xn, _ = _norm_gpu(cfg, g)
    b = GpuRun(m, cfg, dict(g, x=xn), add_residual=0)
    b.forward()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    ia, ib = a.idx.cpu().numpy(), b.idx.cpu().numpy()
    same = np.all(np.sort(ia, 1) == np.sort(ib, 1), axis=1)
    assert same.mean() >= 0.95, f"routing agrees on {same.mean():.3f} of the tokens"
    np.testing.assert_allclose(a.gates.cpu().numpy()[same], b.gates.cpu().numpy()[same],
                               rtol=0, atol=2e-2)
    assert_close(to_np(a.out)[same], to_np(b.out)[same], cfg.act, f"{name} two forms")


def test_prenorm_fused_router_launches_no_norm_pass():
    """Behind the RMSNorm the bf16 layer's kernels are the weighted-centroid
    fold, the fused router, the dispatch (which normalises), the experts and
    the combine: no separate RMSNorm pass and no logits in memory."""
    cfg = small_cases()["small_bf16"]
    g, _ = gpu_inputs(cfg)
    layer = m.MoeLayer(m.cfg_from_layer(cfg), g, device="cuda", norm_w=g["norm_w"],
                       norm_eps=EPS)
    layer.forward(g["x"])
    torch.cuda.synchronize()
    m.trace_enable(True)
    m.trace_read_all()
    layer.forward(g["x"])
    torch.cuda.synchronize()
    names = {n for n, _, _ in m.trace_read_all()}
    m.trace_enable(False)
    assert "rmsnorm" not in names and "gemm_router" not in names and "router_topk" not in names
    assert {"fold_centroids", "router_fused", "dispatch_scatter_norm"} <= names


@pytest.mark.parametrize("name", ["small_fp8", "ragged_fp8"])
def test_forward_fp8_prenorm_vs_oracle(name):
    cfg = small_cases()[name]
    g, c = gpu_inputs(cfg)
    T, K, E = cfg.T, cfg.K, cfg.E

    class R:
        pass

    def run_fp8(add_residual):
        mc = m.cfg_from_layer(cfg)
        mc.add_residual = add_residual
        r = R()
        r.idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
        r.gates = torch.zeros((T, K), dtype=torch.float32, device="cuda")
        r.counts = torch.zeros((E,), dtype=torch.int32, device="cuda")
        r.out = torch.zeros_like(g["x"])
        ws = m.alloc_workspace(mc, m.MOE_WS_FORWARD_PRENORM)
        m.forward_fp8_prenorm(mc, g["x"], g["norm_w"], EPS, g["centroids"], g["bias"],
                              m.fp8_weights(g), r.idx, r.gates, r.counts, r.out, ws)
        torch.cuda.synchronize()
        assert m.get_status() == 0
        return r

    r0, r1 = run_fp8(0), run_fp8(1)
    assert torch.equal(r0.idx, r1.idx) and torch.equal(r0.gates, r1.gates)
    ref = _checked(cfg, c, r0.idx.cpu().numpy(), r0.gates.cpu().numpy(), 1)
    got0, got1 = to_np(r0.out), to_np(r1.out)
    rf = rel_frob(got0, ref["delta"])
    assert rf <= 5e-2, f"relative Frobenius of the MoE term {rf:.3e}"
    # against the oracle that quantises the activations as the kernels do
    refq = _checked(cfg, c, r0.idx.cpu().numpy(), r0.gates.cpu().numpy(), 1, act_quant=True)
    rq = rel_frob(got0, refq["delta"])
    assert rq <= 1e-2, f"relative Frobenius against the quantising oracle {rq:.3e}"
    # the residual is x itself (the normalised tokens would be off by O(1)):
    # with and without it the outputs differ by x, up to the two bf16 roundings
    res = got1 - got0 - to_np(g["x"])
    bound = 2.0 ** -8 * (np.abs(got1) + np.abs(got0)) + 1e-6
    assert np.all(np.abs(res) <= bound)


def test_forward_prenorm_full_size_sampled():
    """V3 prefill layer behind its RMSNorm at full size: invariants on every
    token, routing and outputs on a token sample."""
    cfg = get_config("v3_prefill")
    g, c = gpu_inputs(cfg)
    run = PrenormRun(m, cfg, g, add_residual=1)
    run.forward_prenorm()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    idx_g = run.idx.cpu().numpy()
    counts = run.counts.cpu().numpy()
    assert counts.sum() == cfg.T * cfg.K
    np.testing.assert_array_equal(counts, np.bincount(idx_g.reshape(-1), minlength=cfg.E))
    assert torch.isfinite(run.out.float()).all()
    rng = np.random.default_rng(4321)
    tok = np.sort(rng.choice(cfg.T, 8, replace=False))
    tok[0], tok[-1] = 0, cfg.T - 1
    ref = _checked(cfg, c, idx_g[tok], run.gates.cpu().numpy()[tok], 1, tokens=tok)
    out = to_np(run.out)[tok]
    assert_close(out, ref["out"], cfg.act, "V3 prefill pre-normed, sampled tokens")
