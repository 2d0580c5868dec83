"""GPU parity of the training forward and the backward pass (moe_forward_train,
moe_backward) against the CPU oracle's chain rule (``moe_layer_backward``),
through the C ABI.

Bar: every gradient tensor within relative Frobenius 1e-2 of the oracle's
and max |diff| <= 3e-2 * max |oracle|.  The kernels keep the output gradients
of the rows (g * dout), da, [dgate, dup] and the routed rows' du in bf16
(2^-9 relative each) and accumulate in fp32; a chain of four such roundings
stays far below 1 %.  Routing must match the oracle's on every token whose
top-K margin is >= 1e-5; a token below that margin must hold a valid top-K
of the oracle's keys within 1e-5 (check_near_ties), and only on such
validated tokens does the oracle's backward run on the GPU's choice of
experts (recomputing the gates for it).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from moe_inputs import get_config, make_dout, make_inputs, small_cases
from oracle import moe_oracle as O
from tests._util import (check_near_ties, gpu_inputs, idx_with_counts, rel_frob, to_np,
                         with_gpu_choice)

pytestmark = pytest.mark.gpu

m = pytest.importorskip("mixture_experts_layer_88_b300")

BWD = [k for k, c in small_cases().items() if c.act == "bf16" and c.wgt == "bf16"]


def assert_grad_close(got, want, what, rf=1e-2, ma=3e-2):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    scale = float(np.max(np.abs(want))) if want.size else 0.0
    if scale == 0.0:
        assert not np.any(got), f"{what}: expected zeros"
        return
    r = rel_frob(got, want)
    mx = float(np.max(np.abs(got - want)))
    assert r <= rf, f"{what}: relative Frobenius {r:.3e} > {rf}"
    assert mx <= ma * scale, f"{what}: max-abs {mx:.3e} > {ma} * {scale:.3e}"


def router_term_scale(c, cfg, ref, idx):
    """|dC| bound of the centroid gradient's terms before the renormalisation
    and the Softmax cancel: per expert, sum over tokens of |x_t| times the
    dlogit built from |dg| and |sum_j dg_j g_j| (and, for Softmax, |sum ds s|)
    instead of their differences.  dgates = dout . y carry the bf16 rounding of
    the stored y (2^-9 relative per element), so dC is held to the bf16 bar
    relative to this magnitude; the differences themselves can be much
    smaller than their terms (a token whose dg_k all lie near their gate-
    weighted mean)."""
    x = O._f64(c["x"])
    s = O.expert_scores(O.affinity_logits(x, c["centroids"]), cfg.score_func)
    ix = idx.astype(np.int64)
    dg = ref["dgates"]
    if cfg.normalize:
        tot = np.take_along_axis(s, ix, 1).sum(axis=1, keepdims=True)
        dsa = (np.abs(dg) + np.abs((dg * ref["gates"]).sum(axis=1, keepdims=True))) / tot
    else:
        dsa = np.abs(dg)
    full = np.zeros_like(s)
    np.put_along_axis(full, ix, dsa, axis=1)
    if cfg.score_func == O.SIGMOID:
        a = full * s * (1.0 - s)
    else:
        a = s * (full + (full * s).sum(axis=1, keepdims=True))
    return a.T @ np.abs(x)


class TrainRun:
    """Buffers and calls of the training path for one bf16 config."""

    def __init__(self, cfg, g):
        self.lc = cfg
        self.cfg = m.cfg_from_layer(cfg)
        self.g = g
        self.state = m.alloc_train_state(self.cfg)
        self.grads = m.alloc_grads(self.cfg)
        for t in list(self.state.values()) + list(self.grads.values()):
            if t.is_floating_point():
                t.fill_(float("nan"))
            else:
                t.fill_(-7)
        self.out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
        self.ws_f = m.alloc_workspace(self.cfg, m.MOE_WS_FORWARD_TRAIN)
        self.ws_b = m.alloc_workspace(self.cfg, m.MOE_WS_BACKWARD)

    def _w(self, k):
        return self.g[k] if self.lc.S else None

    def forward(self):
        g = self.g
        m.forward_train(self.cfg, g["x"], g["centroids"], g["bias"], g["w13"], g["w2"],
                        self._w("ws13"), self._w("ws2"), self.state, self.out, self.ws_f)

    def backward(self, dout):
        g = self.g
        m.backward(self.cfg, dout, g["x"], g["centroids"], g["w13"], g["w2"], self._w("ws13"),
                   self._w("ws2"), self.state, self.grads, self.ws_b)


def _run(cfg, g):
    run = TrainRun(cfg, g)
    dout = make_dout(cfg, "cuda")
    run.forward()
    run.backward(dout)
    torch.cuda.synchronize()
    assert m.get_status() == 0
    return run, dout


def _checked_idx(cfg, run, c):
    """The oracle's choice of experts, except on near-tie tokens whose GPU
    choice was validated as a top-K within 1e-5: there the GPU's."""
    idx_o, _, margin, s = O.route(c["x"], c["centroids"], c["bias"], cfg.K, cfg.score_func,
                                  cfg.normalize, cfg.n_groups, cfg.topk_groups)
    idx_g = run.state["idx"].cpu().numpy()
    keep, _ = check_near_ties(cfg, idx_g, margin, s, c["bias"], run.state["gates"].cpu().numpy())
    np.testing.assert_array_equal(np.sort(idx_g, 1)[keep], np.sort(idx_o, 1)[keep])
    idx = idx_o.copy()
    idx[~keep] = idx_g[~keep]
    return idx


def _check_against_oracle(cfg, run, c, dout, what):
    idx = _checked_idx(cfg, run, c)
    ref = O.moe_layer_backward(c, cfg.K, dout.cpu(), cfg.normalize, cfg.score_func,
                               cfg.add_residual, cfg.n_groups, cfg.topk_groups, idx=idx)
    gr = run.grads
    assert_grad_close(to_np(gr["dx"]), ref["dx"], f"{what} dx")
    dc = to_np(gr["dcentroids"])
    bound = router_term_scale(c, cfg, ref, idx)
    assert np.all(np.isfinite(dc))
    assert np.linalg.norm(dc - ref["dcentroids"]) <= 1e-2 * max(np.linalg.norm(bound), 1e-30), \
        f"{what} dcentroids: {rel_frob(dc, ref['dcentroids']):.3e} of the oracle's norm"
    assert np.max(np.abs(dc - ref["dcentroids"])) <= 3e-2 * max(float(np.max(bound)), 1e-30)
    assert_grad_close(to_np(gr["dw13"]), ref["dw13"], f"{what} dw13")
    assert_grad_close(to_np(gr["dw2"]), ref["dw2"], f"{what} dw2")
    if cfg.S:
        assert_grad_close(to_np(gr["dws13"]), ref["dws13"], f"{what} dws13")
        assert_grad_close(to_np(gr["dws2"]), ref["dws2"], f"{what} dws2")
    # experts nobody chose: exactly zero
    counts = run.state["counts"].cpu().numpy()
    for e in np.nonzero(counts == 0)[0]:
        assert not gr["dw13"][e].any() and not gr["dw2"][e].any()
    return ref


@pytest.mark.parametrize("name", BWD)
def test_backward_parity(name):
    cfg = small_cases()[name]
    g, c = gpu_inputs(cfg)
    run, dout = _run(cfg, g)
    _check_against_oracle(cfg, run, c, dout, name)


# Against the oracle that rounds to bf16 where the kernels store (h, act and y
# of the training forward; g * dout, da, [dgate, dup] and du; dx and the
# weight gradients), what remains is the fp32 rounding of the sums and the
# values it moves across a rounding boundary: measured 2e-5 to 2.6e-4 relative
# Frobenius, the largest single difference about one bf16 step.
def assert_grad_tight(got, want, what):
    assert_grad_close(got, want, what, rf=1e-3, ma=1.6e-2)


@pytest.mark.parametrize("name", BWD)
def test_backward_parity_stored_rounding(name):
    cfg = small_cases()[name]
    g, c = gpu_inputs(cfg)
    run, dout = _run(cfg, g)
    idx = _checked_idx(cfg, run, c)
    ref = O.moe_layer_backward(c, cfg.K, dout.cpu(), cfg.normalize, cfg.score_func,
                               cfg.add_residual, cfg.n_groups, cfg.topk_groups, idx=idx,
                               stored_rounding=True)
    gr = run.grads
    keys = ["dx", "dw13", "dw2", "dcentroids"] + (["dws13", "dws2"] if cfg.S else [])
    for k in keys:
        assert_grad_tight(to_np(gr[k]), ref[k], f"{name} {k}")


@pytest.mark.parametrize("name", BWD)
def test_forward_train_state(name):
    """The training forward's output, scores, routing and rows."""
    cfg = small_cases()[name]
    g, c = gpu_inputs(cfg)
    run = TrainRun(cfg, g)
    run.forward()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    def layer(**kw):
        return O.moe_layer(c, cfg.K, cfg.normalize, cfg.score_func, cfg.add_residual,
                           n_groups=cfg.n_groups, topk_groups=cfg.topk_groups, **kw)

    ref = layer()
    st = run.state
    idx = st["idx"].cpu().numpy()
    keep, _ = check_near_ties(cfg, idx, ref["margin"], ref["scores"], c["bias"],
                              st["gates"].cpu().numpy())
    np.testing.assert_array_equal(np.sort(idx, 1)[keep], np.sort(ref["idx"], 1)[keep])
    ref = with_gpu_choice(ref, idx, keep, lambda rows, ix: layer(tokens=rows, idx=ix))
    s = O.expert_scores(O.affinity_logits(c["x"], c["centroids"]), cfg.score_func)
    np.testing.assert_allclose(st["scores"].cpu().numpy(), s, atol=1e-5, rtol=0)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    np.testing.assert_array_equal(st["counts"].cpu().numpy(), counts)
    out = to_np(run.out)
    assert np.all(np.isfinite(out))
    assert rel_frob(out, ref["out"]) <= 1e-2
    # h holds [gate | up] of every row; act = SiLU(gate) * up from it
    x = O._f64(c["x"])
    perm = st["perm_tok"].cpu().numpy()
    off = st["offsets"].cpu().numpy()
    h = to_np(st["h"])
    act = to_np(st["act"])
    I = cfg.I
    for e in range(cfg.E):
        r = np.arange(off[e], off[e + 1])
        if r.size:
            want = x[perm[r]] @ O._f64(c["w13"][e]).T
            assert rel_frob(h[r], want) <= 1e-2
    for sx in range(cfg.S):
        r = cfg.T * cfg.K + sx * cfg.T + np.arange(cfg.T)
        assert rel_frob(h[r], x @ O._f64(c["ws13"][sx]).T) <= 1e-2
    hs = h[:, :I]
    want_act = hs / (1 + np.exp(-hs)) * h[:, I:]
    assert rel_frob(act, want_act) <= 1e-2


def test_backward_deterministic():
    cfg = small_cases()["ragged_bf16"]
    g, _ = gpu_inputs(cfg)
    a, dout = _run(cfg, g)
    b = TrainRun(cfg, g)
    b.forward()
    b.backward(dout)
    torch.cuda.synchronize()
    assert m.get_status() == 0
    for k in a.grads:
        assert torch.equal(a.grads[k], b.grads[k]), k


BWD_EDGE = {
    "bwd_one_token": small_cases()["ragged_bf16"].with_(name="bwd_one_token", T=1),
    "bwd_no_shared": small_cases()["ragged_bf16"].with_(name="bwd_no_shared", S=0),
    "bwd_k_equals_e": small_cases()["ragged_bf16"].with_(name="bwd_k_equals_e", E=8, K=8, T=100),
    "bwd_e1024_k32": small_cases()["ragged_bf16"].with_(name="bwd_e1024_k32", T=160, d=256,
                                                        E=1024, K=32, S=1, I=128),
    "bwd_many_tiles": small_cases()["small_bf16"].with_(name="bwd_many_tiles", T=700, d=1152,
                                                        E=16, K=4, S=2, I=640),
}


@pytest.mark.parametrize("name", list(BWD_EDGE))
def test_backward_edge_cases(name):
    cfg = BWD_EDGE[name]
    g, c = gpu_inputs(cfg)
    run, dout = _run(cfg, g)
    _check_against_oracle(cfg, run, c, dout, name)


def test_backward_hot_expert_long_k():
    """One expert chosen by every token: its weight-gradient tiles run K over
    the whole batch (many 64-token steps) and its input-gradient group spans
    many token blocks."""
    cfg = small_cases()["small_bf16"].with_(name="hot_bwd", T=1500, E=8, K=2)
    g, c = gpu_inputs(cfg)
    g["bias"] = torch.zeros(cfg.E, device="cuda")
    g["bias"][5] = 5.0
    c = dict(c)
    c["bias"] = g["bias"].cpu()
    run, dout = _run(cfg, g)
    assert int(run.state["counts"][5].item()) == cfg.T
    _check_against_oracle(cfg, run, c, dout, "hot expert")


def test_backward_token_block_boundaries():
    """Experts chosen by 1, 63, 64, 65, 383, 384, 385 and 449 tokens: either
    side of the 64-token K step of the weight gradients and of the 384 tokens
    of A they keep in shared memory.  The router is steered through its
    inputs: token t carries +8 on feature e for each of its two experts e and
    centroid e is 1 on feature e and 0 on the other first E features, so the
    chosen logits sit about 8 above the rest (whose random part has a
    standard deviation of about 0.6)."""
    counts = np.array([1, 63, 64, 65, 383, 384, 385, 449])
    idx = idx_with_counts(counts, 2, seed=3)
    cfg = small_cases()["ragged_bf16"].with_(name="bwd_blocks", T=len(idx), E=len(counts), K=2)
    E = cfg.E
    _, c = gpu_inputs(cfg)
    x = c["x"].clone()
    x[:, :E] = 0
    x[torch.arange(cfg.T).repeat_interleave(2), torch.as_tensor(idx.reshape(-1)).long()] = 8.0
    cen = c["centroids"].clone()
    cen[:, :E] = 0
    cen[torch.arange(E), torch.arange(E)] = 1.0
    c = dict(c, x=x, centroids=cen)
    g = {k: v.cuda() for k, v in c.items()}
    run, dout = _run(cfg, g)
    np.testing.assert_array_equal(np.sort(run.state["idx"].cpu().numpy(), 1), np.sort(idx, 1))
    np.testing.assert_array_equal(run.state["counts"].cpu().numpy(), counts)
    _check_against_oracle(cfg, run, c, dout, "block boundaries")


def test_backward_empty_batch_zeroes_gradients():
    cfg = small_cases()["small_bf16"]
    mc = m.cfg_from_layer(cfg, T=0)
    grads = m.alloc_grads(m.cfg_from_layer(cfg))
    for t in grads.values():
        t.fill_(1.0)
    g = make_inputs(cfg, "cuda")
    st = m.alloc_train_state(m.cfg_from_layer(cfg))
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    m.backward(mc, None, g["x"], g["centroids"], g["w13"], g["w2"], g["ws13"], g["ws2"], st,
               grads, ws)
    torch.cuda.synchronize()
    for k in ("dcentroids", "dw13", "dw2", "dws13", "dws2"):
        assert not grads[k].any(), k


def test_backward_v3_full_size_sampled():
    """The V3 prefill layer (T = 8192, d = 7168, E = 256, K = 8, I = 2048) in
    the launch configuration the benchmark times: weight gradients of two
    routed experts (the least and the most loaded) against the oracle on
    their rows, dx on a token sample, every gradient finite, unchosen
    experts zero."""
    cfg = get_config("v3_prefill")
    g = make_inputs(cfg, "cuda")
    run, dout = _run(cfg, g)
    st, gr = run.state, run.grads
    counts = st["counts"].cpu().numpy()
    assert counts.sum() == cfg.T * cfg.K
    for k in ("dx", "dcentroids"):
        assert torch.isfinite(gr[k].float()).all(), k
    idx = st["idx"].cpu().numpy()
    gates = st["gates"].cpu().numpy().astype(np.float64)
    dout_h = O._f64(dout)
    x = O._f64(g["x"])
    nz = np.nonzero(counts)[0]
    for e in (nz[np.argmin(counts[nz])], nz[np.argmax(counts[nz])]):
        rows, slots = np.nonzero(idx == e)
        dye = gates[rows, slots][:, None] * dout_h[rows]
        _, dw13, dw2 = O.swiglu_ffn_backward(x[rows], g["w13"][e].cpu(), g["w2"][e].cpu(), dye)
        assert_grad_close(to_np(gr["dw13"][e]), dw13, f"dw13[{e}]")
        assert_grad_close(to_np(gr["dw2"][e]), dw2, f"dw2[{e}]")
        # rounded where the kernels store: g * dout, h, act, da, dh, the outputs
        _, dw13r, dw2r = O.swiglu_ffn_backward(x[rows], g["w13"][e].cpu(), g["w2"][e].cpu(),
                                               O.round_bf16(dye), rnd=O.round_bf16)
        assert_grad_tight(to_np(gr["dw13"][e]), O.round_bf16(dw13r), f"dw13[{e}] rounded")
        assert_grad_tight(to_np(gr["dw2"][e]), O.round_bf16(dw2r), f"dw2[{e}] rounded")
    # dx on sampled tokens: their K experts, the shared expert, router and residual
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(cfg.T, 3, replace=False))
    host = {k: g[k].cpu() for k in ("centroids", "bias", "ws13", "ws2")}
    for t in toks:
        u = x[t:t + 1]
        it, gt, _, s = O.route(u, host["centroids"], host["bias"], cfg.K, cfg.score_func,
                               cfg.normalize)
        it = idx[t:t + 1]                      # the GPU's choice
        gt = O.gate_values(s, it, cfg.normalize)
        want = dout_h[t:t + 1].copy()
        dg = np.zeros((1, cfg.K))
        for k in range(cfg.K):
            e = int(it[0, k])
            w13, w2 = g["w13"][e].cpu(), g["w2"][e].cpu()
            dg[0, k] = float(np.sum(dout_h[t] * O.swiglu_ffn(u, w13, w2)[0]))
            want += O.swiglu_ffn_backward(u, w13, w2, gt[:, k:k + 1] * dout_h[t:t + 1])[0]
        for sx in range(cfg.S):
            want += O.swiglu_ffn_backward(u, host["ws13"][sx], host["ws2"][sx],
                                          dout_h[t:t + 1])[0]
        want += O.router_backward(u, host["centroids"], s, it, gt, dg, cfg.normalize,
                                  cfg.score_func)[0]
        assert_grad_close(to_np(gr["dx"][t:t + 1]), want, f"dx[{t}]")
    for e in np.nonzero(counts == 0)[0]:
        assert not gr["dw13"][e].any() and not gr["dw2"][e].any()
