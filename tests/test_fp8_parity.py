"""GPU parity of the FP8 layer (block-scaled e4m3 expert weights, V3
walk-through section 4.3) against the CPU oracle, through the C ABI.

The oracle runs the layer on the dequantised weights q * scale with the bf16
activations unquantised; the kernels also quantise the activations (1 x 128
tiles) and round act to e4m3, which is the whole of the looser tolerance:
relative Frobenius error <= 5e-2 on the MoE term.  Routing, counts, the
dispatch order and the bias update are integer results and must be exact.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from moe_inputs import small_cases, get_config, make_inputs, make_tokens
from oracle import moe_oracle as O
from tests._util import check_near_ties, gpu_inputs, idx_with_counts, rel_frob, with_gpu_choice

pytestmark = pytest.mark.gpu

m = pytest.importorskip("mixture_experts_layer_88_b300")

FP8_TOL = 5e-2
SMALL = [k for k, c in small_cases().items() if c.wgt == "e4m3"]


class Fp8Run:
    """Buffers and step-by-step calls of the FP8 path for one config."""

    def __init__(self, cfg, g, add_residual=0):
        self.lc = cfg
        self.cfg = m.cfg_from_layer(cfg)
        self.cfg.add_residual = add_residual
        self.g = g
        T, K, E, d, I = cfg.T, cfg.K, cfg.E, cfg.d, cfg.I
        self.rows_in, self.rows_out, self.shared_row = m.fp8_rows(self.cfg)
        dev = "cuda"
        self.idx = torch.full((T, K), -1, dtype=torch.int32, device=dev)
        self.gates = torch.zeros((T, K), dtype=torch.float32, device=dev)
        self.counts = torch.full((E,), -1, dtype=torch.int32, device=dev)
        self.offsets = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
        self.perm = torch.full((self.shared_row,), -1, dtype=torch.int32, device=dev)
        self.pos = torch.full((T, K), -1, dtype=torch.int32, device=dev)
        self.xq = torch.zeros((self.rows_in, d), dtype=torch.uint8, device=dev)
        self.xs = torch.zeros((d // 128, self.rows_in), dtype=torch.float32, device=dev)
        self.act = torch.zeros((self.rows_out, I), dtype=torch.uint8, device=dev)
        self.act_s = torch.zeros((I // 128, self.rows_out), dtype=torch.float32, device=dev)
        self.y = torch.zeros((self.rows_out, d), dtype=torch.bfloat16, device=dev)
        self.out = torch.zeros((T, d), dtype=torch.bfloat16, device=dev)
        self.w = m.fp8_weights(g)
        self.ws = {w: m.alloc_workspace(self.cfg, w) for w in
                   (m.MOE_WS_ROUTE, m.MOE_WS_DISPATCH, m.MOE_WS_EXPERTS, m.MOE_WS_FORWARD)}

    def route(self):
        g = self.g
        m.route(self.cfg, g["x"], g["centroids"], g["bias"], self.idx, self.gates,
                self.ws[m.MOE_WS_ROUTE])

    def dispatch(self, idx=None):
        m.dispatch_fp8(self.cfg, self.g["x"], self.idx if idx is None else idx, self.counts,
                       self.offsets, self.xq, self.xs, self.perm, self.pos,
                       self.ws[m.MOE_WS_DISPATCH])

    def experts(self):
        m.experts_fp8(self.cfg, self.xq, self.xs, self.offsets, self.counts, self.w, self.act,
                      self.act_s, self.y, self.ws[m.MOE_WS_EXPERTS])

    def combine(self):
        m.combine(self.cfg, self.y, self.gates, self.pos, self.g["x"], self.out)

    def forward(self, out=None):
        g = self.g
        m.forward_fp8(self.cfg, g["x"], g["centroids"], g["bias"], self.w, self.idx, self.gates,
                      self.counts, self.out if out is None else out, self.ws[m.MOE_WS_FORWARD])


def _oracle(cfg, c, tokens=None, idx=None, act_quant=False):
    return O.moe_layer(c, cfg.K, cfg.normalize, cfg.score_func, add_residual=0, tokens=tokens,
                       n_groups=cfg.n_groups, topk_groups=cfg.topk_groups, idx=idx,
                       act_quant=act_quant)


def _checked_ref(cfg, c, ref, idx_g, gates_g, tokens=None, act_quant=False):
    """Routing of the oracle's tokens (ref's rows) against the GPU's: chosen
    sets bit-exact where the K-th vs (K+1)-th margin is >= 1e-5, a valid top-K
    within 1e-5 (and its gates) elsewhere; returns ref with the near-tie rows
    recomputed on the GPU's choice, so every token's output is compared."""
    keep, n_excl = check_near_ties(cfg, idx_g, ref["margin"], ref["scores"], c["bias"], gates_g)
    if cfg.zipf_s == 0:
        assert n_excl <= max(2, len(keep) // 50)
    # Zipf-skewed layers: the most popular experts' Sigmoid scores round to
    # 1.0 in fp32, so their keys tie exactly and nearly every token is a near
    # tie; each is validated above and compared on its own choice below
    np.testing.assert_array_equal(np.sort(idx_g, 1)[keep], np.sort(ref["idx"], 1)[keep])
    tok = np.arange(len(keep)) if tokens is None else np.asarray(tokens)
    return with_gpu_choice(ref, idx_g, keep,
                           lambda rows, ix: _oracle(cfg, c, tokens=tok[rows], idx=ix,
                                                    act_quant=act_quant))


@pytest.mark.parametrize("name", SMALL)
def test_fp8_dispatch_rows_and_quantisation(name):
    """Counts and the order of each expert's rows are those of the oracle;
    offsets are the prefix sums of counts rounded up to 4 rows; every written
    row dequantises to its token within e4m3 rounding of its 1 x 128 tile."""
    cfg = small_cases()[name]
    g, c = gpu_inputs(cfg)
    run = Fp8Run(cfg, g)
    idx_o, _, _, _ = O.route(c["x"], c["centroids"], c["bias"], cfg.K, cfg.score_func,
                             cfg.normalize)
    run.dispatch(torch.as_tensor(idx_o, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert m.get_status() == 0
    counts, offsets, perm, pos = O.dispatch(idx_o, cfg.E)
    np.testing.assert_array_equal(run.counts.cpu().numpy(), counts)
    padded = np.concatenate([[0], np.cumsum((counts + 3) // 4 * 4)])
    got_off = run.offsets.cpu().numpy()
    np.testing.assert_array_equal(got_off, padded)
    gpos = run.pos.cpu().numpy()
    # row within the expert = oracle row within the expert
    np.testing.assert_array_equal(gpos - got_off[idx_o], pos - offsets[idx_o])
    gperm = run.perm.cpu().numpy()
    T = cfg.T
    np.testing.assert_array_equal(gperm[gpos.reshape(-1)], np.repeat(np.arange(T), cfg.K))
    # quantisation of every written row (routed rows and the shared-expert rows)
    xq = run.xq.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()
    xs = run.xs.double().cpu().numpy()
    x = O._f64(c["x"])
    rows = np.concatenate([gpos.reshape(-1), run.shared_row + np.arange(T)])
    toks = np.concatenate([np.repeat(np.arange(T), cfg.K), np.arange(T)])
    kb = np.arange(cfg.d) // 128
    deq = xq[rows] * xs[kb][:, rows].T
    ref = x[toks]
    tile_max = np.abs(ref).reshape(len(toks), -1, 128).max(axis=2)
    np.testing.assert_allclose(xs[:, rows].T, tile_max / 448.0, rtol=1e-6, atol=0)
    tol = np.abs(ref) * 2.0 ** -4 + np.repeat(tile_max / 448.0, 128, axis=1) * 2.0 ** -10
    assert np.all(np.abs(deq - ref) <= tol * (1 + 1e-5) + 1e-30)
    # the codes and scales themselves: the oracle's tile quantisation, bit for bit
    np.testing.assert_array_equal(deq, O.quantize_tiles_e4m3(ref))


@pytest.mark.parametrize("name", SMALL)
def test_fp8_layer_parity(name):
    cfg = small_cases()[name]
    g, c = gpu_inputs(cfg)
    run = Fp8Run(cfg, g)
    run.forward()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    idx = run.idx.cpu().numpy()
    ref = _checked_ref(cfg, c, _oracle(cfg, c), idx, run.gates.cpu().numpy())
    counts, _, _, _ = O.dispatch(idx, cfg.E)
    np.testing.assert_array_equal(run.counts.cpu().numpy(), counts)
    got = run.out.double().cpu().numpy()
    r = rel_frob(got, ref["delta"])
    assert r <= FP8_TOL, f"relative Frobenius {r:.3e}"


# The oracle that also quantises the activations (1 x 128 e4m3 tiles of the
# expert inputs and of the SwiGLU output, as the kernels do) leaves only the
# rounding of fp32 sums, of y to bf16, and rare e4m3 codes that fp32 partial
# sums put on the other side of a rounding boundary: the bf16 bar applies.
FP8Q_TOL = 1e-2


@pytest.mark.parametrize("name", SMALL)
def test_fp8_layer_parity_quantised_activations(name):
    cfg = small_cases()[name]
    g, c = gpu_inputs(cfg)
    run = Fp8Run(cfg, g)
    run.forward()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    ref = _checked_ref(cfg, c, _oracle(cfg, c, act_quant=True), run.idx.cpu().numpy(),
                       run.gates.cpu().numpy(), act_quant=True)
    got = run.out.double().cpu().numpy()
    r = rel_frob(got, ref["delta"])
    assert r <= FP8Q_TOL, f"relative Frobenius {r:.3e}"


@pytest.mark.parametrize("name", SMALL)
def test_fp8_stepwise_equals_forward(name):
    """route -> dispatch_fp8 -> experts_fp8 -> combine gives exactly the
    output of forward_fp8 (every step is deterministic)."""
    cfg = small_cases()[name]
    g, _ = gpu_inputs(cfg)
    run = Fp8Run(cfg, g)
    fwd = torch.zeros_like(run.out)
    run.forward(fwd)
    run.route()
    run.dispatch()
    run.experts()
    run.combine()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    assert torch.equal(run.out, fwd)


def test_fp8_hot_expert_many_token_blocks():
    """One expert chosen by every token: its group spans many token blocks."""
    cfg = small_cases()["small_fp8"].with_(name="hot_fp8", T=900, E=8, K=2)
    g, c = gpu_inputs(cfg)
    g["bias"] = torch.zeros(cfg.E, device="cuda")
    g["bias"][3] = 5.0
    c = dict(c)
    c["bias"] = g["bias"].cpu()
    run = Fp8Run(cfg, g)
    run.forward()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    assert int(run.counts[3].item()) == cfg.T
    idx, gates = run.idx.cpu().numpy(), run.gates.cpu().numpy()
    ref = _checked_ref(cfg, c, _oracle(cfg, c), idx, gates)
    got = run.out.double().cpu().numpy()
    assert rel_frob(got, ref["delta"]) <= FP8_TOL
    refq = _checked_ref(cfg, c, _oracle(cfg, c, act_quant=True), idx, gates, act_quant=True)
    assert rel_frob(got, refq["delta"]) <= FP8Q_TOL


def test_fp8_v3_skewed_full_size_sampled():
    """The Zipf-skewed V3 layer at full size (T=16384): routing and counts on
    every token, layer output on a token sample through the oracle."""
    cfg = get_config("v3_skewed_fp8")
    g = make_inputs(cfg, "cuda")
    run = Fp8Run(cfg, g)
    run.forward()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    idx = run.idx.cpu().numpy()
    counts, _, _, _ = O.dispatch(idx, cfg.E)
    np.testing.assert_array_equal(run.counts.cpu().numpy(), counts)
    assert counts.sum() == cfg.T * cfg.K
    # skew: the most popular expert takes (nearly) every token
    assert counts.max() >= 0.9 * cfg.T
    rng = np.random.default_rng(11)
    tok = np.sort(rng.choice(cfg.T, 48, replace=False))
    host = {k: g[k] for k in ("x", "centroids", "bias", "ws13", "ws13_scale", "ws2",
                              "ws2_scale")}
    host = {k: v.cpu() for k, v in host.items()}

    class _PerExpert:
        def __init__(self, t):
            self.t = t
            self.shape = t.shape

        def __getitem__(self, e):
            return self.t[int(e)].cpu()

    for k in ("w13", "w13_scale", "w2", "w2_scale"):
        host[k] = _PerExpert(g[k])
    ref = _checked_ref(cfg, host, _oracle(cfg, host, tokens=tok), idx[tok],
                       run.gates.cpu().numpy()[tok], tokens=tok)
    got = run.out[torch.as_tensor(tok, device="cuda")].double().cpu().numpy()
    assert rel_frob(got, ref["delta"]) <= FP8_TOL
    # against the oracle that quantises the activations as the kernels do
    refq = _checked_ref(cfg, host, _oracle(cfg, host, tokens=tok, act_quant=True), idx[tok],
                        run.gates.cpu().numpy()[tok], tokens=tok, act_quant=True)
    assert rel_frob(got, refq["delta"]) <= FP8Q_TOL


def test_fp8_bias_update_steps_skewed():
    """Balancing loop on the skewed FP8 layer (reduced width): 8 steps, each a
    fresh batch; the bias after every step equals the oracle's fp32 update from
    the step's counts, the counts equal the histogram of the step's routing,
    and the most loaded expert's bias only goes down."""
    cfg = small_cases()["small_fp8"].with_(name="skew_steps", T=1024)
    g, _ = gpu_inputs(cfg)
    mc = m.cfg_from_layer(cfg)
    layer = m.MoeLayer(mc, g, device="cuda", fp8_path="e4m3")
    bias_o = g["bias"].cpu().numpy().copy()
    hot = None
    for step in range(8):
        x = make_tokens(cfg, "cuda", step=step)
        layer.forward(x)
        stats = layer.update_bias()
        torch.cuda.synchronize()
        assert m.get_status() == 0
        idx = layer.idx.cpu().numpy()
        counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
        np.testing.assert_array_equal(layer.counts.cpu().numpy(), counts)
        bias_o, (mx, mn) = O.update_bias(counts, bias_o, cfg.T, cfg.K, cfg.gamma)
        np.testing.assert_array_equal(layer.bias.cpu().numpy().view(np.uint32),
                                      bias_o.view(np.uint32))
        assert abs(float(stats[0].item()) - mx) < 1e-5
        if hot is None:
            hot = int(np.argmax(counts))
    assert bias_o[hot] < 0


def test_fp8_token_block_boundaries():
    """Experts whose row counts sit on either side of the FP8 tiles' token
    block (160 rows) and of the 16-row MMA step, on a routing fixed by the
    test (K = 2) with the oracle's gates for it: dispatch -> experts ->
    combine against the oracle's layer."""
    counts = np.array([2, 16, 17, 159, 160, 161, 320, 321])
    idx = idx_with_counts(counts, 2, seed=5)
    cfg = small_cases()["ragged_fp8"].with_(name="fp8_blocks", T=len(idx), E=len(counts), K=2)
    g, c = gpu_inputs(cfg)
    ref = _oracle(cfg, c, idx=idx)
    run = Fp8Run(cfg, g)
    run.dispatch(torch.as_tensor(idx, device="cuda"))
    run.gates.copy_(torch.as_tensor(ref["gates"], dtype=torch.float32))
    run.experts()
    run.combine()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    np.testing.assert_array_equal(run.counts.cpu().numpy(), counts)
    got = run.out.double().cpu().numpy()
    assert rel_frob(got, ref["delta"]) <= FP8_TOL
    refq = _oracle(cfg, c, idx=idx, act_quant=True)      # same routing, same gates
    assert rel_frob(got, refq["delta"]) <= FP8Q_TOL


FP8_EDGE = {
    "fp8_one_token": small_cases()["ragged_fp8"].with_(name="fp8_one_token", T=1),
    "fp8_no_shared": small_cases()["ragged_fp8"].with_(name="fp8_no_shared", S=0),
    "fp8_k_equals_e": small_cases()["ragged_fp8"].with_(name="fp8_k_equals_e", E=8, K=8, T=100),
    "fp8_grouped": small_cases()["small_fp8"].with_(name="fp8_grouped", zipf_s=0.0, n_groups=4,
                                                    topk_groups=2),
    # the ABI's limits: E = 1024 with K = 32 (3E padding rows in the FP8 row layout)
    "fp8_e1024_k32": small_cases()["ragged_fp8"].with_(name="fp8_e1024_k32", T=160, d=256,
                                                       E=1024, K=32, S=1, I=128),
}


@pytest.mark.parametrize("name", list(FP8_EDGE))
def test_fp8_edge_cases(name):
    cfg = FP8_EDGE[name]
    g, c = gpu_inputs(cfg)
    run = Fp8Run(cfg, g)
    run.forward()
    torch.cuda.synchronize()
    assert m.get_status() == 0
    idx, gates = run.idx.cpu().numpy(), run.gates.cpu().numpy()
    ref = _checked_ref(cfg, c, _oracle(cfg, c), idx, gates)
    got = run.out.double().cpu().numpy()
    assert rel_frob(got, ref["delta"]) <= FP8_TOL
    refq = _checked_ref(cfg, c, _oracle(cfg, c, act_quant=True), idx, gates, act_quant=True)
    assert rel_frob(got, refq["delta"]) <= FP8Q_TOL
