"""Pins of the oracle's backward pass (``moe_layer_backward``) to things other
than itself: central finite differences of the forward oracle ``moe_layer``
(every entry of every input that has a gradient), Euler's identity for the
down projections (the layer is linear in each W2), and closed forms of the
router term.  Everything runs in fp64 on tiny layers, on the CPU.

The loss is L = sum(dout * out); its gradient with respect to any input is
what ``moe_layer_backward`` returns for that dout.  The chosen experts are
constants of the backward, so every finite-difference step must leave the
top-K choice unchanged; each case checks that.
"""
from __future__ import annotations

import numpy as np
import pytest

from oracle import moe_oracle as O

EPS = 1e-6


def _layer(T=5, d=6, E=8, I=4, S=1, seed=0):
    rng = np.random.default_rng(seed)
    return {
        "x": rng.normal(0, 1.0, (T, d)),
        "centroids": rng.normal(0, 0.5, (E, d)),
        "bias": rng.uniform(-0.05, 0.05, E).astype(np.float32),
        "w13": rng.normal(0, 0.5, (E, 2 * I, d)),
        "w2": rng.normal(0, 0.5, (E, d, I)),
        "ws13": rng.normal(0, 0.5, (S, 2 * I, d)),
        "ws2": rng.normal(0, 0.5, (S, d, I)),
    }


CASES = {
    "sigmoid_renorm_shared": dict(K=2, normalize=1, score_func=O.SIGMOID, add_residual=1, S=1),
    "sigmoid_plain_noshared": dict(K=3, normalize=0, score_func=O.SIGMOID, add_residual=0, S=0),
    "softmax_plain_2shared": dict(K=2, normalize=0, score_func=O.SOFTMAX, add_residual=1, S=2),
    "softmax_renorm": dict(K=3, normalize=1, score_func=O.SOFTMAX, add_residual=0, S=1),
    "grouped_sigmoid": dict(K=3, normalize=1, score_func=O.SIGMOID, add_residual=1, S=1,
                            n_groups=4, topk_groups=2),
}


def _loss(inp, dout, c):
    r = O.moe_layer(inp, c["K"], c["normalize"], c["score_func"], c["add_residual"],
                    n_groups=c.get("n_groups", 0), topk_groups=c.get("topk_groups", 0))
    return float(np.sum(dout * r["out"])), r["idx"]


@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_central_differences(name):
    c = CASES[name]
    inp = _layer(S=c["S"], seed=3)
    rng = np.random.default_rng(11)
    dout = rng.normal(0, 1.0, inp["x"].shape)
    g = O.moe_layer_backward(inp, c["K"], dout, c["normalize"], c["score_func"],
                             c["add_residual"], c.get("n_groups", 0), c.get("topk_groups", 0))
    assert np.min(g["margin"]) > 1e-4          # steps of 1e-6 leave the choice alone
    keys = {"x": "dx", "centroids": "dcentroids", "w13": "dw13", "w2": "dw2",
            "ws13": "dws13", "ws2": "dws2"}
    for key, gk in keys.items():
        want = g[gk]
        assert want.shape == inp[key].shape
        fd = np.zeros_like(want)
        for i in np.ndindex(*inp[key].shape):
            v0 = inp[key][i]
            inp[key][i] = v0 + EPS
            lp, ip = _loss(inp, dout, c)
            inp[key][i] = v0 - EPS
            lm, im = _loss(inp, dout, c)
            inp[key][i] = v0
            assert np.array_equal(ip, g["idx"]) and np.array_equal(im, g["idx"])
            fd[i] = (lp - lm) / (2 * EPS)
        scale = max(1.0, float(np.max(np.abs(want)))) if want.size else 1.0
        err = float(np.max(np.abs(fd - want))) if want.size else 0.0
        assert err <= 1e-6 * scale, f"{name} {gk}: max |fd - grad| = {err:.3e}"


@pytest.mark.parametrize("name", list(CASES))
def test_down_projection_euler_identity(name):
    """The layer is linear in each down projection (routing fixed), so
    sum_e <dW2_e, W2_e> + sum_s <dWs2_s, Ws2_s> = sum(dout * (out - residual))."""
    c = CASES[name]
    inp = _layer(T=7, d=8, E=8, I=6, S=c["S"], seed=5)
    dout = np.random.default_rng(2).normal(0, 1.0, inp["x"].shape)
    g = O.moe_layer_backward(inp, c["K"], dout, c["normalize"], c["score_func"],
                             c["add_residual"], c.get("n_groups", 0), c.get("topk_groups", 0))
    fwd = O.moe_layer(inp, c["K"], c["normalize"], c["score_func"], c["add_residual"],
                      n_groups=c.get("n_groups", 0), topk_groups=c.get("topk_groups", 0))
    lhs = float(np.sum(g["dw2"] * inp["w2"]) + np.sum(g["dws2"] * inp["ws2"]))
    rhs = float(np.sum(dout * fwd["delta"]))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs))


def test_single_renormalised_expert_has_no_router_gradient():
    """K = 1 with renormalisation: the gate is identically 1, so the centroids
    get zero gradient and the tokens get only the expert and residual terms."""
    inp = _layer(T=6, d=5, E=4, I=3, S=1, seed=7)
    dout = np.random.default_rng(4).normal(0, 1.0, inp["x"].shape)
    g = O.moe_layer_backward(inp, 1, dout, 1, O.SIGMOID, 1)
    assert np.all(g["dcentroids"] == 0.0)
    assert np.all(g["dlogit"] == 0.0)
    assert np.all(g["gates"] == 1.0)


def test_router_term_closed_form_one_expert_unnormalised():
    """E = K = 1, no renormalisation, no shared expert, no residual:
    out = sig(x.c) FFN(x), so dL/dc = sum_t (dout_t . FFN(x_t)) sig'(x_t.c) x_t."""
    inp = _layer(T=4, d=5, E=1, I=3, S=0, seed=9)
    dout = np.random.default_rng(6).normal(0, 1.0, inp["x"].shape)
    g = O.moe_layer_backward(inp, 1, dout, 0, O.SIGMOID, 0)
    x = inp["x"]
    z = x @ inp["centroids"][0]
    sg = 1.0 / (1.0 + np.exp(-z))
    w13, w2 = inp["w13"][0], inp["w2"][0]
    h = x @ w13.T
    y = (h[:, :3] / (1.0 + np.exp(-h[:, :3])) * h[:, 3:]) @ w2.T
    want = ((np.sum(dout * y, axis=1) * sg * (1 - sg))[:, None] * x).sum(axis=0)
    np.testing.assert_allclose(g["dcentroids"][0], want, rtol=1e-12, atol=1e-14)


def test_unchosen_experts_get_zero_weight_gradients():
    inp = _layer(T=2, d=4, E=8, I=2, S=0, seed=1)
    dout = np.ones_like(inp["x"])
    g = O.moe_layer_backward(inp, 1, dout, 1, O.SIGMOID, 1)
    chosen = set(np.unique(g["idx"]).tolist())
    for e in range(8):
        if e not in chosen:
            assert not g["dw13"][e].any() and not g["dw2"][e].any()


def test_given_choice_reproduces_router_choice():
    """Passing the router's own choice back in changes nothing."""
    inp = _layer(T=6, d=6, E=8, I=4, S=1, seed=12)
    dout = np.random.default_rng(8).normal(0, 1.0, inp["x"].shape)
    a = O.moe_layer_backward(inp, 3, dout, 1, O.SIGMOID, 1)
    b = O.moe_layer_backward(inp, 3, dout, 1, O.SIGMOID, 1, idx=a["idx"])
    for k in ("dx", "dcentroids", "dw13", "dw2", "dws13", "dws2", "dgates"):
        np.testing.assert_array_equal(a[k], b[k])


def test_stored_rounding_backward():
    """stored_rounding=True rounds the stored values to bf16: dx and the
    weight gradients come out as bf16 values within a few bf16 steps of the
    unrounded gradients; dgates use the rounded y of the training forward,
    and the centroid gradients stay unrounded fp64."""
    inp = _layer(T=16, d=128, E=8, I=64, S=1, seed=21)
    for k in ("x", "centroids", "w13", "w2", "ws13", "ws2"):
        inp[k] = O.round_bf16(inp[k] * 0.2)
    dout = O.round_bf16(np.random.default_rng(4).normal(0, 1.0, inp["x"].shape))
    a = O.moe_layer_backward(inp, 2, dout, 1, O.SIGMOID, 1)
    b = O.moe_layer_backward(inp, 2, dout, 1, O.SIGMOID, 1, idx=a["idx"], stored_rounding=True)
    for k in ("dx", "dw13", "dw2", "dws13", "dws2"):
        assert np.array_equal(O.round_bf16(b[k]), b[k]), k
        rel = np.linalg.norm(b[k] - a[k]) / np.linalg.norm(a[k])
        assert 2.0 ** -16 < rel < 2.0 ** -6, (k, rel)
    assert not np.array_equal(a["dgates"], b["dgates"])
    assert not np.array_equal(O.round_bf16(b["dcentroids"]), b["dcentroids"])
