"""Pins for the CPU oracle: hand-worked golden values, closed forms, brute force
and invariants that the DeepSeekMoE pages fix.  CPU only."""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle import moe_oracle as O
from moe_inputs import small_cases, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

_NS = {"LN3": math.log(3.0), "LN9": math.log(9.0),
       "S2": 1.0 / (1.0 + math.exp(-2.0)), "__builtins__": {}}


def _num(tok):
    return float(eval(tok, _NS))  # fixture tokens are small arithmetic expressions


def _rows(text, conv=_num):
    return [[conv(t) for t in r.split()] for r in text.split("|")]


def _read(name):
    lines = []
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                k, v = ln.split(":", 1)
                lines.append((k.strip(), v.strip()))
    return lines


# ---------------------------------------------------------------- golden cases

def test_golden_routing():
    lines = _read("routing_hand.txt")
    kv = dict(lines[:2])
    C = np.array(_rows(kv["centroids"]))
    X = np.array(_rows(kv["x"]))
    cases = [v for k, v in lines if k == "case"]
    idxs = [v for k, v in lines if k == "idx"]
    gates = [v for k, v in lines if k == "gates"]
    assert len(cases) == 3
    for case, ii, gg in zip(cases, idxs, gates):
        bias_txt, norm_txt = case[len("bias="):].split(" normalize=")
        bias = np.array([float(t) for t in bias_txt.split()], dtype=np.float32)
        norm = int(norm_txt)
        idx, g, margin, _ = O.route(X, C, bias, 2, O.SIGMOID, norm)
        np.testing.assert_array_equal(idx, np.array(_rows(ii, int)))
        np.testing.assert_allclose(g, np.array(_rows(gg)), rtol=0, atol=1e-12)


def test_golden_dispatch():
    kv = dict(_read("dispatch_hand.txt"))
    E = int(kv["E"])
    idx = np.array(_rows(kv["idx"], int), dtype=np.int32)
    counts, offsets, perm, pos = O.dispatch(idx, E)
    np.testing.assert_array_equal(counts, [int(t) for t in kv["counts"].split()])
    np.testing.assert_array_equal(offsets, [int(t) for t in kv["offsets"].split()])
    np.testing.assert_array_equal(perm, [int(t) for t in kv["perm_tok"].split()])
    np.testing.assert_array_equal(pos, np.array(_rows(kv["pos"], int)))


def test_golden_bias_update():
    kv = dict(_read("bias_update_hand.txt"))
    counts = [int(t) for t in kv["counts"].split()]
    bias = np.array([float(t) for t in kv["bias_in"].split()], dtype=np.float32)
    b, stats = O.update_bias(counts, bias, int(kv["T"]), int(kv["K"]), float(kv["gamma"]))
    want = np.array([int(h, 16) for h in kv["bias_out_f32hex"].split()], dtype=np.uint32)
    np.testing.assert_array_equal(b.view(np.uint32), want)
    np.testing.assert_allclose(stats, [float(t) for t in kv["load_stats"].split()])


def test_golden_swiglu():
    kv = dict(_read("swiglu_hand.txt"))
    u = np.array([_rows(kv["u"])[0]])
    w13 = np.array(_rows(kv["w13"]))
    w2 = np.array(_rows(kv["w2"]))
    y = O.swiglu_ffn(u, w13, w2)
    np.testing.assert_allclose(y[0], _rows(kv["y"])[0], rtol=0, atol=1e-14)


def test_golden_layer_two_distinct_experts():
    """The gate of each chosen expert multiplies that expert's own output
    (V3 walk-through, section 3.1 with eqs. (13)-(15)): a hand-worked layer
    whose two chosen experts differ and whose gates are unequal."""
    kv = dict(_read("layer_two_experts_hand.txt"))
    w13 = np.array([_rows(kv[f"w13_{e}"]) for e in range(3)])
    w2 = np.array([_rows(kv[f"w2_{e}"]) for e in range(3)])
    inp = {"x": np.array(_rows(kv["x"])), "centroids": np.array(_rows(kv["centroids"])),
           "bias": np.zeros(3, np.float32), "w13": w13, "w2": w2,
           "ws13": np.zeros((0, 2, 2)), "ws2": np.zeros((0, 2, 1))}
    r = O.moe_layer(inp, 2, normalize=1, add_residual=0)
    np.testing.assert_array_equal(r["idx"], np.array(_rows(kv["idx"], int)))
    np.testing.assert_allclose(r["gates"], np.array(_rows(kv["gates"])), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["delta"], np.array(_rows(kv["out"])), rtol=0, atol=1e-12)
    # the same choice given explicitly reproduces the layer exactly
    r2 = O.moe_layer(inp, 2, normalize=1, add_residual=0, idx=r["idx"])
    np.testing.assert_array_equal(r2["delta"], r["delta"])
    assert np.all(np.isnan(r2["margin"]))
    # another (valid-looking) choice gives that choice's gates and outputs:
    # token 0 on experts 1 and 0 (same set, other listing order) is unchanged
    # up to the slot order; on experts 0 and 2 it uses expert 2's output
    r3 = O.moe_layer(inp, 2, normalize=1, add_residual=0, idx=np.array([[1, 0], [2, 1]]))
    np.testing.assert_allclose(r3["delta"], r["delta"], rtol=0, atol=1e-14)
    r4 = O.moe_layer(inp, 2, normalize=1, add_residual=0, idx=np.array([[0, 2], [2, 1]]))
    assert not np.allclose(r4["delta"][0], r["delta"][0])


# ---------------------------------------------------------------- brute force

def _brute_topk(keys_row, K):
    """The unique K-subset S with: every chosen i beats every unchosen j
    (key_i > key_j, or equal keys and i < j).  Enumerates all C(E, K) subsets."""
    E = len(keys_row)
    good = []
    for S in itertools.combinations(range(E), K):
        Sset = set(S)
        ok = all(keys_row[i] > keys_row[j] or (keys_row[i] == keys_row[j] and i < j)
                 for i in Sset for j in range(E) if j not in Sset)
        if ok:
            good.append(S)
    assert len(good) == 1
    return set(good[0])


@pytest.mark.parametrize("E,K", [(6, 1), (6, 3), (8, 4), (7, 7), (10, 2)])
def test_topk_brute_force(E, K):
    rng = np.random.default_rng(E * 10 + K)
    for trial in range(40):
        # quantised keys force many exact ties
        keys = (rng.integers(0, 5, size=(1, E)) / 4.0).astype(np.float32)
        idx, margin = O.select_topk(keys, K)
        assert set(idx[0].tolist()) == _brute_topk(keys[0].tolist(), K)
        # listed by descending key, ties by ascending index
        ks = keys[0][idx[0]]
        for a in range(K - 1):
            assert ks[a] > ks[a + 1] or (ks[a] == ks[a + 1] and idx[0][a] < idx[0][a + 1])
        if K == E:
            assert margin[0] == np.inf
        else:
            rest = [keys[0][j] for j in range(E) if j not in set(idx[0].tolist())]
            assert margin[0] == pytest.approx(float(ks[-1]) - float(max(rest)))


def test_topk_k1_is_argmax():
    rng = np.random.default_rng(3)
    keys = rng.standard_normal((50, 13)).astype(np.float32)
    idx, _ = O.select_topk(keys, 1)
    np.testing.assert_array_equal(idx[:, 0], np.argmax(keys, axis=1))


# ---------------------------------------------------------------- closed forms / invariants

def test_sigmoid_scores_closed_form():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((4, 6)) * 3
    s = O.expert_scores(L, O.SIGMOID)
    for t in range(4):
        for i in range(6):
            assert s[t, i] == pytest.approx(1.0 / (1.0 + math.exp(-L[t, i])), rel=1e-14)


def test_softmax_scores_match_scipy_and_norenorm_sum_below_one():
    rng = np.random.default_rng(6)
    L = rng.standard_normal((30, 64))
    s = O.expert_scores(L, O.SOFTMAX)
    np.testing.assert_allclose(s, scipy.special.softmax(L, axis=1), rtol=1e-12)
    keys = O.selection_keys(s, np.zeros(64, np.float32))
    idx, _ = O.select_topk(keys, 6)
    g = O.gate_values(s, idx, normalize=0)
    assert np.all(g.sum(axis=1) < 1.0)          # 2024 variant: sum generally < 1
    np.testing.assert_allclose(g, np.take_along_axis(scipy.special.softmax(L, axis=1), idx,
                                                     axis=1), rtol=1e-12)


@pytest.mark.parametrize("name", ["small_bf16", "ragged_bf16", "softmax_norenorm",
                                  "sigmoid_norenorm", "wide_e"])
def test_routing_invariants(name):
    cfg = small_cases()[name]
    inp = make_inputs(cfg, "cpu")
    idx, g, margin, s = O.route(inp["x"], inp["centroids"], inp["bias"], cfg.K,
                                cfg.score_func, cfg.normalize)
    T, K, E = cfg.T, cfg.K, cfg.E
    assert idx.shape == (T, K)
    assert np.all((idx >= 0) & (idx < E))
    assert all(len(set(r.tolist())) == K for r in idx)     # K distinct experts, no drop
    if cfg.normalize:
        np.testing.assert_allclose(g.sum(axis=1), 1.0, atol=1e-12)
    else:
        np.testing.assert_array_equal(g, np.take_along_axis(s, idx.astype(np.int64), 1))
    counts, offsets, perm, pos = O.dispatch(idx, E)
    assert counts.sum() == T * K
    assert offsets[0] == 0 and offsets[-1] == T * K
    np.testing.assert_array_equal(np.diff(offsets), counts)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)                      # ascending token order
        assert np.all((idx[seg] == e).sum(axis=1) == 1)      # each row's token chose e
    for t in range(T):
        for k in range(K):
            assert perm[pos[t, k]] == t
            assert offsets[idx[t, k]] <= pos[t, k] < offsets[idx[t, k] + 1]


def test_bias_changes_selection_not_gates():
    cfg = small_cases()["small_bf16"]
    inp = make_inputs(cfg, "cpu")
    x, C = inp["x"], inp["centroids"]
    idx0, g0, margin, s = O.route(x, C, np.zeros(cfg.E, np.float32), cfg.K)
    # a bias far smaller than every margin leaves the selection and the gates alone
    tiny = (np.arange(cfg.E, dtype=np.float32) - cfg.E / 2) * np.float32(1e-9)
    keep = margin > 1e-6
    idx1, g1, _, _ = O.route(x, C, tiny, cfg.K)
    np.testing.assert_array_equal(idx1[keep], idx0[keep])
    np.testing.assert_array_equal(g1[keep], g0[keep])
    # a large bias on expert 5 forces it into every token's set, at its own score
    big = np.zeros(cfg.E, np.float32)
    big[5] = 10.0
    idx2, g2, _, s2 = O.route(x, C, big, cfg.K)
    assert np.all(idx2[:, 0] == 5)
    chosen = np.take_along_axis(s2, idx2.astype(np.int64), 1)
    np.testing.assert_allclose(g2[:, 0], s2[:, 5] / chosen.sum(axis=1), rtol=1e-13)


def test_update_bias_direction():
    rng = np.random.default_rng(9)
    E, T, K = 32, 100, 8
    for trial in range(20):
        idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
        counts = np.bincount(idx.reshape(-1), minlength=E)
        b0 = rng.uniform(-0.01, 0.01, E).astype(np.float32)
        b1, (mx, mn) = O.update_bias(counts, b0, T, K, 1e-3)
        mean = T * K / E
        for e in range(E):
            if counts[e] > mean:
                assert b1[e] < b0[e]
            elif counts[e] < mean:
                assert b1[e] > b0[e]
            else:
                assert b1[e] == b0[e]
        assert mx == pytest.approx(counts.max() / mean) and mn == pytest.approx(counts.min()
                                                                                / mean)


# ---------------------------------------------------------------- expert / combine special cases

def _dense_swiglu_torch(u, w13, w2):
    """Independent dense SwiGLU via torch.nn.functional, fp64."""
    u = torch.as_tensor(u, dtype=torch.float64)
    w13 = torch.as_tensor(w13, dtype=torch.float64)
    w2 = torch.as_tensor(w2, dtype=torch.float64)
    I = w13.shape[0] // 2
    gate = F.linear(u, w13[:I])
    up = F.linear(u, w13[I:])
    return F.linear(F.silu(gate) * up, w2).numpy()


def test_identical_experts_reduce_to_dense_ffn():
    """With every routed expert identical and renormalised gates, the routed sum
    is the dense FFN itself (sum of gates is 1), plus shared, plus u."""
    cfg = small_cases()["ragged_bf16"]
    inp = make_inputs(cfg, "cpu")
    inp = dict(inp)
    inp["w13"] = inp["w13"][:1].expand(cfg.E, -1, -1)
    inp["w2"] = inp["w2"][:1].expand(cfg.E, -1, -1)
    res = O.moe_layer(inp, cfg.K, normalize=1)
    u = inp["x"].double().numpy()
    want = u + _dense_swiglu_torch(u, inp["w13"][0], inp["w2"][0])
    for s in range(cfg.S):
        want += _dense_swiglu_torch(u, inp["ws13"][s], inp["ws2"][s])
    np.testing.assert_allclose(res["out"], want, rtol=1e-10, atol=1e-12)


def test_zero_routed_down_gives_shared_plus_residual():
    cfg = small_cases()["softmax_norenorm"]
    inp = dict(make_inputs(cfg, "cpu"))
    inp["w2"] = torch.zeros_like(inp["w2"])
    for resid in (0, 1):
        res = O.moe_layer(inp, cfg.K, cfg.normalize, cfg.score_func, add_residual=resid)
        u = inp["x"].double().numpy()
        want = sum(_dense_swiglu_torch(u, inp["ws13"][s], inp["ws2"][s]) for s in range(cfg.S))
        if resid:
            want = want + u
        np.testing.assert_allclose(res["out"], want, rtol=1e-10, atol=1e-12)


def test_routed_combine_weights_by_gate():
    """A single routed expert (E=K=1) with renorm has gate exactly 1; with
    no renorm the gate is its Sigmoid score."""
    rng = np.random.default_rng(11)
    d, I = 8, 4
    inp = {"x": rng.standard_normal((5, d)), "centroids": rng.standard_normal((1, d)),
           "bias": np.zeros(1, np.float32), "w13": rng.standard_normal((1, 2 * I, d)),
           "w2": rng.standard_normal((1, d, I)), "ws13": np.zeros((0, 2 * I, d)),
           "ws2": np.zeros((0, d, I))}
    dense = _dense_swiglu_torch(inp["x"], inp["w13"][0], inp["w2"][0])
    r1 = O.moe_layer(inp, 1, normalize=1, add_residual=0)
    np.testing.assert_allclose(r1["out"], dense, rtol=1e-12)
    r0 = O.moe_layer(inp, 1, normalize=0, add_residual=0)
    sig = 1.0 / (1.0 + np.exp(-(inp["x"] @ inp["centroids"][0])))
    np.testing.assert_allclose(r0["out"], dense * sig[:, None], rtol=1e-12)


def test_token_subset_equals_full_batch():
    cfg = small_cases()["small_bf16"]
    inp = make_inputs(cfg, "cpu")
    full = O.moe_layer(inp, cfg.K)
    tok = [0, 7, 100, 511, 250]
    sub = O.moe_layer(inp, cfg.K, tokens=tok)
    np.testing.assert_array_equal(sub["idx"], full["idx"][tok])
    np.testing.assert_allclose(sub["out"], full["out"][tok], rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- FP8 weights

def _read_fp8_fixture():
    codes, elems, scale = [], [], None
    with open(os.path.join(GOLDEN, "fp8_dequant_hand.txt")) as f:
        for ln in f:
            ln = ln.strip()
            if not ln or ln.startswith("#"):
                continue
            key, rest = ln.split(":", 1)
            if key == "code":
                b, v = rest.split()
                codes.append((int(b, 16), float(v)))
            elif key == "scale":
                scale = [[float(v) for v in row.split()] for row in rest.split("|")]
            elif key == "elem":
                r, c, b, v = rest.split()
                elems.append((int(r), int(c), int(b, 16), float(v)))
    return codes, np.array(scale), elems


def test_golden_fp8_codes_decode():
    """The oracle's upcast of e4m3 codes gives the values the E4M3 definition fixes."""
    codes, _, _ = _read_fp8_fixture()
    bits = torch.tensor([b for b, _ in codes], dtype=torch.uint8).view(torch.float8_e4m3fn)
    got = O._f64(bits)
    want = np.array([v for _, v in codes])
    assert np.array_equal(got, want)


def test_golden_fp8_block_scales():
    """dequantize_blocks applies the scale of each element's own 128 x 128 block."""
    _, scale, elems = _read_fp8_fixture()
    q = torch.zeros((256, 256), dtype=torch.uint8)
    for r, c, b, _ in elems:
        q[r, c] = b
    w = O.dequantize_blocks(q.view(torch.float8_e4m3fn), scale)
    for r, c, _, v in elems:
        assert w[r, c] == v, (r, c, w[r, c], v)
    mask = np.ones((256, 256), bool)
    for r, c, _, _ in elems:
        mask[r, c] = False
    assert np.all(w[mask] == 0.0)


# ---------------------------------------------------------------- stored rounding

def test_stored_rounding_points():
    """moe_layer(stored_rounding=True) rounds each expert's SwiGLU output and
    output rows, and the layer output, to the activation type: the outputs are
    bf16 values, within a few bf16 steps of the unrounded layer, and distinct
    from an expert that skips the rounding of its SwiGLU output."""
    cfg = small_cases()["ragged_bf16"]
    inp = make_inputs(cfg, "cpu")
    exact = O.moe_layer(inp, cfg.K, add_residual=0)
    rnd = O.moe_layer(inp, cfg.K, add_residual=0, act="bf16", stored_rounding=True)
    assert np.array_equal(O.round_bf16(rnd["delta"]), rnd["delta"])
    rel = np.linalg.norm(rnd["delta"] - exact["delta"]) / np.linalg.norm(exact["delta"])
    assert 2.0 ** -14 < rel < 2.0 ** -6, rel
    u = O._f64(inp["x"])
    w13, w2 = inp["w13"][0], inp["w2"][0]
    y = O.swiglu_ffn(u, w13, w2, stored="bf16")
    assert np.array_equal(O.round_bf16(y), y)
    I = cfg.I
    h = u @ O._f64(w13).T
    y_no_act_rounding = O.round_bf16((O.silu(h[:, :I]) * h[:, I:]) @ O._f64(w2).T)
    assert np.any(y != y_no_act_rounding)
    # fp32 layers round to fp32
    tiny = small_cases()["tiny_f32_ragged"]
    t_in = make_inputs(tiny, "cpu")
    t_out = O.moe_layer(t_in, tiny.K, add_residual=0, act="f32", stored_rounding=True)["delta"]
    assert np.array_equal(t_out.astype(np.float32).astype(np.float64), t_out)


def test_dequant_round_weights():
    """dequant_round='bf16' turns each dequantised FP8 weight q * scale into the
    nearest bf16 value (the dequantisation itself is pinned by the FP8
    fixture); the layer moves by the size of that rounding."""
    cfg = small_cases()["ragged_fp8"]
    inp = make_inputs(cfg, "cpu")
    w = O._expert_weight(inp, "w13", 3)
    wr = O._expert_weight(inp, "w13", 3, dequant_round="bf16")
    assert np.array_equal(O.round_bf16(w), wr) and not np.array_equal(w, wr)
    assert np.all(np.abs(wr - w) <= 2.0 ** -8 * np.abs(w))
    a = O.moe_layer(inp, cfg.K, add_residual=0)["delta"]
    b = O.moe_layer(inp, cfg.K, add_residual=0, dequant_round="bf16")["delta"]
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 2.0 ** -14 < rel < 2.0 ** -7, rel


# ---------------------------------------------------------------- FP8 activation quantisation

def _read_e4m3_fixture():
    rounds, tiles = [], []
    with open(os.path.join(GOLDEN, "e4m3_round_hand.txt")) as f:
        for ln in f:
            ln = ln.strip()
            if not ln or ln.startswith("#"):
                continue
            key, rest = ln.split(":", 1)
            parts = rest.split()
            if key == "round":
                rounds.append((float(parts[0]), float(parts[1])))
            elif key == "tile":
                vals = [float(v) for v in parts[1].split(",")]
                codes = [float(v) for v in parts[2].split(",")]
                if "/" in parts[3]:
                    num, den = parts[3].split("/")
                    scale = np.float32(float(num)) / np.float32(float(den))
                else:
                    scale = np.float32(float(parts[3]))
                tiles.append((parts[0], vals, codes, float(scale)))
    return rounds, tiles


def test_golden_e4m3_rounding():
    """round_e4m3 gives the hand-worked values: ties to the even mantissa,
    subnormals, the binade carry and saturation at 448."""
    rounds, _ = _read_e4m3_fixture()
    got = O.round_e4m3(np.array([x for x, _ in rounds]))
    want = np.array([y for _, y in rounds])
    assert np.array_equal(got, want), np.stack([got, want], 1)[got != want]


def test_round_e4m3_matches_torch_cast():
    """round_e4m3 against torch's float32 -> float8_e4m3fn conversion (round to
    nearest even) on every finite e4m3 value, every midpoint between two of
    them, the float32 neighbours of both, and random values over 18 binades;
    all within +-448 (the torch cast does not saturate above)."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    vals = codes[torch.isfinite(codes)].double().unique().numpy()
    pos = vals[vals >= 0]
    pts = np.concatenate([pos, (pos[:-1] + pos[1:]) / 2]).astype(np.float32)
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)),
                          np.nextafter(pts, np.float32(-np.inf))])
    rng = np.random.default_rng(0)
    rnd = (rng.standard_normal(100000) * np.exp(rng.uniform(-12, 6, 100000))).astype(np.float32)
    v = np.concatenate([pts, -pts, rnd])
    v = v[np.abs(v) <= 448]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).double().numpy()
    got = O.round_e4m3(v.astype(np.float64))
    assert np.array_equal(got, want), v[got != want][:8]


def test_golden_e4m3_tiles():
    """quantize_tiles_e4m3 on the hand-worked tiles: codes times the fp32 scale."""
    _, tiles = _read_e4m3_fixture()
    for name, vals, codes, scale in tiles:
        v = np.zeros((1, 128), dtype=np.float32)
        v[0, :len(vals)] = vals
        got = O.quantize_tiles_e4m3(v.astype(np.float64))
        want = np.zeros(128)
        want[:len(codes)] = np.array(codes) * scale
        assert np.array_equal(got[0], want), (name, got[0, :len(codes)], want[:len(codes)])


def test_quantize_tiles_e4m3_properties():
    """Each 1 x 128 tile independently: its largest magnitude maps to the code
    448 and comes back within fp32 rounding; every value comes back within half
    an e4m3 step; scaling a tile by 2^k scales its result by exactly 2^k; an
    all-zero tile stays zero."""
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((16, 384)) * np.exp(rng.uniform(-3, 3, (16, 3))).repeat(128, 1))
    v = v.astype(np.float32).astype(np.float64)
    q = O.quantize_tiles_e4m3(v)
    t, qt = v.reshape(16, 3, 128), q.reshape(16, 3, 128)
    amax = np.abs(t).max(axis=2)
    imax = np.abs(t).argmax(axis=2)
    back = np.take_along_axis(qt, imax[..., None], 2)[..., 0]
    assert np.all(np.abs(np.abs(back) - amax) <= 2.0 ** -20 * amax)
    s = amax[..., None] / 448.0
    assert np.all(np.abs(qt - t) <= 2.0 ** -4 * np.abs(t) + 2.0 ** -10 * s * (1 + 1e-6))
    for k in (-8, -3, 1, 7):
        assert np.array_equal(O.quantize_tiles_e4m3(v * 2.0 ** k), q * 2.0 ** k), k
    z = v.copy()
    z[:, 128:256] = 0.0
    qz = O.quantize_tiles_e4m3(z)
    assert not np.any(qz[:, 128:256])
    assert np.array_equal(qz[:, :128], q[:, :128]) and np.array_equal(qz[:, 256:], q[:, 256:])


def test_swiglu_ffn_fp8_quantises_input_and_swiglu_output():
    """swiglu_ffn_fp8 differs from the unquantised expert by what the two
    e4m3 roundings explain (between 2^-12 and 2^-3 of the output's norm), and
    from each variant that leaves one of the two activations unquantised by
    more than rounding noise: neither quantisation step is missing."""
    rng = np.random.default_rng(9)
    d, I, n = 256, 256, 12
    u = rng.standard_normal((n, d)).astype(np.float32).astype(np.float64)
    w13 = rng.standard_normal((2 * I, d)) * 0.05
    w2 = rng.standard_normal((d, I)) * 0.05
    y = O.swiglu_ffn_fp8(u, w13, w2)
    ref = O.swiglu_ffn(u, w13, w2)
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert 2.0 ** -12 < rel < 2.0 ** -3, rel
    h = O.quantize_tiles_e4m3(u) @ w13.T
    only_in = (O.silu(h[:, :I]) * h[:, I:]) @ w2.T
    h0 = u @ w13.T
    only_out = O.quantize_tiles_e4m3(O.silu(h0[:, :I]) * h0[:, I:]) @ w2.T
    for other in (only_in, only_out):
        assert np.linalg.norm(y - other) > 1e-6 * np.linalg.norm(ref)


def test_fp8_layer_equals_layer_on_dequantised_weights():
    """An FP8 layer is the same layer on the weights q * scale (the activations
    enter unquantised): the oracle's FP8 path agrees bit for bit with its
    plain path fed the dequantised fp64 weights."""
    cfg = small_cases()["ragged_fp8"]
    inp = make_inputs(cfg, "cpu")
    plain = {k: inp[k] for k in ("x", "centroids", "bias")}
    for k in ("w13", "w2", "ws13", "ws2"):
        plain[k] = np.stack([O.dequantize_blocks(inp[k][e], inp[k + "_scale"][e])
                             for e in range(inp[k].shape[0])])
    a = O.moe_layer(inp, cfg.K, cfg.normalize, cfg.score_func, add_residual=0)
    b = O.moe_layer(plain, cfg.K, cfg.normalize, cfg.score_func, add_residual=0)
    assert np.array_equal(a["delta"], b["delta"])
    assert np.array_equal(a["idx"], b["idx"])


def test_fp8_generator_round_trip():
    """Generator check: q * scale reproduces the fp32 draw within e4m3 rounding
    (relative 2^-4, or 2^-10 * scale in the subnormal range), and every block's
    largest |q| is 448."""
    from moe_inputs.gen import _quantize_blocks
    g = torch.Generator().manual_seed(3)
    w = torch.randn((2, 256, 384), generator=g) * 0.01
    q, sc = _quantize_blocks(w)
    deq = O.dequantize_blocks(q[1], sc[1])
    ref = w[1].double().numpy()
    tol = np.abs(ref) * 2.0 ** -4 + np.repeat(np.repeat(sc[1].double().numpy(), 128, 0), 128, 1) * 2.0 ** -10
    assert np.all(np.abs(deq - ref) <= tol * (1 + 1e-6))
    qa = q.float().abs().reshape(2, 2, 128, 3, 128).amax(dim=(2, 4))
    assert torch.all(qa == 448.0)


def test_zipf_targets_capped_and_sum_to_k():
    from moe_inputs.gen import zipf_targets
    f = zipf_targets(256, 8, 1.1)
    assert abs(float(f.sum()) - 8.0) < 1e-9 and float(f.max()) <= 1.0 + 1e-12
    free = f < 1.0 - 1e-12
    r = torch.arange(1, 257, dtype=torch.float64)[free]
    ratio = f[free] * r ** 1.1
    assert float(ratio.max() - ratio.min()) < 1e-9 * float(ratio.max())


# ---------------------------------------------------------------- node-limited routing

def test_golden_group_limited_routing():
    with open(os.path.join(GOLDEN, "routing_groups_hand.txt")) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]
    sv = np.array([[float(v) for v in lines[0].split(":")[1].split()]])
    for ln in lines[1:]:
        spec, want = ln.split(":", 1)[1].split("->")
        kv = dict(item.split("=") for item in spec.split())
        M, K = int(kv["M"]), int(kv["K"])
        bias = np.array([float(v) for v in kv["bias"].split(",")], dtype=np.float32)
        allowed, _ = O.select_groups(sv, 2, M)
        keys = np.where(allowed, O.selection_keys(sv, bias), np.float32(-np.inf))
        idx, _ = O.select_topk(keys.astype(np.float32), K)
        assert idx[0].tolist() == [int(v) for v in want.split(",")], ln


@pytest.mark.parametrize("E,G,M,K", [(8, 4, 2, 3), (12, 3, 2, 4), (16, 8, 3, 5), (8, 2, 1, 4)])
def test_group_limited_routing_brute_force(E, G, M, K):
    """The kept groups are the M-subset with the largest total group score
    (scores distinct), and the chosen experts are the K-subset of the kept
    experts with the largest total key."""
    rng = np.random.default_rng(E * 100 + G * 10 + M)
    gs = E // G
    for _ in range(30):
        s = rng.random((1, E))
        bias = (rng.random(E) * 0.2 - 0.1).astype(np.float32)
        allowed, _ = O.select_groups(s, G, M)
        gscore = s.astype(np.float32).astype(np.float64).reshape(G, gs).sum(axis=1)
        best = max(itertools.combinations(range(G), M), key=lambda c: sum(gscore[list(c)]))
        want_allowed = np.zeros(E, bool)
        for g in best:
            want_allowed[g * gs:(g + 1) * gs] = True
        assert np.array_equal(allowed[0], want_allowed)
        keys = O.selection_keys(s, bias)[0].astype(np.float64)
        cand = np.nonzero(want_allowed)[0]
        bestk = max(itertools.combinations(cand, K), key=lambda c: sum(keys[list(c)]))
        idx, _, _, _ = _route_with_scores(s, bias, K, G, M)
        assert sorted(idx[0].tolist()) == sorted(int(e) for e in bestk)


def _route_with_scores(s, bias, K, G, M):
    allowed, gm = O.select_groups(s, G, M)
    keys = np.where(allowed, O.selection_keys(s, bias), np.float32(-np.inf)).astype(np.float32)
    idx, margin = O.select_topk(keys, K)
    return idx, O.gate_values(s, idx, 1), np.minimum(margin, gm), s


def test_group_limit_with_all_groups_is_plain_topk():
    cfg = small_cases()["small_bf16"]
    inp = make_inputs(cfg, "cpu")
    a = O.route(inp["x"], inp["centroids"], inp["bias"], cfg.K)
    b = O.route(inp["x"], inp["centroids"], inp["bias"], cfg.K, n_groups=4, topk_groups=4)
    c = O.route(inp["x"], inp["centroids"], inp["bias"], cfg.K, n_groups=1, topk_groups=1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[0], c[0])
    assert np.array_equal(a[1], b[1])


def test_group_limit_keeps_experts_in_m_groups():
    cfg = small_cases()["small_bf16"]
    inp = make_inputs(cfg, "cpu")
    idx, gates, _, _ = O.route(inp["x"], inp["centroids"], inp["bias"], cfg.K, n_groups=8,
                               topk_groups=2)
    gs = cfg.E // 8
    for row in idx:
        assert len(set((row // gs).tolist())) <= 2
    np.testing.assert_allclose(gates.sum(axis=1), 1.0, atol=1e-12)


# ---------------------------------------------------------------- RMSNorm in front of the layer

def test_golden_rmsnorm():
    kv = dict(_read("rmsnorm_hand.txt"))
    for c in ("a", "b"):
        x = np.array([_rows(kv[c + "_x"])[0]])
        w = np.array(_rows(kv[c + "_w"])[0])
        xn, inv = O.rmsnorm(x, w, _num(kv[c + "_eps"]))
        np.testing.assert_allclose(inv, [_num(kv[c + "_inv_rms"])], rtol=1e-15, atol=0)
        np.testing.assert_allclose(xn[0], _rows(kv[c + "_xn"])[0], rtol=1e-15, atol=0)


def test_golden_prenorm_router_logits():
    """Router logits behind the RMSNorm: the weighted centroids w * e_i held in
    bf16 (one rounding, nearest even), times inv_rms (V3 walk-through, section
    4.1 with eq. (15)); the unrounded weighted centroids would miss both."""
    kv = dict(_read("rmsnorm_router_hand.txt"))
    x = np.array([_rows(kv["x"])[0]])
    w = np.array(_rows(kv["w"])[0])
    C = np.array(_rows(kv["centroids"]))
    L, inv = O.prenorm_logits(x, w, C, _num(kv["eps"]), "bf16")
    np.testing.assert_allclose(inv, [_num(kv["inv_rms"])], rtol=1e-15, atol=0)
    np.testing.assert_allclose(L[0], _rows(kv["logits"])[0], rtol=1e-14, atol=0)
    exact = inv[:, None] * (x @ (w[None, :] * C).T)
    assert np.all(np.abs(exact[0] - L[0]) > 1e-3)


def test_prenorm_logits_equal_logits_of_normalised_tokens():
    """(x * inv_rms * w) . e_i = inv_rms * (x . (w * e_i)): with weights that are
    powers of two the weighted centroids are exact in bf16 and the two forms
    agree to rounding; with w = 1 they are inv_rms * (x . e_i)."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((20, 64))
    C = O.round_bf16(rng.standard_normal((12, 64)) * 0.1)
    w = 2.0 ** rng.integers(-3, 3, 64)
    L, inv = O.prenorm_logits(x, w, C, 1e-6, "bf16")
    xn, inv2 = O.rmsnorm(x, w, 1e-6)
    np.testing.assert_allclose(inv, inv2, rtol=1e-15)
    np.testing.assert_allclose(L, O.affinity_logits(xn, C), rtol=1e-12, atol=1e-14)
    L1, inv1 = O.prenorm_logits(x, np.ones(64), C, 1e-6, "bf16")
    np.testing.assert_allclose(L1, inv1[:, None] * (x @ C.T), rtol=1e-13, atol=1e-15)
    # f32 weight type: the weighted centroids rounded to float32 instead
    Lf, _ = O.prenorm_logits(x, w * 1.1, C, 1e-6, "f32")
    ewf = (1.1 * w[None, :] * C).astype(np.float32).astype(np.float64)
    np.testing.assert_allclose(Lf, inv[:, None] * (x @ ewf.T), rtol=1e-12, atol=1e-14)


def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(5)
    d = 96
    w = rng.uniform(0.5, 1.5, d)
    # constant row c: inv_rms = 1 / sqrt(c^2 + eps), xn = c * w * inv_rms
    for cval, eps in ((0.5, 1e-6), (-3.0, 1e-6), (1e-3, 1e-6), (2.0, 0.0)):
        xn, inv = O.rmsnorm(np.full((1, d), cval), w, eps)
        np.testing.assert_allclose(inv[0], 1.0 / math.sqrt(cval * cval + eps), rtol=1e-14)
        np.testing.assert_allclose(xn[0], cval * w / math.sqrt(cval * cval + eps), rtol=1e-14)
    # eps = 0: invariant under positive scaling of the row, sign flips with the row
    x = rng.standard_normal((4, d))
    xn0, _ = O.rmsnorm(x, w, 0.0)
    for a in (1e-3, 0.25, 7.0):
        np.testing.assert_allclose(O.rmsnorm(a * x, w, 0.0)[0], xn0, rtol=1e-13, atol=0)
    np.testing.assert_allclose(O.rmsnorm(-x, w, 0.0)[0], -xn0, rtol=0, atol=0)
    # the normalised row (before w) has mean square ms / (ms + eps)
    eps = 0.05
    xn, inv = O.rmsnorm(x, w, eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean((xn / w) ** 2, axis=1), ms / (ms + eps), rtol=1e-13)


def test_round_bf16_ties_and_library():
    # spacing of bfloat16 near 1 is 2^-7: halfway cases go to the even neighbour
    v = np.array([1.0, 1 + 2.0**-8, 1 + 3 * 2.0**-8, -(1 + 3 * 2.0**-8), 1 + 2.0**-8 + 2.0**-20,
                  0.75 + 2.0**-10])
    want = np.array([1.0, 1.0, 1 + 2.0**-6, -(1 + 2.0**-6), 1 + 2.0**-7, 0.75])
    np.testing.assert_array_equal(O.round_bf16(v), want)
    # float32-representable values: one rounding, equal to torch's conversion
    r = np.random.default_rng(6).standard_normal(200000).astype(np.float32)
    t = torch.from_numpy(r).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(r.astype(np.float64)), t)


def test_prenorm_layer_is_layer_of_normalised_tokens():
    """h = x + MoE(RMSNorm(x)).  With w = 1, eps = 0 and rows of +-4 entries,
    RMSNorm(x) = x / 4 exactly, so the pre-normed layer must equal the plain
    layer on x / 4 for the routing and the MoE term, while the residual adds
    x itself (not x / 4)."""
    cfg = small_cases()["tiny"]
    inp = make_inputs(cfg)
    rng = np.random.default_rng(7)
    sgn = rng.choice([-4.0, 4.0], size=tuple(inp["x"].shape))
    x = torch.from_numpy(sgn).to(inp["x"].dtype)
    plain = dict(inp, x=x / 4)
    normed = dict(inp, x=x)
    ones = np.ones(cfg.d)
    r0 = O.moe_layer(plain, cfg.K, cfg.normalize, cfg.score_func, add_residual=1)
    r1 = O.moe_layer(normed, cfg.K, cfg.normalize, cfg.score_func, add_residual=1,
                     norm_w=ones, norm_eps=0.0, act="f32")
    np.testing.assert_array_equal(r1["idx"], r0["idx"])
    np.testing.assert_array_equal(r1["gates"], r0["gates"])
    np.testing.assert_array_equal(r1["delta"], r0["delta"])
    np.testing.assert_array_equal(r1["out"], r1["delta"] + sgn)
    # a non-trivial weight changes the routed input: the MoE term must move
    r2 = O.moe_layer(normed, cfg.K, cfg.normalize, cfg.score_func, add_residual=1,
                     norm_w=np.linspace(0.5, 1.5, cfg.d), norm_eps=0.0, act="f32")
    assert not np.allclose(r2["delta"], r0["delta"])
