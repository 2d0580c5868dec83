"""CPU oracle for the DeepSeekMoE layer forward, load count, bias update and
the training backward.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module.  The CUDA library never calls it and shares no code with it; the two
meet only in the seeded inputs of ``moe_inputs``.

Plain, slow and written to be checked by eye against the pages:
everything is float64 numpy, one step per equation, no blocking or fusion.
Library primitives used as steps: matrix product (``@``), ``np.exp``,
``np.lexsort``, ``np.bincount``, ``np.cumsum``, ``np.frexp``, ``np.round``.

Sources (DeepSeekMoE pages):
- "DeepSeekMoE架构解析" (V3 walk-through), section 2.1, eqs. (13)-(15): Sigmoid
  affinity, hard top-K_r, renormalisation over the chosen experts;
  section 2.2, eq. (16): the balancing bias enters the top-K decision only;
  section 2.2, update rule: overloaded experts b_i -= gamma, underloaded
  b_i += gamma, gamma = 0.001; section 3.1: output = u_t + shared + routed.
- course chapter "MoE" (blog.zero43.top), section 4: the 2024 DeepSeekMoE
  gates are not renormalised (their sum is generally below 1); section 5: the
  bias is updated after every batch and takes effect for the next one;
  section 6: no token is dropped.

Readings where the pages are silent:
- The top-K decision is taken on float32 keys fp32(fp32(s_i) + b_i): the pages
  fix no precision, so the decision uses the CUDA kernel's.  Equal keys go to
  the lower expert index; chosen experts are listed by descending key.
- Expert FFN is SwiGLU without linear biases: W2 (SiLU(Wg u) * (Wu u)).
- Shared experts enter the sum with weight 1, the residual u_t is optional.
- "Overloaded" means count_i * E > T * K (exactly above the mean load); equal
  to the mean leaves b_i unchanged.  The update is float32 arithmetic.
- Softmax mode (2024 layer) normalises over all E experts before selection.
- Node-limited routing ranks groups by the sum of the unbiased scores s of
  all their experts (the page's "affinity scores"); the bias then acts only
  inside the kept groups.
- If the chosen scores sum to 0 the renormalised gates are 0.
- The RMSNorm in front of the layer (V3 walk-through, section 4.1, eps 1e-6) is
  the standard one with a per-channel weight, x * w / sqrt(mean(x^2) + eps);
  the residual adds the un-normalised x.  The experts read the normalised
  tokens held in the activation type (rounded once, like every stored
  activation).  The router reads no stored normalised token: its logit is
  (x * inv_rms * w) . e_i = inv_rms * (x . (w * e_i)), with the weighted
  centroid w * e_i held in the weight type (rounded once, like every stored
  weight) and inv_rms = 1 / sqrt(mean(x^2) + eps) applied to the logit.
- Backward pass (no page writes it out; V3 walk-through, section 2.2, says the
  bias only steers the selection): the gradients of a scalar loss whose
  gradient with respect to the layer output is dout, by the chain rule through
  the forward above.  The chosen experts (top-K, groups) are constants of the
  backward, the bias gets no gradient, and the gradient reaches the centroids
  and the tokens through the gates only (renormalisation, then Sigmoid or
  Softmax).  Pinned by central finite differences of ``moe_layer``.
"""
from __future__ import annotations

import numpy as np

SIGMOID = 0
SOFTMAX = 1


def _f64(a) -> np.ndarray:
    """Exact upcast of a numpy array or a torch tensor (any device/dtype) to fp64."""
    if hasattr(a, "detach"):
        import torch
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch
        return a.detach().to("cpu", torch.float32).numpy()
    return np.asarray(a, dtype=np.float32)


# ----------------------------------------------------------------------------
# RMSNorm in front of the layer (V3 walk-through, section 4.1: an RMSNorm before
# and after the MoE layer, eps = 1e-6)
# ----------------------------------------------------------------------------

def rmsnorm(x, w, eps: float = 1e-6):
    """Root-mean-square normalisation of each token row, then the per-channel
    weight: inv_rms_t = 1 / sqrt(mean_j x_tj^2 + eps), xn_tj = x_tj * inv_rms_t
    * w_j.  x [T, d], w [d] -> (xn [T, d] fp64, inv_rms [T] fp64)."""
    xv = _f64(x)
    inv_rms = 1.0 / np.sqrt(np.mean(xv * xv, axis=1) + eps)
    return xv * inv_rms[:, None] * _f64(w)[None, :], inv_rms


def prenorm_logits(x, w, centroids, eps: float = 1e-6, wgt: str = "bf16"):
    """Router logits of the layer behind its RMSNorm (see header): the RMSNorm
    weight scales the centroids, w * e_i held in the weight type ``wgt``
    (rounded once), and 1/rms scales the logit:
      L[t, i] = inv_rms_t * sum_j x_tj (w_j e_ij).
    Returns (L [T, E] fp64, inv_rms [T] fp64)."""
    xv = _f64(x)
    inv_rms = 1.0 / np.sqrt(np.mean(xv * xv, axis=1) + eps)
    ew = round_act(_f64(w)[None, :] * _f64(centroids), wgt)
    return inv_rms[:, None] * (xv @ ew.T), inv_rms


def round_bf16(v) -> np.ndarray:
    """Round to the nearest bfloat16 value (8 significant bits), ties to even,
    from the exact fp64 value (one rounding).  Normal-range values only."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                     # v = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def round_act(v, act: str) -> np.ndarray:
    """Rounding of a stored activation: 'bf16' or 'f32'."""
    if act == "bf16":
        return round_bf16(v)
    return np.asarray(v, dtype=np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Router: eqs. (15), (16), (14), (13)
# ----------------------------------------------------------------------------

def affinity_logits(u, centroids) -> np.ndarray:
    """u_t^T e_i for every token t and expert i (inner product of eq. 15).
    u [T, d], centroids [E, d] -> [T, E] fp64."""
    return _f64(u) @ _f64(centroids).T


def expert_scores(logits: np.ndarray, score_func: int = SIGMOID) -> np.ndarray:
    """s_{i,t}.  SIGMOID: eq. (15), applied to each expert on its own.
    SOFTMAX: the 2024 gating, normalised over all E experts."""
    if score_func == SIGMOID:
        return 1.0 / (1.0 + np.exp(-logits))
    if score_func == SOFTMAX:
        z = logits - logits.max(axis=1, keepdims=True)
        ez = np.exp(z)
        return ez / ez.sum(axis=1, keepdims=True)
    raise ValueError("score_func")


def selection_keys(s: np.ndarray, bias) -> np.ndarray:
    """Biased keys s_{i,t} + b_i of eq. (16), formed in float32 (see header)."""
    return (s.astype(np.float32) + _f32(bias)[None, :]).astype(np.float32)


def select_topk(keys: np.ndarray, K: int):
    """Top-K_r of eq. (14)/(16): the K largest keys per token, by descending key,
    equal keys to the lower expert index.  Returns idx [T, K] int32 and the
    margin key_(K) - key_(K+1) per token (inf when K == E)."""
    T, E = keys.shape
    idx = np.empty((T, K), dtype=np.int32)
    margin = np.full(T, np.inf)
    experts = np.arange(E)
    for t in range(T):
        # lexsort sorts by the last key first: descending key, then ascending index
        order = np.lexsort((experts, -keys[t].astype(np.float64)))
        idx[t] = order[:K]
        if K < E:
            margin[t] = float(keys[t, order[K - 1]]) - float(keys[t, order[K]])
    return idx, margin


def select_groups(s: np.ndarray, n_groups: int, topk_groups: int):
    """Node-limited routing (V3 walk-through, section 2.3): the experts are split
    into n_groups equal groups of consecutive indices (one group per node); a
    group's score is the sum of the affinity scores s of all its experts; the
    topk_groups best groups are kept (equal scores to the lower group index).
    Scores are summed in fp64 from the fp32-rounded s.  Returns the allowed
    mask [T, E] and the margin between the M-th and (M+1)-th group score."""
    T, E = s.shape
    gs = E // n_groups
    gscore = s.astype(np.float32).astype(np.float64).reshape(T, n_groups, gs).sum(axis=2)
    allowed = np.zeros((T, E), dtype=bool)
    margin = np.full(T, np.inf)
    groups = np.arange(n_groups)
    for t in range(T):
        order = np.lexsort((groups, -gscore[t]))
        for g in order[:topk_groups]:
            allowed[t, g * gs:(g + 1) * gs] = True
        if topk_groups < n_groups:
            margin[t] = gscore[t, order[topk_groups - 1]] - gscore[t, order[topk_groups]]
    return allowed, margin


def gate_values(s: np.ndarray, idx: np.ndarray, normalize: int) -> np.ndarray:
    """g'_{i,t} = s_{i,t} for the chosen experts (eq. 14; the bias is not used),
    then g = g' / sum_j g'_j over the chosen experts (eq. 13) when ``normalize``."""
    g = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    if normalize:
        tot = g.sum(axis=1, keepdims=True)
        g = np.where(tot > 0, g / np.where(tot > 0, tot, 1.0), 0.0)
    return g


def route(u, centroids, bias, K: int, score_func: int = SIGMOID, normalize: int = 1,
          n_groups: int = 0, topk_groups: int = 0):
    """Whole router for the given tokens: idx, gates (fp64), margins, scores.
    With n_groups > 0 the top-K runs only over the experts of the topk_groups
    best groups (select_groups); the returned margin is then the smaller of
    the group margin and the expert margin inside the kept groups."""
    return route_logits(affinity_logits(u, centroids), bias, K, score_func, normalize,
                        n_groups, topk_groups)


def route_logits(logits, bias, K: int, score_func: int = SIGMOID, normalize: int = 1,
                 n_groups: int = 0, topk_groups: int = 0):
    """route() from given affinity logits [T, E] (eqs. (15), (16), (14), (13))."""
    s = expert_scores(logits, score_func)
    keys = selection_keys(s, bias)
    gmargin = None
    if n_groups > 0:
        allowed, gmargin = select_groups(s, n_groups, topk_groups)
        keys = np.where(allowed, keys, np.float32(-np.inf)).astype(np.float32)
    idx, margin = select_topk(keys, K)
    if gmargin is not None:
        margin = np.minimum(margin, gmargin)
    return idx, gate_values(s, idx, normalize), margin, s


# ----------------------------------------------------------------------------
# Dispatch: no-drop assignment of every (token, slot) to its expert
# ----------------------------------------------------------------------------

def dispatch(idx: np.ndarray, E: int):
    """counts[i] = #(t,k) with idx[t,k] = i; offsets = exclusive prefix sum
    (length E+1); rows of expert i are its tokens in ascending token order:
    perm_tok[offsets[i] + r] = r-th such token; pos[t,k] = row of (t,k).
    Nothing is dropped: every (t,k) gets a row (course chapter, section 6)."""
    T, K = idx.shape
    counts = np.bincount(idx.reshape(-1), minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    perm_tok = np.empty(T * K, dtype=np.int64)
    pos = np.empty((T, K), dtype=np.int64)
    for t in range(T):
        for k in range(K):
            i = idx[t, k]
            pos[t, k] = fill[i]
            perm_tok[fill[i]] = t
            fill[i] += 1
    return counts, offsets, perm_tok, pos


# ----------------------------------------------------------------------------
# Experts and combine
# ----------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def dequantize_blocks(q, scale, block: int = 128) -> np.ndarray:
    """Block-wise FP8 weight of the V3 walk-through, section 4.3 (128 x 128
    blocks, one fp32 scale each): w[r, c] = q[r, c] * scale[r // 128, c // 128],
    in fp64.  ``q`` holds e4m3 values (decoded exactly by the upcast)."""
    qv = _f64(q)
    sc = _f64(scale)
    return qv * np.repeat(np.repeat(sc, block, axis=0), block, axis=1)


def _expert_weight(inp: dict, key: str, e: int, dequant_round: str = None):
    """Weight ``key`` of expert e, dequantised when the layer stores FP8 blocks;
    with ``dequant_round`` ('bf16') each dequantised weight q * scale is then
    rounded once to that type, as a layer that multiplies in it holds it."""
    w = inp[key][e]
    if key + "_scale" in inp:
        w = dequantize_blocks(w, inp[key + "_scale"][e])
        if dequant_round is not None:
            w = round_act(w, dequant_round)
    return w


def round_e4m3(v) -> np.ndarray:
    """Nearest e4m3 value, ties to even, saturating at +-448.  The format (the
    FP8 type of the V3 walk-through, section 4.3): 1 sign bit, 4 exponent
    bits with bias 7, 3 mantissa bits, largest finite value 448, no
    infinities.  A binade [2^e, 2^(e+1)) holds 8 values 2^(e-3) apart for
    e = -6 .. 8; below 2^-6 the subnormals are 2^-9 apart.  fp64 in, fp64 out
    (every e4m3 value is exact in fp64)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                       # a = m 2^ex, 0.5 <= m < 1
    e = np.clip(ex - 1, -6, 8)                # binade of a (subnormals share e = -6)
    step = np.ldexp(1.0, e - 3)
    q = np.round(a / step) * step             # np.round: halves go to the even step
    q = np.minimum(q, 448.0)
    return np.copysign(q, v)


def quantize_tiles_e4m3(v, tile: int = 128) -> np.ndarray:
    """Online FP8 quantisation of activations (V3 walk-through, section 4.3):
    every 1 x 128 tile along the last axis gets the fp32 scale
    s = max|v| / 448 and its values the e4m3 codes q = e4m3(v * (448 / max|v|)),
    so the tile's largest value lands on 448.  The page fixes no precision for
    forming the code; it is taken in float32 (max|v|, 448 / max|v| and the
    product each rounded once), as the CUDA kernels form it.  Returns q * s in
    fp64 (an all-zero tile stays zero)."""
    v32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    n, m = v32.shape
    t = v32.reshape(n, m // tile, tile)
    amax = np.abs(t).max(axis=2, keepdims=True)
    safe = np.where(amax > 0, amax, np.float32(1))
    inv = np.where(amax > 0, np.float32(448) / safe, np.float32(0)).astype(np.float32)
    q = round_e4m3((t * inv).astype(np.float32))
    scale = (amax / np.float32(448)).astype(np.float32)
    return (q * scale.astype(np.float64)).reshape(n, m)


def swiglu_ffn(u: np.ndarray, w13, w2, stored: str = None) -> np.ndarray:
    """One expert: W2 (SiLU(Wg u) * (Wu u)); w13 [2I, d] = [Wg; Wu], w2 [d, I].
    u [n, d] fp64 -> [n, d] fp64.  With ``stored`` ('bf16' or 'f32') the
    SwiGLU output and the expert output are rounded once to that type, as a
    layer that stores them does (reading: act and y are stored in the
    activation type)."""
    w13 = _f64(w13)
    I = w13.shape[0] // 2
    h = u @ w13.T
    a = silu(h[:, :I]) * h[:, I:]
    if stored is not None:
        a = round_act(a, stored)
    y = a @ _f64(w2).T
    return y if stored is None else round_act(y, stored)


def swiglu_ffn_fp8(u: np.ndarray, w13, w2) -> np.ndarray:
    """One expert of an FP8 layer as the V3 walk-through, section 4.3, runs it:
    the expert's input rows and its SwiGLU output are quantised in 1 x 128
    tiles (``quantize_tiles_e4m3``) before the GEMM that reads them; the
    weights are the dequantised 128 x 128 blocks.  Products are summed in
    fp64: the promotion to fp32 every 128 elements changes only the rounding
    order."""
    w13 = _f64(w13)
    I = w13.shape[0] // 2
    h = quantize_tiles_e4m3(u) @ w13.T
    a = silu(h[:, :I]) * h[:, I:]
    return quantize_tiles_e4m3(a) @ _f64(w2).T


def moe_layer(inp: dict, K: int, normalize: int = 1, score_func: int = SIGMOID,
              add_residual: int = 1, tokens=None, n_groups: int = 0,
              topk_groups: int = 0, norm_w=None, norm_eps: float = 1e-6,
              act: str = "bf16", idx=None, wgt: str = None,
              act_quant: bool = False, stored_rounding: bool = False,
              dequant_round: str = None) -> dict:
    """Forward of one DeepSeekMoE layer for all tokens, or for the listed token
    ids.  out_t = [u_t] + sum_s FFN_s(u_t) + sum_k g_{t,k} FFN_{idx[t,k]}(u_t).

    ``inp`` holds x, centroids, bias, w13, w2, ws13, ws2 (see moe_inputs), and
    for FP8 layers their 128 x 128 block scales (``*_scale``); activations are
    used as stored (bf16), unquantised.  Expert weights are read one expert at
    a time, so large layers can be evaluated on a token sample.

    With ``norm_w`` the layer sits behind its RMSNorm: the experts read
    u = RMSNorm(x) held in the activation type ``act`` (rounded once), the
    router takes its logits from x by prenorm_logits (weighted centroids in
    the weight type ``wgt``), and the residual adds x itself
    (h = x + MoE(RMSNorm(x))).

    ``idx`` [n, K], when given, replaces the router's own choice for these
    tokens (another valid top-K where keys tie within rounding); the gates
    are then those of eq. (13)/(14) for that choice and the margin is NaN.

    ``act_quant`` (FP8 layers): every expert also quantises its input rows and
    its SwiGLU output to e4m3 in 1 x 128 tiles (``swiglu_ffn_fp8``), as the
    page's FP8 scheme does; without it the activations stay as stored.

    ``stored_rounding`` (bf16 and fp32 weights): every expert's SwiGLU output
    and output rows are rounded once to the activation type ``act``, and so is
    the layer output, the points where a layer that stores them in that type
    rounds (the sums stay fp64).

    ``dequant_round`` (FP8 layers): each dequantised weight is rounded once to
    that type ('bf16'), the weights a layer that dequantises to bf16 and
    multiplies on bf16 tensor cores uses.

    Returns out (fp64), delta = out - residual, idx, gates, margin, and the
    scores s [n, E] of every expert."""
    x = inp["x"]
    if tokens is not None:
        tokens = np.asarray(tokens, dtype=np.int64)
        x = x[tokens] if not hasattr(x, "detach") else x[_torch_index(tokens, x)]
    resid = _f64(x)
    if norm_w is not None:
        u = round_act(rmsnorm(resid, norm_w, norm_eps)[0], act)
        logits = prenorm_logits(resid, norm_w, inp["centroids"], norm_eps,
                                wgt if wgt is not None else act)[0]
    else:
        u = resid
        logits = affinity_logits(u, inp["centroids"])
    n = u.shape[0]
    if idx is None:
        idx, gates, margin, scores = route_logits(logits, inp["bias"], K, score_func,
                                                  normalize, n_groups, topk_groups)
    else:
        scores = expert_scores(logits, score_func)
        idx = np.asarray(idx, dtype=np.int32).reshape(n, K)
        gates = gate_values(scores, idx, normalize)
        margin = np.full(n, np.nan)
    d = u.shape[1]
    delta = np.zeros((n, d))
    S = inp["ws13"].shape[0]
    if act_quant:
        ffn = swiglu_ffn_fp8
    elif stored_rounding:
        def ffn(x_, w13_, w2_):
            return swiglu_ffn(x_, w13_, w2_, stored=act)
    else:
        ffn = swiglu_ffn
    def weight(key, e):
        return _expert_weight(inp, key, e, dequant_round)

    for s in range(S):
        delta += ffn(u, weight("ws13", s), weight("ws2", s))
    routed = np.zeros((n, K, d))
    for e in np.unique(idx):
        rows, slots = np.nonzero(idx == e)
        routed[rows, slots] = ffn(u[rows], weight("w13", int(e)), weight("w2", int(e)))
    for k in range(K):
        delta += gates[:, k:k + 1] * routed[:, k]
    out = delta + resid if add_residual else delta.copy()
    if stored_rounding:
        out = round_act(out, act)
        delta = out - resid if add_residual else out.copy()
    return {"out": out, "delta": delta, "idx": idx, "gates": gates, "margin": margin,
            "scores": scores}


def _torch_index(tokens, ref):
    import torch
    return torch.as_tensor(tokens, device=ref.device)


# ----------------------------------------------------------------------------
# Backward pass: gradients of L with dL/d(out) = dout, chosen experts fixed
# ----------------------------------------------------------------------------

def _keep(v):
    return v


def swiglu_ffn_backward(u: np.ndarray, w13, w2, dy: np.ndarray, rnd=_keep):
    """Gradients of one expert y = W2 a, a = SiLU(g) * v, [g; v] = W13 u, for
    rows u [n, d] and output gradients dy [n, d]:
      da = dy W2,  dW2 = dy^T a,
      dg = da * v * SiLU'(g) with SiLU'(g) = sig(g) (1 + g (1 - sig(g))),
      dv = da * SiLU(g),  dh = [dg, dv],  dW13 = dh^T u,  du = dh W13.
    ``rnd`` is applied where a layer that stores them rounds: h, a, da, dh
    and du (identity by default).  Returns du [n, d], dw13 [2I, d],
    dw2 [d, I], all fp64."""
    w13 = _f64(w13)
    w2 = _f64(w2)
    I = w13.shape[0] // 2
    h = rnd(u @ w13.T)
    g, v = h[:, :I], h[:, I:]
    sig = 1.0 / (1.0 + np.exp(-g))
    a = rnd(g * sig * v)
    da = rnd(dy @ w2)
    dw2 = dy.T @ a
    dg = da * v * sig * (1.0 + g * (1.0 - sig))
    dv = da * g * sig
    dh = rnd(np.concatenate([dg, dv], axis=1))
    return rnd(dh @ w13), dh.T @ u, dw2


def router_backward(u: np.ndarray, centroids, s: np.ndarray, idx: np.ndarray,
                    gates: np.ndarray, dgates: np.ndarray, normalize: int,
                    score_func: int = SIGMOID):
    """Gradients through eqs. (13)-(15) for fixed chosen experts idx.
    Renormalised gates g_k = s_k / sum_j s_j (chosen j) give
      ds_k = (dg_k - sum_j dg_j g_j) / sum_j s_j   (0 when the sum is 0),
    otherwise ds_k = dg_k; experts not chosen get ds = 0.  Then
      SIGMOID: dlogit_i = ds_i s_i (1 - s_i)
      SOFTMAX: dlogit_i = s_i (ds_i - sum_j ds_j s_j)   (all E experts)
    and logit_i = u . e_i gives du = dlogit C, dC = dlogit^T u.
    Returns du [n, d], dcentroids [E, d], dlogit [n, E]."""
    T, E = s.shape
    ix = idx.astype(np.int64)
    sc = np.take_along_axis(s, ix, axis=1)
    if normalize:
        tot = sc.sum(axis=1, keepdims=True)
        inner = (dgates * gates).sum(axis=1, keepdims=True)
        ds_c = np.where(tot > 0, (dgates - inner) / np.where(tot > 0, tot, 1.0), 0.0)
    else:
        ds_c = dgates
    ds = np.zeros((T, E))
    np.put_along_axis(ds, ix, ds_c, axis=1)
    if score_func == SIGMOID:
        dlogit = ds * s * (1.0 - s)
    elif score_func == SOFTMAX:
        dlogit = s * (ds - (ds * s).sum(axis=1, keepdims=True))
    else:
        raise ValueError("score_func")
    C = _f64(centroids)
    return dlogit @ C, dlogit.T @ u, dlogit


def moe_layer_backward(inp: dict, K: int, dout, normalize: int = 1,
                       score_func: int = SIGMOID, add_residual: int = 1,
                       n_groups: int = 0, topk_groups: int = 0, idx=None,
                       stored_rounding: bool = False) -> dict:
    """Backward of ``moe_layer`` (no RMSNorm in front) for all T tokens:
    dout [T, d] is dL/d(out).  The routed term g_k FFN_k(u) gives
      dgates[t, k] = dout_t . FFN_k(u_t),  dFFN_k = g_k dout_t,
    the shared experts get dout_t itself, the residual passes dout_t to u_t,
    and the router adds its term through the gates (router_backward).
    Returns dx [T, d], dcentroids [E, d], dw13 [E, 2I, d], dw2 [E, d, I],
    dws13 [S, 2I, d], dws2 [S, d, I], dgates [T, K], dlogit [T, E], idx,
    gates, margin; every array fp64.  Weight gradients of experts that no
    token chose are zero.  ``idx`` [T, K], when given, replaces the router's
    own choice (another valid choice where keys tie); the gates are then
    those of eq. (13)/(14) for that choice and the margin is NaN.

    ``stored_rounding``: values a bf16 training layer stores are rounded once
    to bf16 where it stores them: the training forward's h = [gate | up], act
    and y; the row gradients g * dout, da, [dgate, dup] and du; and the
    outputs dx and the weight gradients.  Sums stay fp64; dgates, dlogit and
    the centroid gradients are not rounded."""
    u = _f64(inp["x"])
    go = _f64(dout)
    rnd = round_bf16 if stored_rounding else _keep
    T, d = u.shape
    if idx is None:
        idx, gates, margin, s = route(u, inp["centroids"], inp["bias"], K, score_func,
                                      normalize, n_groups, topk_groups)
    else:
        s = expert_scores(affinity_logits(u, inp["centroids"]), score_func)
        idx = np.asarray(idx, dtype=np.int32)
        gates = gate_values(s, idx, normalize)
        margin = np.full(T, np.nan)
    w13 = inp["w13"]
    E = w13.shape[0]
    I = w13.shape[1] // 2
    S = inp["ws13"].shape[0]
    dx = go.copy() if add_residual else np.zeros((T, d))
    dw13 = np.zeros((E, 2 * I, d))
    dw2 = np.zeros((E, d, I))
    dws13 = np.zeros((S, 2 * I, d))
    dws2 = np.zeros((S, d, I))
    dgates = np.zeros((T, K))
    for sx in range(S):
        du, dw13_s, dw2_s = swiglu_ffn_backward(u, _expert_weight(inp, "ws13", sx),
                                                _expert_weight(inp, "ws2", sx), go, rnd)
        dx += du
        dws13[sx] = rnd(dw13_s)
        dws2[sx] = rnd(dw2_s)
    for e in np.unique(idx):
        rows, slots = np.nonzero(idx == e)
        ue = u[rows]
        w13e = _expert_weight(inp, "w13", int(e))
        w2e = _expert_weight(inp, "w2", int(e))
        if stored_rounding:
            # the training forward's y: from the stored h, act stored, y stored
            he = rnd(ue @ _f64(w13e).T)
            ye = rnd(rnd(silu(he[:, :I]) * he[:, I:]) @ _f64(w2e).T)
        else:
            ye = swiglu_ffn(ue, w13e, w2e)
        dgates[rows, slots] = np.sum(go[rows] * ye, axis=1)
        dye = rnd(gates[rows, slots][:, None] * go[rows])
        du, dw13_e, dw2_e = swiglu_ffn_backward(ue, w13e, w2e, dye, rnd)
        dw13[e], dw2[e] = rnd(dw13_e), rnd(dw2_e)
        np.add.at(dx, rows, du)
    du_r, dcent, dlogit = router_backward(u, inp["centroids"], s, idx, gates, dgates,
                                          normalize, score_func)
    dx = rnd(dx + du_r)
    return {"dx": dx, "dcentroids": dcent, "dw13": dw13, "dw2": dw2, "dws13": dws13,
            "dws2": dws2, "dgates": dgates, "dlogit": dlogit, "idx": idx, "gates": gates,
            "margin": margin}


# ----------------------------------------------------------------------------
# Load count and bias update (section 2.2 of the V3 walk-through)
# ----------------------------------------------------------------------------

def update_bias(counts, bias, T: int, K: int, gamma: float = 1e-3):
    """b_i -= gamma if expert i took more than the mean load T*K/E, += gamma if
    less, unchanged if equal.  Comparison in integers (count_i*E vs T*K), the
    add in float32.  Returns (new bias fp32 [E], (max/mean, min/mean))."""
    c = np.asarray(counts, dtype=np.int64)
    E = c.shape[0]
    b = _f32(bias).copy()
    g = np.float32(gamma)
    over = c * E > T * K
    under = c * E < T * K
    b[over] = (b[over] - g).astype(np.float32)
    b[under] = (b[under] + g).astype(np.float32)
    mean = T * K / E
    return b, (float(c.max()) / mean, float(c.min()) / mean)
