"""Shared helpers of the GPU parity tests: run the CUDA path step by step
through the C ABI and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from moe_inputs import make_inputs

# Tolerances.  bf16: the stated bar for layer outputs (relative Frobenius 1e-2,
# max-abs 3e-2).  fp32: fp32 accumulation over at most a few thousand terms,
# relative error ~1e-6; 1e-4 leaves margin.  Gates: fp32 scores, 1e-5 abs.
TOL = {"bf16": (1e-2, 3e-2), "f32": (1e-4, 1e-4)}
GATE_ATOL = 1e-5
MARGIN_EXCLUDE = 1e-5


def gpu_inputs(cfg, seed=None):
    """Inputs on the GPU plus CPU views for the oracle (small configs are drawn
    on the CPU and copied, large ones drawn on the GPU)."""
    big = cfg.T * cfg.d > 4_000_000 or cfg.E * cfg.I * cfg.d > 50_000_000
    if big:
        g = make_inputs(cfg, "cuda", seed)
        return g, g
    c = make_inputs(cfg, "cpu", seed)
    g = {k: v.cuda() for k, v in c.items()}
    return g, c


def valid_topk_choice(chosen, keys, K, gscore=None, topk_groups=0, tol=MARGIN_EXCLUDE):
    """True when `chosen` (the K expert ids a kernel picked for one token) is a
    top-K of the oracle's fp32 keys [E] that rounding could have produced:
    K distinct ids, and no unchosen key above the smallest chosen key by more
    than tol.  With node-limited routing (gscore [G] = the oracle's group
    scores, topk_groups = M) the kept groups are unknown, so every M-subset G*
    of the groups that is itself a valid top-M within tol (min over G* >= max
    outside - tol) is tried: the choice is valid if for one such G* every
    chosen expert lies in G* and is a top-K within tol of G*'s experts."""
    chosen = np.asarray(chosen, dtype=np.int64)
    E = keys.shape[0]
    if len(set(chosen.tolist())) != K or chosen.min() < 0 or chosen.max() >= E:
        return False
    keys = np.asarray(keys, dtype=np.float64)

    def topk_ok(allowed):
        if not allowed[chosen].all():
            return False
        rest = allowed.copy()
        rest[chosen] = False
        return (not rest.any()) or keys[chosen].min() >= keys[rest].max() - tol

    if gscore is None:
        return topk_ok(np.ones(E, dtype=bool))
    G = gscore.shape[0]
    gs = E // G
    order = np.sort(gscore)[::-1]
    thr = order[topk_groups - 1]
    cand = [g for g in range(G) if gscore[g] >= thr - tol]
    assert len(cand) <= topk_groups + 6, "too many groups within tol to enumerate"
    import itertools
    for sub in itertools.combinations(cand, topk_groups):
        inside = np.zeros(G, dtype=bool)
        inside[list(sub)] = True
        if (~inside).any() and gscore[inside].min() < gscore[~inside].max() - tol:
            continue
        if topk_ok(np.repeat(inside, gs)):
            return True
    return False


def check_near_ties(cfg, idx_g, margin, scores, bias, gates_g=None, tol=MARGIN_EXCLUDE):
    """Tokens whose K-th vs (K+1)-th key margin (or group margin) in the oracle
    is below tol are excluded from the bit-exact comparison; each of them must
    still carry a valid choice (valid_topk_choice on the oracle's fp32 keys
    and, with node-limited routing, its group scores), and, when gates_g is
    given, the gates of eq. (13)/(14) for that choice within GATE_ATOL.
    Returns (keep, n_excluded): keep marks the tokens compared bit-exactly."""
    from oracle import moe_oracle as O
    keep = np.asarray(margin) >= tol
    excl = np.nonzero(~keep)[0]
    if excl.size:
        s = np.asarray(scores)[excl]
        if gates_g is not None:
            want = O.gate_values(s, np.asarray(idx_g)[excl], cfg.normalize)
            np.testing.assert_allclose(np.asarray(gates_g)[excl], want, rtol=0, atol=GATE_ATOL)
        keys = O.selection_keys(s, bias).astype(np.float64)
        gsc = None
        if cfg.n_groups:
            gs = cfg.E // cfg.n_groups
            gsc = s.astype(np.float32).astype(np.float64).reshape(len(excl), cfg.n_groups,
                                                                  gs).sum(axis=2)
        for j, t in enumerate(excl):
            assert valid_topk_choice(idx_g[t], keys[j], cfg.K,
                                     None if gsc is None else gsc[j], cfg.topk_groups, tol), \
                f"token {t}: chosen {sorted(idx_g[t].tolist())} is not a top-{cfg.K} " \
                f"within {tol} of the oracle's keys"
    return keep, int(excl.size)


def with_gpu_choice(ref, idx_g, keep, rerun):
    """The oracle result `ref` (a moe_layer dict over some tokens) with the
    rows of the excluded tokens (~keep, already validated by check_near_ties)
    recomputed by the oracle on the kernel's own choice of experts:
    rerun(rows, idx) must return moe_layer(..., tokens=<those rows' token
    ids>, idx=idx).  Every token is then comparable."""
    rows = np.nonzero(~np.asarray(keep))[0]
    if rows.size == 0:
        return ref
    sub = rerun(rows, np.asarray(idx_g)[rows])
    out = dict(ref)
    for k in ("out", "delta", "idx", "gates"):
        out[k] = np.array(ref[k], copy=True)
        out[k][rows] = sub[k]
    return out


def idx_with_counts(counts, K, seed=0):
    """A routing [T, K] (T = sum(counts) / K) in which expert e is chosen by
    exactly counts[e] tokens, each token's K experts distinct (every count
    must stay below T), tokens in a seeded random order."""
    counts = np.asarray(counts)
    T = int(counts.sum()) // K
    assert T * K == counts.sum() and counts.max() < T
    ids = np.repeat(np.arange(len(counts)), counts)
    idx = ids.reshape(K, T).T          # expert ids T apart: distinct per token
    assert all(len(set(r)) == K for r in idx.tolist())
    rng = np.random.default_rng(seed)
    return np.ascontiguousarray(idx[rng.permutation(T)]).astype(np.int32)


def rel_frob(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_close(got, want, dtype, what=""):
    rf, ma = TOL[dtype]
    r = rel_frob(got, want)
    m = float(np.max(np.abs(np.asarray(got, np.float64) - want))) if np.size(want) else 0.0
    assert r <= rf, f"{what}: relative Frobenius {r:.3e} > {rf}"
    assert m <= ma, f"{what}: max-abs {m:.3e} > {ma}"
    return r, m


class GpuRun:
    """Buffers and step-by-step calls of the CUDA path for one config."""

    def __init__(self, m, cfg, inp_gpu, add_residual=None):
        self.m = m
        self.lc = cfg
        self.cfg = m.cfg_from_layer(cfg)
        if add_residual is not None:
            self.cfg.add_residual = add_residual
        self.inp = inp_gpu
        T, K, E, S, d, I = cfg.T, cfg.K, cfg.E, cfg.S, cfg.d, cfg.I
        dev = "cuda"
        adt = inp_gpu["x"].dtype
        self.idx = torch.full((T, K), -1, dtype=torch.int32, device=dev)
        self.gates = torch.full((T, K), float("nan"), dtype=torch.float32, device=dev)
        self.counts = torch.full((E,), -1, dtype=torch.int32, device=dev)
        self.offsets = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
        self.xp = torch.zeros((T * K, d), dtype=adt, device=dev)
        self.perm = torch.full((T * K,), -1, dtype=torch.int32, device=dev)
        self.pos = torch.full((T, K), -1, dtype=torch.int32, device=dev)
        R = T * K + S * T
        self.act = torch.zeros((R, I), dtype=adt, device=dev)
        self.y = torch.zeros((R, d), dtype=adt, device=dev)
        self.out = torch.zeros((T, d), dtype=adt, device=dev)
        self.ws = {w: m.alloc_workspace(self.cfg, w) for w in
                   (m.MOE_WS_ROUTE, m.MOE_WS_DISPATCH, m.MOE_WS_EXPERTS, m.MOE_WS_FORWARD)}

    def route(self):
        g = self.inp
        self.m.route(self.cfg, g["x"], g["centroids"], g["bias"], self.idx, self.gates,
                     self.ws[self.m.MOE_WS_ROUTE])

    def dispatch(self, idx=None):
        self.m.dispatch(self.cfg, self.inp["x"], self.idx if idx is None else idx, self.counts,
                        self.offsets, self.xp, self.perm, self.pos,
                        self.ws[self.m.MOE_WS_DISPATCH])

    def experts(self):
        g = self.inp
        self.m.experts(self.cfg, self.xp, g["x"], self.offsets, g["w13"], g["w2"],
                       g["ws13"] if self.lc.S else None, g["ws2"] if self.lc.S else None,
                       self.act, self.y, self.ws[self.m.MOE_WS_EXPERTS])

    def combine(self, gates=None, pos=None):
        self.m.combine(self.cfg, self.y, self.gates if gates is None else gates,
                       self.pos if pos is None else pos, self.inp["x"], self.out)

    def forward(self):
        g = self.inp
        self.m.forward(self.cfg, g["x"], g["centroids"], g["bias"], g["w13"], g["w2"],
                       g["ws13"] if self.lc.S else None, g["ws2"] if self.lc.S else None,
                       self.idx, self.gates, self.counts, self.out,
                       self.ws[self.m.MOE_WS_FORWARD])

    def status(self):
        return self.m.get_status()


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()
