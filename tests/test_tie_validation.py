"""CPU checks of the near-tie rule the GPU parity tests apply: a token whose
K-th vs (K+1)-th key margin is below 1e-5 is not compared bit-exactly, but its
choice must be a top-K of the oracle's fp32 keys within 1e-5 (and, with
node-limited routing, inside a valid set of kept groups).  Wrong choices are
planted here, on the CPU, and must be rejected."""
import numpy as np
import pytest

from moe_inputs import small_cases, make_inputs
from oracle import moe_oracle as O
from tests._util import check_near_ties, valid_topk_choice, with_gpu_choice

TOL = 1e-5


def test_exact_tie_accepts_either_expert():
    keys = np.array([0.9, 0.5, 0.5, 0.1])
    assert valid_topk_choice([0, 1], keys, 2)
    assert valid_topk_choice([0, 2], keys, 2)
    assert valid_topk_choice([2, 0], keys, 2)          # listing order is free
    assert not valid_topk_choice([1, 2], keys, 2)      # the clear winner is missing
    assert not valid_topk_choice([0, 3], keys, 2)


def test_tolerance_edge():
    base = 0.5
    keys = np.array([0.9, base, base - 5e-6, base - 2e-5])
    assert valid_topk_choice([0, 2], keys, 2, tol=TOL)        # 5e-6 below: within
    assert not valid_topk_choice([0, 3], keys, 2, tol=TOL)    # 2e-5 below: not


def test_malformed_choices_rejected():
    keys = np.array([0.9, 0.5, 0.5, 0.1])
    assert not valid_topk_choice([0, 0], keys, 2)      # repeated expert
    assert not valid_topk_choice([0, 4], keys, 2)      # out of range
    assert not valid_topk_choice([0, -1], keys, 2)
    assert not valid_topk_choice([0], keys, 2)         # too few


def test_k_equals_e_takes_all():
    keys = np.array([0.3, 0.2, 0.1])
    assert valid_topk_choice([2, 0, 1], keys, 3)


def test_grouped_choice_follows_kept_groups():
    # 4 groups of 2 experts, keep 2 groups; group scores 1.0, 0.8, 0.8 (tie), 0.1
    gscore = np.array([1.0, 0.8, 0.8, 0.1])
    keys = np.array([0.6, 0.4, 0.5, 0.3, 0.45, 0.35, 0.9, 0.05])
    # kept {0, 1}: top-2 of experts 0..3 -> {0, 2}; kept {0, 2}: experts 0,1,4,5 -> {0, 4}
    assert valid_topk_choice([0, 2], keys, 2, gscore, 2)
    assert valid_topk_choice([0, 4], keys, 2, gscore, 2)
    # expert 6 has the largest key but its group (score 0.1) is never kept
    assert not valid_topk_choice([0, 6], keys, 2, gscore, 2)
    # {0, 1}: expert 1 loses to expert 2 inside kept {0, 1} and to 4 in {0, 2}
    assert not valid_topk_choice([0, 1], keys, 2, gscore, 2)
    # with a clear group order (no tie) only the first two groups may serve
    gclear = np.array([1.0, 0.8, 0.7, 0.1])
    assert valid_topk_choice([0, 2], keys, 2, gclear, 2)
    assert not valid_topk_choice([0, 4], keys, 2, gclear, 2)


def test_check_near_ties_rejects_a_planted_wrong_choice():
    """Oracle routing of a small layer, with near-tie tokens forced by equal
    centroids; a "kernel" result that picks a clearly losing expert for an
    excluded token fails, the oracle's own choice and the tied alternative pass."""
    cfg = small_cases()["small_bf16"].with_(name="ties", T=32, E=8, K=2, bias_range=0.0)
    c = make_inputs(cfg, "cpu")
    cent = c["centroids"].clone()
    cent[3] = cent[5]                                   # experts 3 and 5 always tie
    c["centroids"] = cent
    idx_o, gates_o, margin, s = O.route(c["x"], cent, c["bias"], cfg.K)
    tied = np.nonzero(margin < TOL)[0]
    assert tied.size > 0
    keep, n = check_near_ties(cfg, idx_o, margin, s, c["bias"], gates_o)
    assert n == tied.size and not keep[tied].any()
    # swap 3 <-> 5 on tied tokens that chose one of them as the K-th: still valid
    alt = idx_o.copy()
    for t in tied:
        for k in range(cfg.K):
            if alt[t, k] in (3, 5):
                alt[t, k] = 8 - alt[t, k]
    check_near_ties(cfg, alt, margin, s, c["bias"], O.gate_values(s, alt, cfg.normalize))
    # a clearly worse expert on one tied token: rejected
    bad = idx_o.copy()
    t = tied[0]
    keys = O.selection_keys(s[t:t + 1], c["bias"])[0]
    worst = int(np.argmin(keys))
    bad[t, 0] = worst if worst not in bad[t] else bad[t, 0]
    with pytest.raises(AssertionError):
        check_near_ties(cfg, bad, margin, s, c["bias"])
    # right experts, wrong gates: rejected
    with pytest.raises(AssertionError):
        check_near_ties(cfg, idx_o, margin, s, c["bias"], gates_o[:, ::-1].copy())


def test_with_gpu_choice_recomputes_only_excluded_rows():
    cfg = small_cases()["small_bf16"].with_(name="ties2", T=16, E=8, K=2, bias_range=0.0)
    c = make_inputs(cfg, "cpu")

    def layer(**kw):
        return O.moe_layer(c, cfg.K, cfg.normalize, cfg.score_func, add_residual=0, **kw)

    ref = layer()
    keep = np.ones(cfg.T, dtype=bool)
    keep[[3, 7]] = False
    other = ref["idx"].copy()
    other[3] = other[3][::-1]                          # same set, other order
    other[7, 1] = [e for e in range(cfg.E) if e not in other[7]][0]
    got = with_gpu_choice(ref, other, keep, lambda rows, ix: layer(tokens=rows, idx=ix))
    np.testing.assert_array_equal(got["delta"][keep], ref["delta"][keep])
    np.testing.assert_allclose(got["delta"][3], ref["delta"][3], rtol=1e-12, atol=1e-15)
    want7 = layer(tokens=[7], idx=other[7:8])["delta"][0]
    np.testing.assert_allclose(got["delta"][7], want7, rtol=1e-12, atol=1e-15)
    assert not np.allclose(got["delta"][7], ref["delta"][7])
