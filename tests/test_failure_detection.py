"""Failure detection on the device without a fault: a bounded barrier wait
(the one every GEMM role uses) that runs out sets the device error word, the
host reads MOE_ERR_DEVICE_TIMEOUT once, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

from moe_inputs import small_cases
from oracle import moe_oracle as O
from tests._util import gpu_inputs, assert_close, to_np, check_near_ties, with_gpu_choice

pytestmark = pytest.mark.gpu

m = pytest.importorskip("mixture_experts_layer_88_b300")

MOE_ERR_DEVICE_TIMEOUT = 5


def test_bounded_wait_runs_out_and_context_stays_usable():
    assert m.get_status() == 0
    t0 = time.perf_counter()
    m.selftest_wait_timeout(20_000_000)                # 20 ms
    st = m.get_status()                                 # synchronises the stream
    dt = time.perf_counter() - t0
    assert st == MOE_ERR_DEVICE_TIMEOUT
    assert 0.015 < dt < 2.0, f"the wait gave up after {dt:.3f} s"
    assert m.get_status() == 0                          # read once, then cleared
    # the same context still runs the layer correctly
    cfg = small_cases()["small_bf16"]
    g, c = gpu_inputs(cfg)
    mc = m.cfg_from_layer(cfg)
    mc.add_residual = 0
    layer = m.MoeLayer(mc, g, device="cuda")
    out = layer.forward(g["x"])
    assert m.get_status() == 0
    ref = O.moe_layer(c, cfg.K, cfg.normalize, cfg.score_func, add_residual=0)
    idx_g = layer.idx.cpu().numpy()
    keep, _ = check_near_ties(cfg, idx_g, ref["margin"], ref["scores"], c["bias"],
                              layer.gates.cpu().numpy())
    np.testing.assert_array_equal(np.sort(idx_g, 1)[keep], np.sort(ref["idx"], 1)[keep])
    ref = with_gpu_choice(ref, idx_g, keep, lambda rows, ix: O.moe_layer(
        c, cfg.K, cfg.normalize, cfg.score_func, add_residual=0, tokens=rows, idx=ix))
    assert_close(to_np(out), ref["delta"], "bf16", "layer after a timeout")
