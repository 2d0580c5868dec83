"""moe_experts_static: the expert FFNs for callers that cannot allocate device
memory (a runtime that reserves all device memory at start-up, or a plugin
whose host owns the allocator and hands out no scratch).  It keeps its scratch
in a fixed array inside the library instead of a caller workspace.

The file is named to be collected last.  Each case calls the new entry point
twice in a row through the C ABI and checks both results against moe_experts
(the workspace entry point) within the layer-output tolerance of the suite,
and, since both run the same deterministic kernels, bit for bit.
"""
import ctypes

import pytest
import torch

from moe_inputs import small_cases
from oracle import moe_oracle as O
from tests._util import GpuRun, gpu_inputs, assert_close, to_np

pytestmark = pytest.mark.gpu

m = pytest.importorskip("mixture_experts_layer_88_b300")


def _static_call(run, act, y):
    g = run.inp
    lc = run.lc
    code = m._lib.lib().moe_experts_static(
        ctypes.byref(run.cfg), run.xp.data_ptr(), g["x"].data_ptr(), run.offsets.data_ptr(),
        g["w13"].data_ptr(), g["w2"].data_ptr(),
        g["ws13"].data_ptr() if lc.S else None, g["ws2"].data_ptr() if lc.S else None,
        act.data_ptr(), y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return code


@pytest.mark.parametrize("name", ["small_bf16", "ragged_bf16", "softmax_norenorm", "tiny"])
def test_experts_static_matches_workspace_entry_point(name):
    cfg = small_cases()[name]
    g, c = gpu_inputs(cfg)
    run = GpuRun(m, cfg, g)
    idx_o, _, _, _ = O.route(c["x"], c["centroids"], c["bias"], cfg.K, cfg.score_func,
                             cfg.normalize)
    run.dispatch(torch.as_tensor(idx_o, dtype=torch.int32, device="cuda"))
    run.experts()                                   # reference: caller workspace
    torch.cuda.synchronize()
    act_ref, y_ref = to_np(run.act), to_np(run.y)
    for call in range(2):
        act = torch.full_like(run.act, float("nan"))
        y = torch.full_like(run.y, float("nan"))
        assert _static_call(run, act, y) == 0
        torch.cuda.synchronize()
        assert m.get_status() == 0
        assert_close(to_np(act), act_ref, cfg.act, f"{name} act, call {call}")
        assert_close(to_np(y), y_ref, cfg.act, f"{name} y, call {call}")
        # both entry points run the same deterministic kernels: bit for bit
        assert torch.equal(act, run.act) and torch.equal(y, run.y), f"{name} call {call}"


def test_experts_static_rejects_bad_arguments():
    cfg = m.make_cfg(64, 256, 16, 4, 1, 128)
    lib = m._lib.lib()
    # null operands: rejected on the host before anything is launched
    assert lib.moe_experts_static(ctypes.byref(cfg), None, None, None, None, None, None,
                                  None, None, None, None) == 1
    # more groups than the fixed scratch holds (E + S beyond its capacity)
    big = m.make_cfg(64, 256, 1024, 4, 65, 128)
    assert lib.moe_experts_static(ctypes.byref(big), None, None, None, None, None, None,
                                  None, None, None, None) == 1
