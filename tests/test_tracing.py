"""Launch tracing (moe_trace_enable / moe_trace_read): every kernel a forward
launches is recorded once per launch with its event-timed duration; nothing
is recorded while tracing is off."""
import pytest
import torch

from moe_inputs import small_cases
from tests._util import gpu_inputs

m = pytest.importorskip("mixture_experts_layer_88_b300")


def test_trace_read_without_records_needs_no_gpu():
    m.trace_enable(False)
    assert m.trace_read_all() == []


@pytest.mark.gpu
def test_forward_kernels_traced_once_each():
    cfg = small_cases()["small_bf16"]
    g, _ = gpu_inputs(cfg)
    layer = m.MoeLayer(m.cfg_from_layer(cfg), g, device="cuda")
    layer.forward(g["x"])                     # first call outside the trace
    torch.cuda.synchronize()
    m.trace_enable(True)
    m.trace_read_all()
    layer.forward(g["x"])
    layer.update_bias()
    torch.cuda.synchronize()
    rec = {name: (n, ms) for name, n, ms in m.trace_read_all()}
    m.trace_enable(False)
    # E <= 256 experts: the router is one fused kernel (no logits in memory)
    for name in ("router_fused", "dispatch_count", "dispatch_scan", "dispatch_rank",
                 "dispatch_scatter", "build_groups",
                 "gemm_gateup_swiglu", "gemm_down", "combine", "update_bias"):
        assert name in rec, f"{name} not traced: {sorted(rec)}"
        n, ms = rec[name]
        assert n == 1 and ms > 0.0
    assert "gemm_router" not in rec and "router_topk" not in rec
    assert m.trace_read_all() == []           # read clears the record
    layer.forward(g["x"])                     # tracing off: nothing recorded
    torch.cuda.synchronize()
    assert m.trace_read_all() == []


@pytest.mark.gpu
def test_wide_router_traces_split_gemm_and_topk():
    """More than 256 experts: the split-K router GEMM and the top-K kernel."""
    cfg = small_cases()["wide_e"]
    g, _ = gpu_inputs(cfg)
    layer = m.MoeLayer(m.cfg_from_layer(cfg), g, device="cuda")
    layer.forward(g["x"])
    torch.cuda.synchronize()
    m.trace_enable(True)
    m.trace_read_all()
    layer.forward(g["x"])
    torch.cuda.synchronize()
    rec = {name: n for name, n, _ in m.trace_read_all()}
    m.trace_enable(False)
    assert rec.get("gemm_router") == 1 and rec.get("router_topk") == 1
    assert "router_fused" not in rec


@pytest.mark.gpu
def test_trace_events_captured_into_a_graph():
    """Steps captured into a CUDA graph with tracing on record their events as
    graph nodes: after a replay the trace holds every launch of the captured
    steps with its device time, as eager steps would."""
    cfg = small_cases()["small_bf16"]
    g, _ = gpu_inputs(cfg)
    layer = m.MoeLayer(m.cfg_from_layer(cfg), g, device="cuda")
    out = torch.empty_like(g["x"])
    layer.step(g["x"], out)
    torch.cuda.synchronize()
    m.trace_enable(True)
    m.trace_read_all()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(3):
            layer.step(g["x"], out)
    graph.replay()
    torch.cuda.synchronize()
    rec = {name: (n, ms) for name, n, ms in m.trace_read_all()}
    m.trace_enable(False)
    assert m.get_status() == 0
    for name in ("router_fused", "dispatch_scatter", "gemm_gateup_swiglu", "gemm_down",
                 "combine", "update_bias"):
        n, ms = rec[name]
        assert n == 3 and ms > 0.0, (name, n, ms)
