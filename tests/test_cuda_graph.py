"""The layer step (forward + bias update) captured into a CUDA graph and
replayed equals the eager step bit for bit, step after step: every launch is
stream-ordered, allocates nothing and, after the first eager call on a device,
makes no host query."""
import pytest
import torch

from moe_inputs import small_cases
from tests._util import gpu_inputs

pytestmark = pytest.mark.gpu

m = pytest.importorskip("mixture_experts_layer_88_b300")


@pytest.mark.parametrize("name,prenorm", [("small_bf16", False), ("small_fp8", False),
                                          ("softmax_norenorm", False), ("small_bf16", True)])
def test_layer_step_replayed_from_cuda_graph(name, prenorm):
    cfg = small_cases()[name]
    g, _ = gpu_inputs(cfg)
    kw = dict(norm_w=g["norm_w"]) if prenorm else {}
    eager = m.MoeLayer(m.cfg_from_layer(cfg), dict(g, bias=g["bias"].clone()), device="cuda",
                       **kw)
    graphed = m.MoeLayer(m.cfg_from_layer(cfg), dict(g, bias=g["bias"].clone()), device="cuda",
                         **kw)
    x = g["x"]
    out_e, out_g = torch.empty_like(x), torch.empty_like(x)
    eager.step(x, out_e)              # first calls: kernel attributes, occupancy, buffers
    graphed.step(x, out_g)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        graphed.step(x, out_g)
    for _ in range(3):                # the bias moves every step: replay must follow it
        eager.step(x, out_e)
        graph.replay()
        torch.cuda.synchronize()
        assert m.get_status() == 0
        assert torch.equal(eager.idx, graphed.idx) and torch.equal(eager.counts, graphed.counts)
        assert torch.equal(out_e, out_g)
        assert torch.equal(eager.bias, graphed.bias)
