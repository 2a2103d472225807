"""The layer inside CUDA graphs.

A forward enqueues only kernels (no allocation, no host synchronisation, no
host-side decision that depends on device data), so it can be captured once
and replayed.  Replays must reproduce the eager results bit for bit (every
kernel is deterministic), also after new token values are written into the
captured input buffer; the same holds for a captured training step (forward,
backward, bias update).
"""
import pytest
import torch

from sparse_moe_layer_fwd_b300 import inputs as I
from sparse_moe_layer_fwd_b300 import moe as M
from sparse_moe_layer_fwd_b300.layer import MoeLayer

pytestmark = pytest.mark.gpu


def _inputs(wl):
    return {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in I.make_inputs(wl).items()}


@pytest.mark.parametrize("shape", [dict(T=700, d=512, h=256, E=128, k=8),   # tensor-core router, pair tiles
                                   dict(T=64, d=256, h=256, E=16, k=4)],    # FFMA router, 1-SM tiles
                         ids=["E128", "E16"])
def test_forward_graph_replays_bit_exact(shape):
    wl = I.custom(dtype="bf16", seed=31, **shape)
    inp = _inputs(wl)
    x = inp["x"]
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    layer.forward(x)  # eager call first: one-time host set-up happens outside the capture
    torch.cuda.synchronize()
    ref = (layer.y.clone(), layer.topk_idx.clone(), layer.gates.clone(), layer.load_counts.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x)
    for t in (layer.y, layer.topk_idx, layer.gates, layer.load_counts):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    for a, b in zip((layer.y, layer.topk_idx, layer.gates, layer.load_counts), ref):
        assert torch.equal(a, b)
    # new tokens in the captured buffer: the replay follows them
    x.copy_(torch.randn(x.shape, generator=torch.Generator().manual_seed(5)).to(x.dtype).cuda())
    g.replay()
    eager = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    eager.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(layer.y, eager.y) and torch.equal(layer.topk_idx, eager.topk_idx)


def test_training_step_graph_replays_bit_exact():
    wl = I.custom(T=500, d=256, h=256, E=8, k=2, dtype="bf16", seed=32)
    inp = _inputs(wl)
    x = inp["x"]
    dy = torch.randn((wl.T, wl.d), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).cuda()
    bias0 = inp["bias"].clone()
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_TRAINING)
    layer.forward(x)
    g0 = layer.backward(x, dy)
    layer.bias_update(1e-3)
    torch.cuda.synchronize()
    ref = {n: v.clone() for n, v in g0.items()}
    ref_bias = inp["bias"].clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x)
        grads = layer.backward(x, dy)  # its output tensors come from the graph's pool
        layer.bias_update(1e-3)
    inp["bias"].copy_(bias0)
    graph.replay()
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    assert torch.equal(inp["bias"], ref_bias)
    for n in ref:
        assert torch.equal(grads[n], ref[n]), n
