"""The tensor-core router (bf16 tokens, 96 experts or more) against the oracle.

The router weights are split into three bf16 terms that carry their 24
significant bits, so every product is exact and the logits must agree with
the float64 logits to fp32 accumulation accuracy: each error within one fp32
epsilon of the logit's sum of |products| (an fp32 loop of d FMAs may in the
worst case be off by d of them), and on average within a tenth of it.  A
single tensor-core accumulator carried through a whole 7168-deep slice was 17
times over that bound (its additions lose toward zero); the kernel folds each
64-deep K step into fp32 registers instead.  The selection, gates and load
counts follow the same acceptance rules as the rest of the layer.  Cases
cover one token, ragged token tiles, several 256-expert blocks with padded
expert rows, split-K slices, one unsplit 7168-deep slice (25000 tokens: the
partial logits would pass 24 MiB with two), exact ties from duplicated router
rows, and a NaN token.
"""
EPS32 = 2.0 ** -23
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_moe_layer_fwd_b300 import inputs as I
from sparse_moe_layer_fwd_b300 import moe as M
from sparse_moe_layer_fwd_b300.layer import MoeLayer
from tests.parity import check_load, check_routing, np64, npi

pytestmark = pytest.mark.gpu


def _route(wl, inp):
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_ROUTE_ONLY)
    layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    return layer


def _inputs(wl):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
            for k, v in I.make_inputs(wl, experts=False).items()}


def _logits(layer, wl):
    """Sum of the split-K partial logits, in slice order, as the top-k does."""
    n_split = layer.regions["router_part"][1] // (wl.T * wl.E * 4)
    part = layer.region("router_part", torch.float32, (n_split, wl.T, wl.E))
    u = torch.zeros(wl.T, wl.E, dtype=torch.float32, device=part.device)
    for s in range(part.shape[0]):
        u += part[s]
    return u.double().cpu().numpy()


SHAPES = [
    dict(T=1, d=1024, E=256, k=8),
    dict(T=37, d=7168, E=256, k=8),      # one ragged token tile
    dict(T=300, d=2048, E=128, k=6),     # two token tiles, 128 padded expert rows
    dict(T=1000, d=7168, E=256, k=8),    # split-K over many slices
    dict(T=513, d=1024, E=384, k=8),     # two expert blocks, ragged third token tile
    dict(T=25000, d=7168, E=256, k=8),   # one slice over the whole model width
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"T{s['T']}_d{s['d']}_E{s['E']}_k{s['k']}" for s in SHAPES])
def test_tc_router_matches_oracle(shape):
    wl = I.custom(h=128, dtype="bf16", seed=11 + shape["T"], **shape)
    inp = _inputs(wl)
    layer = _route(wl, inp)
    x64, wr64, b64 = np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"])
    # logits: fp32 accumulation of exact products, against float64
    u_ref = x64 @ wr64.T
    u = _logits(layer, wl)
    if shape["T"] >= 25000:
        assert layer.regions["router_part"][1] == wl.T * wl.E * 4  # one K slice
    mag = np.abs(x64) @ np.abs(wr64).T  # sum of |products| per logit
    rel = np.abs(u - u_ref) / np.maximum(EPS32 * mag, 1e-300)
    assert rel.max() <= 1.0 and rel.mean() <= 0.1, (rel.max(), rel.mean())
    ref = O.route(x64, wr64, b64, wl.k)
    gidx = npi(layer.topk_idx)
    flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref, 1e-5)
    check_load(npi(layer.load_counts), gidx, ref["idx"], wl.E, flips)


def test_tc_router_duplicate_rows_tie_to_lower_index():
    wl = I.custom(T=300, d=7168, h=128, E=256, k=2, dtype="bf16", seed=3, bias="zero")
    inp = _inputs(wl)
    inp["w_router"][200] = inp["w_router"][17]
    inp["bias"][17] = inp["bias"][200] = 50.0
    layer = _route(wl, inp)
    u = _logits(layer, wl)
    # identical router rows give bit-identical logits in every token
    assert np.array_equal(u[:, 17], u[:, 200])
    idx = npi(layer.topk_idx)
    assert (idx[:, 0] == 17).all() and (idx[:, 1] == 200).all()
    g = layer.gates.cpu().numpy()
    assert np.array_equal(g[:, 0], g[:, 1])


def test_tc_router_nan_token_is_isolated():
    wl = I.custom(T=300, d=1024, h=128, E=256, k=8, dtype="bf16", seed=5)
    inp = _inputs(wl)
    inp["x"][123, 45] = float("nan")
    layer = _route(wl, inp)
    u = _logits(layer, wl)
    assert np.isnan(u[123]).all() and np.isfinite(np.delete(u, 123, axis=0)).all()
    # all biased scores NaN: they rank below every number, lowest indices win
    assert npi(layer.topk_idx)[123].tolist() == list(range(8))
    ref = O.route(np.delete(np64(inp["x"]), 123, 0), np64(inp["w_router"]), np64(inp["bias"]), wl.k)
    gidx = np.delete(npi(layer.topk_idx), 123, 0)
    gg = np.delete(layer.gates.cpu().numpy().astype(np.float64), 123, 0)
    check_routing(gidx, gg, ref, 1e-5)
