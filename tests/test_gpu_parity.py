"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Small and medium workloads (the oracle finishes each in seconds): the tiny
fp32 layer, the mini-model bf16 layer, the 200-step bias-balancing run, and
edge cases (one token, ragged token counts, k = E, one expert, non-power-of-
two E, empty batch, NaN tokens, exact ties).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_moe_layer_fwd_b300 import inputs as I
from sparse_moe_layer_fwd_b300 import moe as M
from sparse_moe_layer_fwd_b300.layer import MoeLayer
from tests.parity import check_load, check_output, check_routing, np64, npi

pytestmark = pytest.mark.gpu
GAMMA = 1e-3


def _to_cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _oracle_weights(inp):
    ex = (np64(inp["w_gate"]), np64(inp["w_up"]), np64(inp["w_down"]))
    sh = (np64(inp["sh_gate"]), np64(inp["sh_up"]), np64(inp["sh_down"]))
    return ex, sh


def run_and_check(wl, inp, flags=0, check_bias=True):
    """Full forward through the C ABI, then every check against the oracle."""
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, flags)
    y = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    x64, wr64, b64 = np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"])
    ref = O.route(x64, wr64, b64, wl.k)
    gidx, ggates = npi(layer.topk_idx), layer.gates.cpu().numpy().astype(np.float64)
    flips = check_routing(gidx, ggates, ref, {"f32": 1e-6, "bf16": 1e-5}[wl.dtype])
    gload = npi(layer.load_counts)
    check_load(gload, gidx, ref["idx"], wl.E, flips)
    ex, sh = _oracle_weights(inp)
    out = O.moe_forward_dense(x64, wr64, b64, ex, sh, wl.k, idx_override=gidx)
    stats = check_output(np64(y), out["y"], wl.dtype)
    if check_bias:
        b_before = inp["bias"].cpu().numpy().copy()
        layer.bias_update(GAMMA)
        torch.cuda.synchronize()
        b_ref = O.bias_update(b_before, gload, GAMMA, wl.T * wl.k)
        assert np.array_equal(inp["bias"].cpu().numpy(), b_ref)
    return layer, stats, flips


def test_tiny_fp32_layer():
    wl = I.WORKLOADS["tiny_fp32"]
    inp = _to_cuda(I.make_inputs(wl))
    _, stats, _ = run_and_check(wl, inp)
    assert stats["rel_l2"] < 1e-5


def test_dispatch_is_a_stable_counting_sort():
    wl = I.WORKLOADS["tiny_fp32"].with_(T=300)
    inp = _to_cuda(I.make_inputs(wl))
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    layer.forward(inp["x"])
    torch.cuda.synchronize()
    TK = wl.T * wl.k
    idx = npi(layer.topk_idx).ravel()
    perm = npi(layer.region("perm", torch.int32, (TK,)))
    inv = npi(layer.region("inv", torch.int32, (TK,)))
    # pairs sorted by expert, ties in pair order: numpy's stable argsort
    assert np.array_equal(perm, np.argsort(idx, kind="stable"))
    assert np.array_equal(inv[perm], np.arange(TK))
    xp = layer.region("x_perm", torch.float32, (TK, wl.d)).cpu()
    assert torch.equal(xp, inp["x"].cpu()[torch.from_numpy(perm // wl.k)])
    groups = npi(layer.region("groups", torch.int32, (5 * wl.E + 10,)))
    load = np.bincount(idx, minlength=wl.E)
    off = groups[:wl.E + 2]
    assert np.array_equal(off[:wl.E], np.concatenate([[0], np.cumsum(load)[:-1]]))
    assert off[wl.E] == TK and off[wl.E + 1] == TK + wl.T


def test_bias_dynamics_200_steps():
    """Route + dispatch + bias update on a fresh batch every step; counts and
    the updated bias must be bit-exact each step, the oracle being fed the
    GPU's previous bias."""
    wl = I.WORKLOADS["bias_dynamics"]
    inp = I.make_inputs(wl)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    layer = MoeLayer.from_inputs(dev, wl.k, wl.dtype, M.MOE_ROUTE_ONLY)
    wr64 = np64(inp["w_router"])
    shares = []
    x = dev["x"]
    for step in range(wl.steps):
        if step > 0:
            x = I.next_x(wl, inp, "cuda")
        b_prev = dev["bias"].cpu().numpy().copy()
        layer.forward(x)
        layer.bias_update(GAMMA)
        torch.cuda.synchronize()
        ref = O.route_and_update(np64(x), wr64, b_prev, wl.k, GAMMA)
        gidx = npi(layer.topk_idx)
        flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref, 1e-6)
        gload = npi(layer.load_counts)
        check_load(gload, gidx, ref["idx"], wl.E, flips)
        b_ref = O.bias_update(b_prev, gload, GAMMA, wl.T * wl.k)
        assert np.array_equal(dev["bias"].cpu().numpy(), b_ref), f"step {step}"
        if flips == 0:
            assert np.array_equal(dev["bias"].cpu().numpy(), ref["bias_new"])
        shares.append(gload / (wl.T * wl.k))
    shares = np.array(shares)
    # the skewed start is pulled towards the uniform share 1/16 = 6.25%
    spread0 = shares[:10].max(axis=1) - shares[:10].min(axis=1)
    spread1 = shares[-10:].max(axis=1) - shares[-10:].min(axis=1)
    assert spread1.mean() < spread0.mean()


def test_mini_bf16_layer():
    wl = I.WORKLOADS["mini_bf16"]
    inp = _to_cuda(I.make_inputs(wl))
    _, stats, _ = run_and_check(wl, inp)
    assert stats["rel_l2"] < 1e-2


def test_tensor_cores_match_cuda_core_cross_check():
    wl = I.WORKLOADS["mini_bf16"].with_(T=2048)
    inp = _to_cuda(I.make_inputs(wl))
    a = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    b = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_SIMT_EXPERTS)
    ya, yb = a.forward(inp["x"]).clone(), b.forward(inp["x"])
    torch.cuda.synchronize()
    assert torch.equal(a.topk_idx, b.topk_idx)
    ha = a.region("h", torch.bfloat16, (wl.T * wl.k + wl.T, wl.h)).double()
    hb = b.region("h", torch.bfloat16, (wl.T * wl.k + wl.T, wl.h)).double()
    assert ((ha - hb).norm() / hb.norm()).item() < 4e-3
    assert ((ya.double() - yb.double()).norm() / yb.double().norm()).item() < 4e-3


EDGE = [
    dict(T=1, d=256, h=128, E=16, k=4),
    dict(T=37, d=256, h=128, E=16, k=4),
    dict(T=50, d=128, h=256, E=8, k=8),      # k = E: every expert selected
    dict(T=64, d=128, h=128, E=1, k=1),      # one routed expert, gate 1
    dict(T=200, d=256, h=128, E=20, k=3),    # E not a power of two
    dict(T=600, d=128, h=128, E=4, k=2),     # several token tiles per expert
    dict(T=100, d=384, h=640, E=40, k=6),
    dict(T=64, d=128, h=128, E=1024, k=32),  # the largest E and k the description accepts
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", EDGE, ids=[f"T{s['T']}_d{s['d']}_h{s['h']}_E{s['E']}_k{s['k']}" for s in EDGE])
def test_edge_shapes(shape, dtype):
    wl = I.custom(dtype=dtype, seed=shape["T"] + shape["E"], **shape)
    inp = _to_cuda(I.make_inputs(wl))
    run_and_check(wl, inp)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_batch(dtype):
    wl = I.custom(T=0, d=256, h=128, E=16, k=4, dtype=dtype)
    inp = _to_cuda(I.make_inputs(wl.with_(T=8)))
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, T=0)
    layer.load_counts.fill_(7)
    layer.forward(inp["x"][:0])
    torch.cuda.synchronize()
    assert int(layer.load_counts.abs().sum()) == 0
    b0 = inp["bias"].clone()
    layer.bias_update(GAMMA)
    torch.cuda.synchronize()
    # zero tokens: every expert is exactly at the mean load, nothing moves
    assert torch.equal(inp["bias"], b0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nan_token_is_isolated(dtype):
    wl = I.custom(T=40, d=256, h=128, E=16, k=4, dtype=dtype, seed=5)
    inp = _to_cuda(I.make_inputs(wl))
    inp["x"][7, 3] = float("nan")
    layer, _, _ = run_and_check(wl, inp, check_bias=False)
    # a NaN token's scores are all NaN: they rank below every number and
    # the lowest indices win the ties
    assert npi(layer.topk_idx)[7].tolist() == [0, 1, 2, 3]
    assert torch.isnan(layer.y[7].float()).all()
    assert torch.isfinite(layer.y[torch.arange(40, device="cuda") != 7].float()).all()


@pytest.mark.parametrize("dtype,d", [("f32", 256), ("bf16", 7168)])
def test_duplicate_router_rows_tie_to_lower_index(dtype, d):
    wl = I.custom(T=64, d=d, h=128, E=16, k=2, dtype=dtype, seed=3, bias="zero")
    inp = _to_cuda(I.make_inputs(wl))
    inp["w_router"][9] = inp["w_router"][4]
    inp["bias"][4] = inp["bias"][9] = 50.0
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    layer.forward(inp["x"])
    torch.cuda.synchronize()
    idx = npi(layer.topk_idx)
    # experts 4 and 9 have identical logits for every token; both are
    # selected, 4 in the first slot
    assert (idx[:, 0] == 4).all() and (idx[:, 1] == 9).all()
    g = layer.gates.cpu().numpy()
    assert np.array_equal(g[:, 0], g[:, 1]) and np.allclose(g, 0.5, atol=0)


def test_host_io_entry_matches_device_entry():
    wl = I.WORKLOADS["mini_bf16"].with_(T=1024)
    inp = _to_cuda(I.make_inputs(wl))
    a = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    ya = a.forward(inp["x"]).cpu()
    b = MoeLayer.from_inputs(inp, wl.k, wl.dtype, host_io=True)
    x_host = inp["x"].cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    b.forward_host_io(x_host, y_host)
    torch.cuda.synchronize()
    assert torch.equal(ya, y_host)
    assert torch.equal(a.topk_idx, b.topk_idx)


def test_error_word_is_clear():
    assert M.moe_last_error() == M.MOE_OK


def test_small_config_layer():
    """The "small" configuration: 8 routed experts, top-2 (full layer)."""
    wl = I.WORKLOADS["small_bf16"]
    inp = _to_cuda(I.make_inputs(wl))
    _, stats, _ = run_and_check(wl, inp)
    assert stats["rel_l2"] < 1e-2


# routing over a spread of (E, k), both router kernels (CUDA cores below 96
# experts or for fp32 tokens, tensor cores from 96 experts with bf16 tokens)
EK = [(8, 1), (8, 2), (8, 8), (32, 3), (64, 6), (96, 8), (128, 1), (160, 5), (512, 8), (1024, 32)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("E,k", EK, ids=[f"E{e}_k{k}" for e, k in EK])
def test_routing_over_expert_counts(E, k, dtype):
    wl = I.custom(T=333, d=512, h=128, E=E, k=k, dtype=dtype, seed=E + k)
    inp = {n: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for n, v in I.make_inputs(wl, experts=False).items()}
    b_before = inp["bias"].cpu().numpy().copy()
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_ROUTE_ONLY)
    layer.forward(inp["x"])
    layer.bias_update(GAMMA)
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    ref = O.route(np64(inp["x"]), np64(inp["w_router"]), b_before.astype(np.float64), k)
    gidx = npi(layer.topk_idx)
    flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref,
                          {"f32": 1e-6, "bf16": 1e-5}[dtype])
    gload = npi(layer.load_counts)
    check_load(gload, gidx, ref["idx"], E, flips)
    assert np.array_equal(inp["bias"].cpu().numpy(), O.bias_update(b_before, gload, GAMMA, wl.T * k))


def test_many_experts_on_cta_pair_tiles():
    """384 experts (two 256-expert router blocks, 385 groups in the tile
    table) with about 96 tokens per expert, so both GEMMs take the CTA-pair
    tiles; the sparse oracle on every row."""
    wl = I.custom(T=4608, d=256, h=256, E=384, k=8, dtype="bf16", seed=17)
    inp = _to_cuda(I.make_inputs(wl))
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    y = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    x64, wr64, b64 = np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"])
    ref = O.route(x64, wr64, b64, wl.k)
    gidx = npi(layer.topk_idx)
    flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref, 1e-5)
    check_load(npi(layer.load_counts), gidx, ref["idx"], wl.E, flips)
    ex, sh = _oracle_weights(inp)
    out = O.moe_forward_sparse(x64, wr64, b64, ex, sh, wl.k, idx_override=gidx)
    check_output(np64(y), out["y"], "bf16")
