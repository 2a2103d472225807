"""Backward of the layer on the GPU against the float64 oracle.

The oracle (pinned by finite differences of the forward oracle) is evaluated
on the GPU's own selection, so a tolerated near-tie flip cannot make the two
differ.  Every gradient -- tokens, routed and shared expert weights, router
weights -- is compared with relative L2 error below 1e-2 (the layer's bf16
bar: the backward rounds g*dy, dH and dA|dB to bf16 and accumulates in
fp32), and locally: every row (one output unit of one expert, one token of
dx, one expert of dW_r) within 3e-2 of the larger of its reference row's
norm and the tensor's typical row norm, and dx element by element within
5e-2 * rms(reference).  (A weight-gradient element of an expert with a
handful of tokens is a sum of a few products of heavy-tailed factors, so
its largest elements sit far above the tensor's rms; a per-row bound
catches a localised error without that bias.)
Shapes cover ragged token tiles, experts that no token selected (their
gradients must be exactly zero), partial 256-row blocks of the weight
gradients, and several token tiles per expert.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_moe_layer_fwd_b300 import inputs as I
from sparse_moe_layer_fwd_b300 import moe as M
from sparse_moe_layer_fwd_b300.layer import MoeLayer
from tests.parity import np64, npi

pytestmark = pytest.mark.gpu
TOL = 1e-2
MAX_ABS_RMS = 5e-2
ROW_TOL = 3e-2

SHAPES = [
    dict(T=300, d=256, h=256, E=8, k=2),
    dict(T=1000, d=512, h=384, E=16, k=4),    # partial 256-row blocks of dW
    dict(T=64, d=256, h=128, E=40, k=2),      # many experts without tokens
    dict(T=513, d=384, h=256, E=12, k=3),     # ragged tiles, 384 = 1.5 blocks
    dict(T=2048, d=256, h=256, E=4, k=2),     # several token tiles per expert
]


def _rel(a, b):
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


def _max_abs_over_rms(a, b):
    """max |a - b| in units of rms(b) (0 where b is all zero and a equals it)."""
    rms = np.sqrt(np.mean(b * b))
    mx = np.abs(a - b).max()
    return mx / rms if rms > 0 else (0.0 if mx == 0 else np.inf)


def _worst_row(a, b):
    """Largest row error of a gradient (rows along the last axis), each row's
    error measured against the larger of its own reference norm and the rms
    of the tensor's non-zero reference row norms: a wrong row shows up at
    any size, while a row whose reference nearly cancels (a few tokens whose
    upstream gradient is close to zero) is held to the tensor's scale rather
    than to its own.  Rows whose reference is zero must be exactly zero."""
    a2, b2 = a.reshape(-1, a.shape[-1]), b.reshape(-1, b.shape[-1])
    nb = np.linalg.norm(b2, axis=1)
    nd = np.linalg.norm(a2 - b2, axis=1)
    zero = nb == 0
    assert np.all(nd[zero] == 0), "non-zero gradient where the reference is zero"
    if not (~zero).any():
        return 0.0
    typical = np.sqrt(np.mean(nb[~zero] ** 2))
    return float((nd[~zero] / np.maximum(nb[~zero], typical)).max())


CASES = [(s, False) for s in SHAPES] + [(SHAPES[1], True), (SHAPES[3], True), (SHAPES[4], True)]


@pytest.mark.parametrize("shape,grad_bf16", CASES,
                         ids=[f"T{s['T']}_d{s['d']}_h{s['h']}_E{s['E']}_k{s['k']}" + ("_bf16grad" if b else "")
                              for s, b in CASES])
def test_backward_matches_oracle(shape, grad_bf16):
    """(grad_bf16: MOE_GRAD_BF16, the weight gradients rounded once to bf16 --
    a relative error of at most 2^-9 per element on top of the fp32 path's,
    inside the same bounds.)"""
    wl = I.custom(dtype="bf16", seed=7 + shape["T"], **shape)
    inp = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in I.make_inputs(wl).items()}
    flags = M.MOE_TRAINING | (M.MOE_GRAD_BF16 if grad_bf16 else 0)
    layer = MoeLayer.from_inputs(inp, wl.k, "bf16", flags)
    layer.forward(inp["x"])
    gen = torch.Generator().manual_seed(wl.T + 99)
    dy = torch.randn((wl.T, wl.d), generator=gen).to(torch.bfloat16).cuda()
    g = layer.backward(inp["x"], dy)
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    ex = (np64(inp["w_gate"]), np64(inp["w_up"]), np64(inp["w_down"]))
    sh = (np64(inp["sh_gate"]), np64(inp["sh_up"]), np64(inp["sh_down"]))
    idx = npi(layer.topk_idx)
    ref = O.moe_backward_dense(np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"]), ex, sh,
                               wl.k, np64(dy), idx_override=idx)
    errs = {n: _rel(np64(g[n]), ref[n]) for n in
            ["dx", "dW_gate", "dW_up", "dW_down", "dsh_gate", "dsh_up", "dsh_down", "dW_router"]}
    assert all(v < TOL for v in errs.values()), errs
    rows = {n: _worst_row(np64(g[n]), ref[n]) for n in errs}
    assert all(v <= ROW_TOL for v in rows.values()), rows
    assert _max_abs_over_rms(np64(g["dx"]), ref["dx"]) <= MAX_ABS_RMS
    empty = np.setdiff1d(np.arange(wl.E), np.unique(idx))
    for n in ["dW_gate", "dW_up", "dW_down"]:
        assert g[n].dtype == (torch.bfloat16 if grad_bf16 else torch.float32)
        assert np.all(np64(g[n])[empty] == 0.0)
    assert np.all(np64(g["dW_router"])[empty] == 0.0)


def test_backward_is_deterministic():
    wl = I.custom(T=700, d=256, h=256, E=8, k=2, dtype="bf16", seed=3)
    inp = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in I.make_inputs(wl).items()}
    layer = MoeLayer.from_inputs(inp, wl.k, "bf16", M.MOE_TRAINING)
    dy = torch.randn((wl.T, wl.d), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    layer.forward(inp["x"])
    a = {n: v.clone() for n, v in layer.backward(inp["x"], dy).items()}
    layer.forward(inp["x"])
    b = layer.backward(inp["x"], dy)
    torch.cuda.synchronize()
    for n in a:
        assert torch.equal(a[n], b[n]), n
