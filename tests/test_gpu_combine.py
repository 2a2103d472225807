"""The gated combine against the rows it combines, bit for bit.

y[t] = Y_sh[t] + sum_j gates[t, j] * Y_perm[inv[t*k + j]], in fp32 in that
slot order from the bf16 rows (the shared expert's row is Y_perm row
T*k + t), rounded once to bf16.  These tests recompute that sum on the host
from the workspace and require y to match it bit for bit wherever the
float64 value of the sum lies farther from a bf16 rounding midpoint than the
fp32 evaluation can move it (k + 1 roundings, each at most 2^-24 of the
running sum, bounded by the sum of the terms' magnitudes) -- nearer a
midpoint the fp32 result may round either way.  A wrong row, gate, slot or
token anywhere shows up as a mismatch far from any midpoint.
"""
import numpy as np
import pytest
import torch

from sparse_moe_layer_fwd_b300 import inputs as I
from sparse_moe_layer_fwd_b300 import moe as M
from sparse_moe_layer_fwd_b300.layer import MoeLayer

pytestmark = pytest.mark.gpu


def _bf16_midpoint_distance(v: np.ndarray) -> np.ndarray:
    """Distance of each float64 value to the nearest point halfway between
    two adjacent bf16 values (the one between v truncated to bf16 and the
    next bf16 away from zero)."""
    bits = v.astype(np.float32).view(np.uint32).astype(np.uint64)
    lo = (bits & ~np.uint64(0xFFFF)).astype(np.uint32).view(np.float32).astype(np.float64)
    step = np.abs(np.spacing(lo.astype(np.float32)).astype(np.float64)) * 65536.0
    mid = lo + np.copysign(step / 2, v)
    return np.abs(v - mid)


def _check_fold(layer, inp, wl):
    y = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    T, k, d = wl.T, wl.k, wl.d
    TK = T * k
    yp = layer.region("y_perm", torch.bfloat16, (TK + T, d)).float().cpu().numpy().astype(np.float64)
    inv = layer.region("inv", torch.int32, (TK,)).cpu().numpy().astype(np.int64).reshape(T, k)
    g = layer.gates.cpu().numpy().astype(np.float64)
    ref = yp[TK:TK + T].copy()
    mag = np.abs(ref)
    for j in range(k):
        term = g[:, j:j + 1] * yp[inv[:, j]]
        ref += term
        mag += np.abs(term)
    got = y.float().cpu().numpy().astype(np.float64)
    ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16).float().numpy().astype(np.float64)
    near_mid = _bf16_midpoint_distance(ref) <= (k + 1) * 2.0 ** -24 * mag
    bad = (got != ref_bf16) & ~near_mid
    assert near_mid.mean() < 1e-2, near_mid.mean()
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:5])
    # the shared rows really are the shared expert's: not all zero
    assert np.abs(yp[TK:TK + T]).max() > 0


@pytest.mark.parametrize("name,kw", [
    ("v3_32experts", None),
    # ragged: 1000 tokens, shared tiles of 250
    ("ragged", dict(T=1000, d=1024, h=512, E=32, k=4, dtype="bf16", seed=21)),
])
def test_combine_matches_its_arithmetic(name, kw):
    wl = I.WORKLOADS["v3_prefill_32experts"] if kw is None else I.custom(**kw)
    inp = I.make_inputs(wl, device="cuda")
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    _check_fold(layer, inp, wl)
    del layer, inp
    torch.cuda.empty_cache()


def test_combine_block_scaled():
    """The same with both products on block-scaled e4m3 codes."""
    wl = I.custom(T=1000, d=1024, h=512, E=32, k=4, dtype="bf16", seed=22)
    inp = I.make_inputs(wl, device="cuda")
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_FP8_BLOCK)
    _check_fold(layer, inp, wl)
    del layer, inp
    torch.cuda.empty_cache()


def test_combine_repeats():
    """Back-to-back forwards on one workspace give the same y."""
    wl = I.custom(T=1000, d=1024, h=512, E=32, k=4, dtype="bf16", seed=23)
    inp = I.make_inputs(wl, device="cuda")
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    y0 = layer.forward(inp["x"]).clone()
    for _ in range(5):
        y1 = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    assert torch.equal(y0, y1)
    _check_fold(layer, inp, wl)
    del layer, inp
    torch.cuda.empty_cache()
