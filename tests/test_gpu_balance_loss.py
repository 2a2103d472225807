"""Sequence-wise balance loss on the GPU against the float64 oracle.

The loss is computed from the router state of the forward just run (partial
logits in the workspace, the GPU's selection), so the oracle is fed the
float64 affinities of the same inputs and the GPU's selection: a tolerated
top-k flip cannot make the two disagree.  Covers both router kernels, the
configurations' own sequence lengths (the mini model's 32 x 256 batch, the
small configuration's 128-token context), a short last sequence and a NaN
token, which makes its own sequence's loss NaN and no other.
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
ALPHA = 1e-4

CASES = [
    ("tiny_fp32", dict(), 64),
    ("mini_bf16", dict(), 256),
    ("small_bf16", dict(), 128),
    ("v3_prefill", dict(T=2048), 1024),       # tensor-core router, two K slices
    ("v3_decode", dict(), 128),
    ("mini_bf16", dict(T=300), 128),          # last sequence of 44 tokens
]


def _run(wl, seq_len, mutate=None):
    inp = {n: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for n, v in I.make_inputs(wl, experts=False).items()}
    if mutate:
        mutate(inp)
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_ROUTE_ONLY)
    layer.forward(inp["x"])
    loss = layer.balance_loss(seq_len, ALPHA)
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    _, s = O.router_affinity(np64(inp["x"]), np64(inp["w_router"]))
    ref = O.sequence_balance_loss(s, npi(layer.topk_idx), seq_len, ALPHA)
    return loss.cpu().numpy().astype(np.float64), ref, layer


@pytest.mark.parametrize("name,over,seq_len", CASES,
                         ids=[f"{n}_{o.get('T', 'T')}_S{s}" for n, o, s in CASES])
def test_balance_loss_matches_oracle(name, over, seq_len):
    wl = I.WORKLOADS[name].with_(**over)
    got, ref, _ = _run(wl, seq_len)
    assert got.shape == ref.shape
    assert np.all(np.abs(got - ref) <= 2e-5 * np.abs(ref)), (got[:4], ref[:4])
    # balanced routing sits near alpha; nothing is far from it here
    assert np.all(ref > 0.5 * ALPHA) and np.all(ref < 4 * ALPHA)


def test_balance_loss_is_deterministic_and_isolates_nan():
    wl = I.WORKLOADS["mini_bf16"].with_(T=1024)

    def poison(inp):
        inp["x"][300, 5] = float("nan")

    got, ref, layer = _run(wl, 256, poison)
    assert np.isnan(got[1]) and np.isnan(ref[1])
    fin = np.arange(4) != 1
    assert np.all(np.abs(got[fin] - ref[fin]) <= 2e-5 * np.abs(ref[fin]))
    again = layer.balance_loss(256, ALPHA)
    torch.cuda.synchronize()
    assert np.array_equal(again.cpu().numpy()[fin], got[fin].astype(np.float32))
