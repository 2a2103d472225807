"""The failure path of the bounded device waits, on the GPU, without a fault.

A kernel whose only wait is on a barrier that nothing arrives on gives up
after its limit, sets the device error word and returns; the host reads
MOE_ERR_DEVICE_TIMEOUT from moe_last_error, the next read is MOE_OK again, and
the context stays usable: a forward right after it matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_moe_layer_fwd_b300 import inputs as I
from sparse_moe_layer_fwd_b300 import moe as M
from sparse_moe_layer_fwd_b300.layer import MoeLayer
from tests.parity import check_output, np64, npi

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_context_survives():
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    t0 = time.perf_counter()
    M.moe_selftest_timeout(200)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert M.moe_last_error() == M.ERR_CODE["MOE_ERR_DEVICE_TIMEOUT"]
    assert M.moe_last_error() == M.MOE_OK  # read-and-reset
    assert 0.15 < waited < 5.0, waited
    # the context is intact: a forward afterwards is correct
    wl = I.custom(T=300, d=256, h=256, E=16, k=4, dtype="bf16", seed=21)
    inp = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in I.make_inputs(wl).items()}
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    y = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    ex = (np64(inp["w_gate"]), np64(inp["w_up"]), np64(inp["w_down"]))
    sh = (np64(inp["sh_gate"]), np64(inp["sh_up"]), np64(inp["sh_down"]))
    ref = O.moe_forward_dense(np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"]), ex, sh,
                              wl.k, idx_override=npi(layer.topk_idx))
    check_output(np64(y), ref["y"], "bf16")
