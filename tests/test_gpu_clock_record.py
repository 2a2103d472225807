"""The tensor-core kernels' in-band clock record (moe_sm_clock_record): after
forwards of the V3-width 32-expert layer, the gate/up, down and router slots
hold cycles and nanoseconds whose ratio is a plausible SM clock (the
32-expert layer routes on the CUDA cores, so the router slot stays empty);
reset clears them; a route-only pass with 256 experts (the tensor-core
router) touches the router slot only."""
import pytest
import torch

from sparse_moe_layer_fwd_b300 import inputs as I
from sparse_moe_layer_fwd_b300 import moe as M
from sparse_moe_layer_fwd_b300.layer import MoeLayer

pytestmark = pytest.mark.gpu


def test_clock_record_counts_the_expert_gemms():
    wl = I.WORKLOADS["v3_prefill_32experts"]
    inp = I.make_inputs(wl, device="cuda")
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    layer.forward(inp["x"])
    torch.cuda.synchronize()
    M.moe_sm_clock_record(reset=True)
    zero = M.moe_sm_clock_record()
    assert all(v["cycles"] == 0 and v["ns"] == 0 for v in zero.values())
    for _ in range(3):
        layer.forward(inp["x"])
    torch.cuda.synchronize()
    rec = M.moe_sm_clock_record(reset=True)
    assert M.moe_last_error() == M.MOE_OK
    for slot in ("gate_up", "down"):
        assert rec[slot]["ns"] > 0, slot
        # every CTA's span, summed: between 300 MHz and the part's 2032 MHz
        # maximum (with some margin for the counters' granularity)
        assert 300.0 < rec[slot]["mhz"] < 2200.0, (slot, rec[slot]["mhz"])
    assert rec["backward"]["ns"] == 0 and rec["router"]["ns"] == 0
    del layer, inp
    torch.cuda.empty_cache()
    wl = I.custom(T=2048, d=1024, h=512, E=256, k=8, dtype="bf16", seed=31)
    inp = I.make_inputs(wl, device="cuda")
    ro = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_ROUTE_ONLY)
    ro.forward(inp["x"])
    torch.cuda.synchronize()
    rec = M.moe_sm_clock_record(reset=True)
    assert M.moe_last_error() == M.MOE_OK
    assert rec["router"]["ns"] > 0 and 300.0 < rec["router"]["mhz"] < 2200.0
    assert rec["gate_up"]["ns"] == 0 and rec["down"]["ns"] == 0
