"""moe_route_noalloc: routing whose scratch is the library's static device
array, for callers that must not allocate device memory or pass a workspace
(for example a plugin whose host framework owns all device memory).

It must give exactly what moe_forward gives with MOE_ROUTE_ONLY, on two calls
in a row (the second call must not be affected by what the first left in the
shared array), and must refuse a problem whose scratch would not fit.  This
file is collected last on purpose, and works alone in a fresh process too.
"""
import pytest
import torch

from sparse_moe_layer_fwd_b300 import moe as M

pytestmark = pytest.mark.gpu


def _route_reference(desc_ro, x, w_router, bias, T, k, E):
    """The existing entry point: moe_forward with MOE_ROUTE_ONLY and a
    caller-allocated workspace."""
    ws_bytes = M.moe_workspace_size(desc_ro)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    load = torch.empty((E,), dtype=torch.int32, device="cuda")
    M.moe_forward(desc_ro, x, w_router, bias, None, None, None, idx, gates, load, ws, ws_bytes,
                  torch.cuda.current_stream())
    return idx, gates, load


@pytest.mark.parametrize("shape", [
    dict(T=256, d=256, E=16, k=4, dtype="f32"),
    dict(T=1000, d=7168, E=256, k=8, dtype="bf16"),
    dict(T=8192, d=7168, E=256, k=8, dtype="bf16"),
], ids=["tiny_fp32", "v3_router_1000_tokens", "v3_router_8192_tokens"])
def test_noalloc_routing_matches_workspace_routing_twice(shape):
    T, d, E, k, dtype = shape["T"], shape["d"], shape["E"], shape["k"], shape["dtype"]
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator("cuda").manual_seed(T + E)
    w_router = torch.randn((E, d), generator=g, device="cuda") / d ** 0.5
    bias = (torch.rand((E,), generator=g, device="cuda") - 0.5) * 0.02
    desc = M.make_desc(T, d, 128, E, k, dtype)
    desc_ro = M.make_desc(T, d, 128, E, k, dtype, M.MOE_ROUTE_ONLY)
    assert M.moe_workspace_size(desc_ro) <= M.MOE_STATIC_SCRATCH_BYTES
    for call in range(2):  # two calls in a row, different batches
        x = torch.randn((T, d), generator=g, device="cuda").to(tdt)
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        gates = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
        load = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        M.moe_route_noalloc(desc, x, w_router, bias, idx, gates, load,
                            torch.cuda.current_stream())
        ref_idx, ref_gates, ref_load = _route_reference(desc_ro, x, w_router, bias, T, k, E)
        torch.cuda.synchronize()
        assert M.moe_last_error() == M.MOE_OK
        assert torch.equal(idx, ref_idx), f"call {call}"
        assert torch.equal(gates, ref_gates), f"call {call}"  # same kernels: identical
        assert torch.equal(load, ref_load), f"call {call}"
        assert int(load.sum()) == T * k


def test_noalloc_calls_reserve_no_device_memory():
    """After one call (which may load the library's module on this device and
    with it the static array), further calls leave the device's free memory
    unchanged: they allocate nothing."""
    T, d, E, k = 512, 1024, 64, 6
    g = torch.Generator("cuda").manual_seed(5)
    x = torch.randn((T, d), generator=g, device="cuda").to(torch.bfloat16)
    w_router = torch.randn((E, d), generator=g, device="cuda") / d ** 0.5
    bias = torch.zeros((E,), device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    load = torch.empty((E,), dtype=torch.int32, device="cuda")
    desc = M.make_desc(T, d, 128, E, k, "bf16")
    M.moe_route_noalloc(desc, x, w_router, bias, idx, gates, load, torch.cuda.current_stream())
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        M.moe_route_noalloc(desc, x, w_router, bias, idx, gates, load,
                            torch.cuda.current_stream())
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert M.moe_last_error() == M.MOE_OK
    assert free1 == free0
    assert int(load.sum()) == T * k
