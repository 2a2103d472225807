"""FP8 (e4m3) gate/up products with per-row scales against the float64
oracle (reading 10).

Per-row quantization (moe_quantize_rows_e4m3, and the tokens inside the
forward) must give the oracle's codes and scales bit for bit: both sides take
the same fp32 division and nearest-even rounding.  The layer with
MOE_FP8_GATE_UP is compared with the oracle's fp8 reading (gate/up on per-row
dequantized operands, W_down and the routing unquantized) under the bf16
tolerances; the routing checks are those of the bf16 layer.  (The block-scaled
mode, both products in e4m3, is tested in test_gpu_fp8_block.py.)
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


def _special_rows(a):
    """Rows that exercise the rounding: zeros, a wide dynamic range (e4m3
    subnormals and underflow to zero), exact ties between codes."""
    cols = a.shape[1]
    a[0] = 0
    e = torch.arange(cols) % 48 - 40                     # 2^-40 .. 2^7
    a[1] = (torch.where(torch.arange(cols) % 2 == 0, 1.0, -1.5) * torch.pow(2.0, e.float()))
    tie = torch.tensor([448.0, 432.0, -432.0, 1.0625, 1.1875, 0.0, -3.25, 240.0, 232.0, 2.0 ** -7])
    a[2] = tie.repeat(cols // len(tie) + 1)[:cols]       # midpoints round to the even code
    return a


SHAPES = [(1, 128), (37, 7168), (300, 384), (4096, 2048)]


@pytest.mark.parametrize("rows,cols", SHAPES, ids=[f"{r}x{c}" for r, c in SHAPES])
def test_quantize_rows_bit_exact(rows, cols):
    gen = torch.Generator().manual_seed(rows + cols)
    row_scale = torch.pow(2.0, torch.randint(-20, 20, (rows, 1), generator=gen).float())
    a = torch.randn(rows, cols, generator=gen) * row_scale
    if rows >= 3:
        a = _special_rows(a)
    a = a.to(torch.bfloat16)
    packed = MoeLayer.quantize(a.cuda())
    torch.cuda.synchronize()
    codes, scales = MoeLayer.unpack(packed, rows, cols)
    q, sc, _ = O.quantize_rows_e4m3(a.float().numpy())
    assert np.array_equal(scales.cpu().numpy(), sc)
    assert np.array_equal(codes.cpu().numpy(), q)


def test_quantize_nan_row_gets_unit_scale():
    a = torch.randn(4, 256, generator=torch.Generator().manual_seed(1))
    a[2, 17] = float("nan")
    a = a.to(torch.bfloat16)
    codes, scales = MoeLayer.unpack(MoeLayer.quantize(a.cuda()), 4, 256)
    torch.cuda.synchronize()
    q, sc, _ = O.quantize_rows_e4m3(a.float().numpy())
    g = codes.cpu().numpy()
    assert np.array_equal(scales.cpu().numpy(), sc) and sc[2] == 1.0
    assert (g[2, 17] & 0x7F) == 0x7F and (q[2, 17] & 0x7F) == 0x7F  # NaN codes
    mask = np.ones_like(g, dtype=bool)
    mask[2, 17] = False
    assert np.array_equal(g[mask], q[mask])


def _fetch(inp):
    def get(e):
        return (np64(inp["w_gate"][e]), np64(inp["w_up"][e]), np64(inp["w_down"][e]))
    return get


MODES = {"gate_up": M.MOE_FP8_GATE_UP}


def _check_fp8(wl, mode, n_rows=None):
    flags = MODES[mode]
    inp = I.make_inputs(wl, device="cuda")
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, flags)
    y = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    x64, wr64, b64 = np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"])
    ref = O.route(x64, wr64, b64, wl.k)
    gidx = npi(layer.topk_idx)
    flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref, 1e-5)
    check_load(npi(layer.load_counts), gidx, ref["idx"], wl.E, flips)
    # the tokens' codes and scales in the workspace: the oracle's, bit for bit
    xq = layer.region("x_q", torch.uint8, (layer.regions["x_q"][1],))
    codes, scales = MoeLayer.unpack(xq, wl.T, wl.d)
    q, sc, _ = O.quantize_rows_e4m3(inp["x"].float().cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), q)
    assert np.array_equal(scales.cpu().numpy(), sc)
    if n_rows is None or n_rows >= wl.T:
        rows = np.arange(wl.T)
    else:
        rows = np.sort(np.random.default_rng(wl.seed).choice(wl.T, n_rows, replace=False))
    sh = (np64(inp["sh_gate"]), np64(inp["sh_up"]), np64(inp["sh_down"]))
    g_rows = O.gate_weights(ref["s"][rows], gidx[rows])
    y_ref = O.fp8_gate_up_rows(x64[rows], gidx[rows], g_rows, _fetch(inp), sh)
    stats = check_output(np64(y[torch.from_numpy(rows).cuda()]), y_ref, "bf16")
    # the quantization is visible: the unquantized layer differs by more
    y_bf = O.expert_output_rows(x64[rows], gidx[rows], g_rows, _fetch(inp), sh)
    stats["rel_l2_vs_unquantized"] = float(np.linalg.norm(y_bf - y_ref) / np.linalg.norm(y_bf))
    del layer, inp, y
    torch.cuda.empty_cache()
    return stats, flips


CASES = [(m, *c) for m in MODES for c in (
    ("small_bf16", dict(), None),
    ("v3_decode", dict(), None),
    ("v3_prefill", dict(), 48),
)] + [
    ("gate_up", "mini_bf16", dict(T=2048), None),
    ("gate_up", "v3_decode_zipf", dict(), None),
]


@pytest.mark.parametrize("mode,name,over,n_rows", CASES,
                         ids=[f"{m}-{n}_{o.get('T', 'T')}" for m, n, o, _ in CASES])
def test_fp8_layer_matches_oracle(mode, name, over, n_rows):
    stats, flips = _check_fp8(I.WORKLOADS[name].with_(**over), mode, n_rows)
    print(f"{mode} {name}: {stats} flips={flips}")
    assert stats["rel_l2_vs_unquantized"] > 2 * stats["rel_l2"]


EDGES = [
    dict(T=1, d=1024, h=256, E=16, k=4),       # one token: 16-token tiles of one row
    dict(T=300, d=1024, h=384, E=16, k=4),     # ragged token tiles, h not a multiple of 256
    dict(T=513, d=2048, h=512, E=8, k=8),      # k = E: every expert takes every token
]


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("shape", EDGES, ids=[f"T{s['T']}_h{s['h']}_E{s['E']}_k{s['k']}" for s in EDGES])
def test_fp8_edges(shape, mode):
    stats, _ = _check_fp8(I.custom(dtype="bf16", seed=7 + shape["T"], **shape), mode)
    print(mode, shape, stats)
