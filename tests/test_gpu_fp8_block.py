"""Block-scaled FP8 experts (MOE_FP8_BLOCK) against the float64 oracle's
reading 11: 128 x 128 weight blocks, 1 x 128 activation blocks, power-of-two
scales, the hidden rows quantized from their unrounded values.

* Block quantization of weights (moe_quantize_blocks_e4m3) and of the tokens
  inside the forward: codes and exponents bit for bit (both sides take the
  same exact power-of-two scaling and nearest-even rounding of an exact
  value).
* The layer: routing as the bf16 layer; outputs within the bf16 bar (rel L2
  1e-2, max |diff| 5e-2 * rms), derived for this reading before measuring:
  the GPU's fp32 H and the oracle's float64 H can round to neighbouring codes
  only where they straddle a rounding boundary.
* The hidden rows' codes written by the first GEMM: equal to the oracle's
  except for such boundary cases (a small fraction, one e4m3 step apart).
* V3 widths: the 32-expert prefill layer on 256 rows, the Zipf-skewed decode
  layer on all rows, and at the full V3 prefill size the routing on every
  token and the hidden rows and down-projection rows of four experts.
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


def _codes_equal(got, ref):
    """Codes equal bit for bit, NaN codes (0x7f / 0xff) matched as NaN."""
    gn, rn = (got & 0x7F) == 0x7F, (ref & 0x7F) == 0x7F
    assert np.array_equal(gn, rn), "NaN codes differ"
    assert np.array_equal(got[~gn], ref[~rn])


def _special(a):
    """Rows exercising the format: a block of zeros, a wide dynamic range,
    exact midpoints between codes."""
    rows, cols = a.shape
    if rows * cols > 128 * 128:
        a[:128, :128] = 0
    e = torch.arange(128) % 48 - 40
    a[1, -128:] = torch.where(torch.arange(128) % 2 == 0, 1.0, -1.5) * torch.pow(2.0, e.float())
    tie = torch.tensor([448.0, 432.0, -432.0, 1.0625, 1.1875, 0.0, -3.25, 240.0, 232.0, 2.0 ** -7])
    a[2, :] = tie.repeat(cols // len(tie) + 1)[:cols]
    return a


SHAPES = [(128, 128), (256, 384), (2048, 7168), (7168, 2048)]


@pytest.mark.parametrize("rows,cols", SHAPES, ids=[f"{r}x{c}" for r, c in SHAPES])
def test_quantize_blocks_bit_exact(rows, cols):
    gen = torch.Generator().manual_seed(rows + 3 * cols)
    blk_scale = torch.pow(2.0, torch.randint(-20, 20, (rows // 128, 1, cols // 128, 1),
                                             generator=gen).float())
    a = (torch.randn(rows // 128, 128, cols // 128, 128, generator=gen) * blk_scale)
    a = _special(a.reshape(rows, cols)).to(torch.bfloat16)
    if rows >= 256:
        a[130, 5] = float("nan")
        a[131, 260] = float("inf")
        a[132, 261] = float("-inf")
    packed = MoeLayer.quantize_blocks(a.cuda())
    torch.cuda.synchronize()
    codes, ex = MoeLayer.unpack_blocks(packed, rows, cols)
    q, e, _ = O.quantize_blocks_e4m3(a.float().numpy(), 128)
    _codes_equal(codes.cpu().numpy(), q)
    assert np.array_equal(ex.cpu().numpy().astype(np.int64) - 127, e)


def test_quantize_blocks_rejects_bad_sizes():
    a = torch.zeros((128, 100), dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    assert M.moe_quantize_blocks_e4m3(a, 128, 100, out, check=False) == M.ERR_CODE["MOE_ERR_SHAPE"]
    assert M.moe_quantize_blocks_e4m3(a, 100, 128, out, check=False) == M.ERR_CODE["MOE_ERR_SHAPE"]
    assert M.moe_e4m3_block_packed_bytes(128, 100) == 0


def _layer(wl, inp=None):
    if inp is None:
        inp = {n: (v.cuda() if isinstance(v, torch.Tensor) else v)
               for n, v in I.make_inputs(wl).items()}
    layer = MoeLayer.from_inputs(inp, wl.k, "bf16", M.MOE_FP8_BLOCK)
    y = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert M.moe_last_error() == M.MOE_OK
    return inp, layer, y


def _fetch(inp):
    return lambda e: (np64(inp["w_gate"][e]), np64(inp["w_up"][e]), np64(inp["w_down"][e]))


def _check_hidden_codes(layer, inp, wl, experts):
    """The first GEMM's H codes and exponents for the rows of `experts`
    against the oracle's H (from the block-dequantized tokens and weights)
    quantized in 1 x 128 blocks: returns the fraction of codes that differ,
    and checks that every differing code is one e4m3 step from the oracle's."""
    off, nbytes = layer.regions["h_q"]
    rows_h = wl.T * wl.k + wl.T
    hq = layer.workspace[off:off + nbytes]
    codes, ex = MoeLayer.unpack_blocks(hq, rows_h, wl.h, act_rows=True)
    g_off = layer.region("groups", torch.int32, (wl.E + 2,)).cpu().numpy()
    perm = layer.region("perm", torch.int32, (wl.T * wl.k,)).cpu().numpy()
    x64 = np64(inp["x"])
    diff = total = 0
    for e in experts:
        r0, r1 = int(g_off[e]), int(g_off[e + 1])
        if r1 == r0:
            continue
        tok = perm[r0:r1] // wl.k
        wg, wu, _ = _fetch(inp)(e)
        xq = O.quantize_blocks_e4m3(x64[tok], 1, codes=False)[2]
        hid = O.silu(xq @ O.quantize_blocks_e4m3(wg, 128, codes=False)[2].T) * (
            xq @ O.quantize_blocks_e4m3(wu, 128, codes=False)[2].T)
        qr, er, dr = O.quantize_blocks_e4m3(hid, 1)
        got_c = codes[r0:r1].cpu().numpy()
        got_e = ex[r0:r1].cpu().numpy().astype(np.int64) - 127
        # exponents: equal except where the block maximum sits on a boundary
        assert (got_e != er).mean() < 1e-3
        same_e = np.repeat(got_e == er, 128, axis=1)
        d = (got_c != qr) & same_e
        diff += int(d.sum())
        total += int(same_e.sum())
        if d.any():  # neighbouring e4m3 values: positions one apart on the grid
            gv, rv = _code_values(got_c[d]), _code_values(qr[d])
            assert np.all((np.sign(gv) == np.sign(rv)) | (gv == 0) | (rv == 0))
            assert np.all(np.abs(np.searchsorted(GRID, np.abs(gv)) -
                                 np.searchsorted(GRID, np.abs(rv))) <= 1)
    return diff / max(total, 1)


def _code_value(c):
    if c & 0x7F == 0x7F:
        return np.nan
    sgn = -1.0 if c >> 7 else 1.0
    e, m = (c >> 3) & 15, c & 7
    return sgn * (np.ldexp(1 + m / 8, e - 7) if e else np.ldexp(m / 8, -6))


CODE_VALUE = np.array([_code_value(c) for c in range(256)])
GRID = np.unique(np.abs(CODE_VALUE[np.isfinite(CODE_VALUE)]))


def _code_values(codes):
    return CODE_VALUE[np.asarray(codes, dtype=np.int64)]


LAYERS = [
    dict(T=300, d=256, h=256, E=8, k=2),
    dict(T=1000, d=512, h=384, E=16, k=4),   # h = 3 blocks: a partial word of exponents
    dict(T=64, d=256, h=128, E=40, k=2),     # many experts without tokens
    dict(T=513, d=384, h=256, E=12, k=3),    # ragged tiles
    dict(T=2048, d=256, h=256, E=4, k=2),    # five token tiles of <= 240 per expert
    dict(T=16, d=512, h=512, E=64, k=8),     # decode-like: tiles of 16 tokens
    dict(T=1, d=1024, h=256, E=16, k=4),     # one token
    dict(T=513, d=2048, h=512, E=8, k=8),    # k = E: every expert takes every token
    dict(T=700, d=640, h=640, E=6, k=2),     # d, h = 5 blocks: a partial exponent word
]


@pytest.mark.parametrize("shape", LAYERS,
                         ids=[f"T{s['T']}_d{s['d']}_h{s['h']}_E{s['E']}_k{s['k']}" for s in LAYERS])
def test_block_layer_matches_oracle(shape):
    wl = I.custom(dtype="bf16", seed=11 + shape["T"], **shape)
    inp, layer, y = _layer(wl)
    x64, wr64, b64 = np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"])
    ref = O.route(x64, wr64, b64, wl.k)
    gidx = npi(layer.topk_idx)
    flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref, 1e-5)
    check_load(npi(layer.load_counts), gidx, ref["idx"], wl.E, flips)
    sh = (np64(inp["sh_gate"]), np64(inp["sh_up"]), np64(inp["sh_down"]))
    y_ref = O.fp8_block_expert_rows(x64, gidx, O.gate_weights(ref["s"], gidx), _fetch(inp), sh,
                                    gate_up=True, down=True)
    stats = check_output(np64(y), y_ref, "bf16")
    # the tokens' codes and exponents inside the call: bit for bit
    off, nbytes = layer.regions["x_q"]
    xc, xe = MoeLayer.unpack_blocks(layer.workspace[off:off + nbytes], wl.T, wl.d, act_rows=True)
    q, e, _ = O.quantize_blocks_e4m3(x64, 1)
    _codes_equal(xc.cpu().numpy(), q)
    assert np.array_equal(xe.cpu().numpy().astype(np.int64) - 127, e)
    frac = _check_hidden_codes(layer, inp, wl, range(wl.E))
    assert frac < 1e-3, frac
    # quantization changes the layer by a few per cent, no more
    y_exact = O.expert_output_rows(x64, gidx, O.gate_weights(ref["s"], gidx), _fetch(inp), sh)
    rel_q = np.linalg.norm(np64(y) - y_exact) / np.linalg.norm(y_exact)
    assert rel_q < 0.1, rel_q
    print(f"{wl.name}: {stats} H codes differing {frac:.2e} fp8 vs exact {rel_q:.3f}")


def test_block_nan_token_is_isolated():
    wl = I.custom(T=200, d=256, h=256, E=8, k=2, dtype="bf16", seed=5)
    inp = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in I.make_inputs(wl).items()}
    inp["x"][17, 3] = float("nan")
    _, layer, y = _layer(wl, inp)
    yn = np64(y)
    assert np.isnan(yn[17]).all()
    assert np.isfinite(np.delete(yn, 17, axis=0)).all()


def test_block_layer_v3_widths_32_experts():
    """V3 expert widths (d = 7168, h = 2048), 32 experts with about 256
    tokens each: the prefill regime (two token tiles per expert), 256 rows."""
    wl = I.WORKLOADS["v3_prefill_32experts"]
    inp = I.make_inputs(wl, device="cuda")
    _, layer, y = _layer(wl, inp)
    x64, wr64, b64 = np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"])
    ref = O.route(x64, wr64, b64, wl.k)
    gidx = npi(layer.topk_idx)
    flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref, 1e-5)
    check_load(npi(layer.load_counts), gidx, ref["idx"], wl.E, flips)
    rows = np.sort(np.random.default_rng(7).choice(wl.T, 256, replace=False))
    sh = (np64(inp["sh_gate"]), np64(inp["sh_up"]), np64(inp["sh_down"]))
    y_ref = O.fp8_block_expert_rows(x64[rows], gidx[rows], O.gate_weights(ref["s"][rows], gidx[rows]),
                                    _fetch(inp), sh, gate_up=True, down=True)
    stats = check_output(np64(y[torch.from_numpy(rows).cuda()]), y_ref, "bf16")
    print(f"v3 widths, 32 experts: {stats}")
    del layer, inp, y
    torch.cuda.empty_cache()


def test_block_layer_v3_decode_zipf():
    wl = I.WORKLOADS["v3_decode_zipf"]
    inp = I.make_inputs(wl, device="cuda")
    _, layer, y = _layer(wl, inp)
    x64, wr64, b64 = np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"])
    ref = O.route(x64, wr64, b64, wl.k)
    gidx = npi(layer.topk_idx)
    flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref, 1e-5)
    assert flips == 0
    sh = (np64(inp["sh_gate"]), np64(inp["sh_up"]), np64(inp["sh_down"]))
    y_ref = O.fp8_block_expert_rows(x64, gidx, O.gate_weights(ref["s"], gidx), _fetch(inp), sh,
                                    gate_up=True, down=True)
    stats = check_output(np64(y), y_ref, "bf16")
    print(f"v3 decode zipf: {stats}")
    del layer, inp, y
    torch.cuda.empty_cache()


def test_block_layer_v3_prefill_full_size():
    """The full V3 prefill layer in block-scaled FP8, in the launch
    configuration bench.py times: routing on every token; for four experts
    (the most and least loaded among others) the hidden rows' codes and the
    ungated down-projection rows against the oracle."""
    wl = I.WORKLOADS["v3_prefill"]
    inp = I.make_inputs(wl, device="cuda")
    _, layer, y = _layer(wl, inp)
    x64, wr64, b64 = np64(inp["x"]), np64(inp["w_router"]), np64(inp["bias"])
    ref = O.route(x64, wr64, b64, wl.k)
    gidx = npi(layer.topk_idx)
    flips = check_routing(gidx, layer.gates.cpu().numpy().astype(np.float64), ref, 1e-5)
    assert flips == 0
    load = npi(layer.load_counts)
    check_load(load, gidx, ref["idx"], wl.E, flips)
    experts = [int(np.argmax(load)), int(np.argmin(load)), 7, 200]
    frac = _check_hidden_codes(layer, inp, wl, experts)
    assert frac < 1e-3, frac
    g_off = layer.region("groups", torch.int32, (wl.E + 2,)).cpu().numpy()
    perm = layer.region("perm", torch.int32, (wl.T * wl.k,)).cpu().numpy()
    yp = layer.region("y_perm", torch.bfloat16, (wl.T * wl.k, wl.d))
    for e in experts:
        r0, r1 = int(g_off[e]), int(g_off[e + 1])
        tok = perm[r0:r1] // wl.k
        ye = O.fp8_block_swiglu_expert(x64[tok], *_fetch(inp)(e), gate_up=True, down=True)
        check_output(np64(yp[r0:r1]), ye, "bf16")
    del layer, inp, y
    torch.cuda.empty_cache()
