"""Plant plausible mistakes in the oracle (on the CPU) and require that at
least one pin catches each of them.  This is what makes the pins a real
check: a pin set that passes a broken oracle would not pin anything."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from tests.oracle_pins import PINS

F64 = np.float64


def _sigmoid_flipped(u):
    return 1.0 / (1.0 + np.exp(np.asarray(u, F64)))


def _biased_minus(s, bias):
    return np.asarray(s, F64) - np.asarray(bias, F64)[None, :]


def _biased_none(s, bias):
    return np.asarray(s, F64) + 0.0 * np.asarray(bias, F64)[None, :]


def _topk_high_index_ties(z, k):
    z = np.asarray(z, F64)
    key = np.where(np.isnan(z), -np.inf, z)
    E = z.shape[1]
    order = np.argsort(-key[:, ::-1], axis=1, kind="stable")
    return (E - 1 - order[:, :k]).astype(np.int64)


def _topk_smallest(z, k):
    z = np.asarray(z, F64)
    return np.argsort(z, axis=1, kind="stable")[:, :k].astype(np.int64)


def _topk_nan_first(z, k):
    z = np.asarray(z, F64)
    key = np.where(np.isnan(z), np.inf, z)
    return np.argsort(-key, axis=1, kind="stable")[:, :k].astype(np.int64)


def _topk_unordered(z, k):
    z = np.asarray(z, F64)
    key = np.where(np.isnan(z), -np.inf, z)
    order = np.argsort(-key, axis=1, kind="stable")[:, :k]
    return np.sort(order, axis=1).astype(np.int64)


def _gates_unnormalised(s, idx):
    return np.take_along_axis(np.asarray(s, F64), idx, axis=1)


def _gates_softmax(s, idx):
    sel = np.exp(np.take_along_axis(np.asarray(s, F64), idx, axis=1))
    return sel / sel.sum(axis=1, keepdims=True)


def _route_biased_gates(x, w_router, bias, k):
    u, s = O.router_affinity(x, w_router)
    z = O.biased_scores(s, bias)
    idx = O.select_topk(z, k)
    return {"u": u, "s": s, "z": z, "idx": idx,
            "gates": O.gate_weights(z, idx), "gap": O.topk_gap(z, k)}


def _silu_wrong(z):
    z = np.asarray(z, F64)
    return z * O.sigmoid(-z)


def _swiglu_silu_on_up(x, w_gate, w_up, w_down):
    x = np.asarray(x, F64)
    return ((x @ np.asarray(w_gate, F64).T) * O.silu(x @ np.asarray(w_up, F64).T)) @ np.asarray(w_down, F64).T


def _swiglu_down_untransposed(x, w_gate, w_up, w_down):
    x = np.asarray(x, F64)
    hmid = O.silu(x @ np.asarray(w_gate, F64).T) * (x @ np.asarray(w_up, F64).T)
    return hmid @ np.asarray(w_down, F64)  # W_down used untransposed


def _swiglu_no_up(x, w_gate, w_up, w_down):
    x = np.asarray(x, F64)
    return O.silu(x @ np.asarray(w_gate, F64).T) @ np.asarray(w_down, F64).T


def _dense_no_shared(x, w_router, bias, experts, shared, k, idx_override=None):
    z = (np.zeros_like(shared[0]), shared[1], shared[2])
    return _ORIG["moe_forward_dense"](x, w_router, bias, experts, z, k, idx_override)


def _dense_mask_with_s(x, w_router, bias, experts, shared, k, idx_override=None):
    r = O.route(x, w_router, bias, k)
    idx = r["idx"]
    T, E = r["s"].shape
    mask = np.zeros((T, E))
    np.put_along_axis(mask, idx, np.take_along_axis(r["s"], idx, axis=1), axis=1)
    wg, wu, wd = experts
    y = O.swiglu_expert(x, *shared)
    for e in range(E):
        y = y + mask[:, e:e + 1] * O.swiglu_expert(x, wg[e], wu[e], wd[e])
    out = dict(r)
    out.update({"idx": idx, "gates": O.gate_weights(r["s"], idx), "y": y})
    return out


def _sparse_first_slot_only(x, w_router, bias, experts, shared, k, idx_override=None):
    r = O.route(x, w_router, bias, k)
    idx, gates = r["idx"], r["gates"]
    wg, wu, wd = experts
    y = O.swiglu_expert(x, *shared)
    for t in range(idx.shape[0]):
        e = int(idx[t, 0])
        y[t] += gates[t, 0] * O.swiglu_expert(x[t:t + 1], wg[e], wu[e], wd[e])[0]
    out = dict(r)
    out.update({"y": y})
    return out


def _rows_ungated(x_rows, idx_rows, gate_rows, get_expert, shared):
    return _ORIG["expert_output_rows"](x_rows, idx_rows, np.ones_like(gate_rows), get_expert, shared)


def _load_no_minlength(idx, n_experts):
    return np.bincount(np.asarray(idx).ravel()).astype(np.int64)


def _load_per_token(idx, n_experts):
    return np.bincount(np.asarray(idx)[:, 0], minlength=n_experts).astype(np.int64)


def _bias_sign_flipped(bias, load, gamma, tk):
    b = np.asarray(bias, np.float32).astype(F64)
    load = np.asarray(load, np.int64)
    sgn = np.sign(load.shape[0] * load - int(tk))
    return (b + F64(np.float32(gamma)) * sgn).astype(np.float32)


def _bias_floor_mean(bias, load, gamma, tk):
    b = np.asarray(bias, np.float32).astype(F64)
    load = np.asarray(load, np.int64)
    sgn = np.sign(load - int(tk) // load.shape[0])
    return (b - F64(np.float32(gamma)) * sgn).astype(np.float32)


def _bias_no_round(bias, load, gamma, tk):
    b = np.asarray(bias, np.float32).astype(F64)
    load = np.asarray(load, np.int64)
    sgn = np.sign(load.shape[0] * load - int(tk))
    return b - gamma * sgn


def _gap_off_by_one(z, k):
    z = np.asarray(z, F64)
    srt = -np.sort(-z, axis=1)
    return srt[:, k - 2] - srt[:, k - 1] if k >= 2 else srt[:, 0] - srt[:, 1]


def _router_no_sigmoid(x, w_router):
    u = np.asarray(x, F64) @ np.asarray(w_router, F64).T
    return u, u


def _balance_unnormalised(s, idx, seq_len, alpha=1e-4):
    s = np.asarray(s, F64)
    idx = np.asarray(idx)
    T, E = s.shape
    k = idx.shape[1]
    out = []
    for t0 in range(0, T, seq_len):
        S = min(T, t0 + seq_len) - t0
        f = E / (k * S) * np.bincount(idx[t0:t0 + S].ravel(), minlength=E)
        out.append(alpha * float((f * s[t0:t0 + S].sum(0) / S).sum()))  # s, not s / sum_j s
    return np.array(out)


def _balance_whole_batch(s, idx, seq_len, alpha=1e-4):
    return _ORIG["sequence_balance_loss"](s, idx, np.asarray(s).shape[0], alpha)


def _balance_first_slot(s, idx, seq_len, alpha=1e-4):
    idx = np.asarray(idx)
    # counts only the first slot of every token (k kept in E/(k S))
    return _ORIG["sequence_balance_loss"](s, idx[:, :1], seq_len, alpha) / idx.shape[1]


def _balance_no_e_factor(s, idx, seq_len, alpha=1e-4):
    return _ORIG["sequence_balance_loss"](s, idx, seq_len, alpha) / np.asarray(s).shape[1]


def _bwd_expert_silu_prime(x, w_gate, w_up, w_down, dy):
    x, dy = np.asarray(x, F64), np.asarray(dy, F64)
    wg, wu, wd = (np.asarray(w, F64) for w in (w_gate, w_up, w_down))
    a, c = x @ wg.T, x @ wu.T
    sg = O.sigmoid(a)
    dh = dy @ wd
    da = dh * c * sg  # drops the a (1 - sigmoid(a)) term of silu'
    dc = dh * (a * sg)
    return da @ wg + dc @ wu, da.T @ x, dc.T @ x, dy.T @ (a * sg * c)


def _bwd_expert_down_without_silu(x, w_gate, w_up, w_down, dy):
    dx, dg, du, _ = _ORIG["swiglu_expert_backward"](x, w_gate, w_up, w_down, dy)
    x = np.asarray(x, F64)
    a, c = x @ np.asarray(w_gate, F64).T, x @ np.asarray(w_up, F64).T
    return dx, dg, du, np.asarray(dy, F64).T @ (a * c)  # a * c instead of silu(a) * c


def _bwd_no_shared_dx(x, w_router, bias, experts, shared, k, dy, idx_override=None):
    out = _ORIG["moe_backward_dense"](x, w_router, bias, experts, shared, k, dy, idx_override)
    out["dx"] = out["dx"] - _ORIG["swiglu_expert_backward"](x, *shared, dy)[0]
    return out


def _bwd_gate_no_quotient(x, w_router, bias, experts, shared, k, dy, idx_override=None):
    out = _ORIG["moe_backward_dense"](x, w_router, bias, experts, shared, k, dy, idx_override)
    r = O.route(x, w_router, bias, k)
    s, idx = r["s"], out["idx"]
    x64 = np.asarray(x, F64)
    ds = np.zeros_like(s)
    dg_sel = np.take_along_axis(out["dG"], idx, axis=1)
    np.put_along_axis(ds, idx, dg_sel / np.take_along_axis(s, idx, axis=1).sum(1, keepdims=True), axis=1)
    du = ds * s * (1 - s)
    out["dx"] = out["dx"] - out["du"] @ np.asarray(w_router, F64) + du @ np.asarray(w_router, F64)
    out["dW_router"], out["du"] = du.T @ x64, du
    return out


def _bwd_router_no_sigmoid_grad(x, w_router, bias, experts, shared, k, dy, idx_override=None):
    out = _ORIG["moe_backward_dense"](x, w_router, bias, experts, shared, k, dy, idx_override)
    s = O.route(x, w_router, bias, k)["s"]
    du = out["du"] / (s * (1 - s))  # ds in place of du
    x64 = np.asarray(x, F64)
    out["dx"] = out["dx"] - out["du"] @ np.asarray(w_router, F64) + du @ np.asarray(w_router, F64)
    out["dW_router"], out["du"] = du.T @ x64, du
    return out


def _quant_wrong_max(a):
    import torch
    t = torch.as_tensor(np.asarray(a, dtype=np.float32))
    amax = t.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / 240.0, torch.ones_like(amax))  # 240: not e4m3's max
    q = (t / scale).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), scale.squeeze(-1).numpy(), (q.double() * scale.double()).numpy()


def _quant_per_column(a):
    q, s, d = _ORIG["quantize_rows_e4m3"](np.asarray(a, dtype=np.float32).T)
    return q.T, s, d.T


def _quant_truncate(a):
    import torch
    t = torch.as_tensor(np.asarray(a, dtype=np.float32))
    amax = t.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    r = (t / scale).double()
    # round toward zero to 3 mantissa bits instead of to nearest
    e = torch.floor(torch.log2(r.abs().clamp_min(2.0 ** -9))).clamp_min(-6)
    step = torch.pow(2.0, e - 3)
    tr = (torch.trunc(r / step) * step).float()
    q = tr.to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), scale.squeeze(-1).numpy(), (q.double() * scale.double()).numpy()


def _fp8_unquantized_tokens(x_rows, idx_rows, gate_rows, get_expert, shared):
    def q(w):
        return (_ORIG["quantize_rows_e4m3"](w[0])[2], _ORIG["quantize_rows_e4m3"](w[1])[2],
                np.asarray(w[2], F64))
    return _ORIG["expert_output_rows"](x_rows, idx_rows, gate_rows, lambda e: q(get_expert(e)),
                                       q(shared))


def _fp8_down_quantized(x_rows, idx_rows, gate_rows, get_expert, shared):
    xq = _ORIG["quantize_rows_e4m3"](x_rows)[2]

    def q(w):
        return tuple(_ORIG["quantize_rows_e4m3"](m)[2] for m in w)
    return _ORIG["expert_output_rows"](xq, idx_rows, gate_rows, lambda e: q(get_expert(e)),
                                       q(shared))


def _fp8_codes_only(x_rows, idx_rows, gate_rows, get_expert, shared):
    # drops the scales: codes taken as values
    def codes(a):
        return _ORIG["quantize_rows_e4m3"](a)[0].view(np.int8).astype(F64)
    xq = codes(x_rows)

    def q(w):
        return codes(w[0]), codes(w[1]), np.asarray(w[2], F64)
    return _ORIG["expert_output_rows"](xq, idx_rows, gate_rows, lambda e: q(get_expert(e)),
                                       q(shared))














def _e4m3_round_half_away(v):
    v = np.asarray(v, dtype=F64)
    out = np.full(v.shape, np.nan)
    fin = ~np.isnan(v)
    a = np.minimum(np.abs(v[fin]), 448.0)
    _, ex = np.frexp(a)
    k = np.maximum(ex - 1, -6) - 3
    q = np.floor(np.ldexp(a, -k) + 0.5)  # halves away from zero
    out[fin] = np.copysign(np.minimum(np.ldexp(q, k), 448.0), v[fin])
    return out


def _e4m3_round_truncate(v):
    v = np.asarray(v, dtype=F64)
    out = np.full(v.shape, np.nan)
    fin = ~np.isnan(v)
    a = np.minimum(np.abs(v[fin]), 448.0)
    _, ex = np.frexp(a)
    k = np.maximum(ex - 1, -6) - 3
    out[fin] = np.copysign(np.ldexp(np.floor(np.ldexp(a, -k)), k), v[fin])
    return out


def _e4m3_round_two_bits(v):
    v = np.asarray(v, dtype=F64)
    out = np.full(v.shape, np.nan)
    fin = ~np.isnan(v)
    a = np.minimum(np.abs(v[fin]), 448.0)
    _, ex = np.frexp(a)
    k = np.maximum(ex - 1, -6) - 2  # a 2-bit mantissa
    out[fin] = np.copysign(np.ldexp(np.rint(np.ldexp(a, -k)), k), v[fin])
    return out


def _blockexp_floor(amax):
    e = _ORIG["block_exponent"](amax)
    return np.where(np.asarray(amax) > 0, e - 1, e)


def _blockexp_wrong_max(amax):
    amax = np.asarray(amax, dtype=F64)
    return _ORIG["block_exponent"](amax * (448.0 / 240.0))


def _blockexp_unclamped_nan(amax):
    amax = np.asarray(amax, dtype=F64)
    e = np.zeros(amax.shape, dtype=np.int64)
    ok = amax > 0
    e[ok] = np.ceil(np.log2(amax[ok] / 448.0)).astype(np.int64)
    return e


def _qblocks_64_wide(a, block_rows):
    a = np.asarray(a, dtype=F64)
    R, C = a.shape
    parts = [_ORIG["quantize_blocks_e4m3"](np.repeat(a[:, j:j + 64], 2, axis=1)[:, :128],
                                           block_rows) for j in range(0, C, 64)]
    codes = np.concatenate([p[0][:, :64] for p in parts], axis=1)
    deq = np.concatenate([p[2][:, :64] for p in parts], axis=1)
    e = _ORIG["quantize_blocks_e4m3"](a, block_rows)[1]
    return codes, e, deq


def _qblocks_rows_only(a, block_rows):
    return _ORIG["quantize_blocks_e4m3"](a, 1)


def _qblocks_whole_row(a, block_rows):
    a = np.asarray(a, dtype=F64)
    R, C = a.shape
    amax = np.abs(a.reshape(R // block_rows, block_rows * C)).max(axis=1)
    e = _ORIG["block_exponent"](amax)
    sc = np.repeat(np.ldexp(1.0, e), block_rows)[:, None]
    dq = _ORIG["e4m3_round"](a / sc)
    return _ORIG["e4m3_code"](dq), np.repeat(e[:, None], C // 128, axis=1), dq * sc


def _fp8_block_h_rounded_bf16(x, w_gate, w_up, w_down, gate_up, down):
    q = _ORIG["quantize_blocks_e4m3"]
    x = np.asarray(x, dtype=F64)
    if gate_up:
        xq = q(x, 1)[2]
        g, u = xq @ q(w_gate, 128)[2].T, xq @ q(w_up, 128)[2].T
    else:
        g, u = x @ np.asarray(w_gate, F64).T, x @ np.asarray(w_up, F64).T
    import torch
    hid = torch.as_tensor(_ORIG["silu"](g) * u).to(torch.bfloat16).to(torch.float64).numpy()
    if down:
        return q(hid, 1)[2] @ q(w_down, 128)[2].T
    return hid @ np.asarray(w_down, F64).T


def _fp8_block_down_ignored(x, w_gate, w_up, w_down, gate_up, down):
    return _ORIG["fp8_block_swiglu_expert"](x, w_gate, w_up, w_down, gate_up, False)


def _fp8_block_weights_unquantized(x, w_gate, w_up, w_down, gate_up, down):
    q = _ORIG["quantize_blocks_e4m3"]
    x = np.asarray(x, dtype=F64)
    xq = q(x, 1)[2] if gate_up else x
    hid = _ORIG["silu"](xq @ np.asarray(w_gate, F64).T) * (xq @ np.asarray(w_up, F64).T)
    return (q(hid, 1)[2] if down else hid) @ np.asarray(w_down, F64).T


def _fp8_block_rows_ungated(x_rows, idx_rows, gate_rows, get_expert, shared, gate_up, down):
    return _ORIG["fp8_block_expert_rows"](x_rows, idx_rows, np.ones_like(gate_rows), get_expert,
                                          shared, gate_up, down)


def _fp8_block_rows_no_shared(x_rows, idx_rows, gate_rows, get_expert, shared, gate_up, down):
    z = tuple(np.zeros_like(np.asarray(w, F64)) for w in shared)
    return _ORIG["fp8_block_expert_rows"](x_rows, idx_rows, gate_rows, get_expert, z, gate_up,
                                          down)


_ORIG = {name: getattr(O, name) for name in dir(O) if not name.startswith("_")}

MUTATIONS = [
    ("sigmoid", _sigmoid_flipped),
    ("biased_scores", _biased_minus),
    ("biased_scores", _biased_none),
    ("select_topk", _topk_high_index_ties),
    ("select_topk", _topk_smallest),
    ("select_topk", _topk_nan_first),
    ("select_topk", _topk_unordered),
    ("gate_weights", _gates_unnormalised),
    ("gate_weights", _gates_softmax),
    ("route", _route_biased_gates),
    ("silu", _silu_wrong),
    ("swiglu_expert", _swiglu_silu_on_up),
    ("swiglu_expert", _swiglu_down_untransposed),
    ("swiglu_expert", _swiglu_no_up),
    ("moe_forward_dense", _dense_no_shared),
    ("moe_forward_dense", _dense_mask_with_s),
    ("moe_forward_sparse", _sparse_first_slot_only),
    ("expert_output_rows", _rows_ungated),
    ("load_counts", _load_no_minlength),
    ("load_counts", _load_per_token),
    ("bias_update", _bias_sign_flipped),
    ("bias_update", _bias_floor_mean),
    ("bias_update", _bias_no_round),
    ("topk_gap", _gap_off_by_one),
    ("router_affinity", _router_no_sigmoid),
    ("sequence_balance_loss", _balance_unnormalised),
    ("sequence_balance_loss", _balance_whole_batch),
    ("sequence_balance_loss", _balance_first_slot),
    ("sequence_balance_loss", _balance_no_e_factor),
    ("swiglu_expert_backward", _bwd_expert_silu_prime),
    ("swiglu_expert_backward", _bwd_expert_down_without_silu),
    ("moe_backward_dense", _bwd_no_shared_dx),
    ("moe_backward_dense", _bwd_gate_no_quotient),
    ("moe_backward_dense", _bwd_router_no_sigmoid_grad),
    ("quantize_rows_e4m3", _quant_wrong_max),
    ("quantize_rows_e4m3", _quant_per_column),
    ("quantize_rows_e4m3", _quant_truncate),
    ("fp8_gate_up_rows", _fp8_unquantized_tokens),
    ("fp8_gate_up_rows", _fp8_down_quantized),
    ("fp8_gate_up_rows", _fp8_codes_only),
    ("e4m3_round", _e4m3_round_half_away),
    ("e4m3_round", _e4m3_round_truncate),
    ("e4m3_round", _e4m3_round_two_bits),
    ("block_exponent", _blockexp_floor),
    ("block_exponent", _blockexp_wrong_max),
    ("block_exponent", _blockexp_unclamped_nan),
    ("quantize_blocks_e4m3", _qblocks_64_wide),
    ("quantize_blocks_e4m3", _qblocks_rows_only),
    ("quantize_blocks_e4m3", _qblocks_whole_row),
    ("fp8_block_swiglu_expert", _fp8_block_h_rounded_bf16),
    ("fp8_block_swiglu_expert", _fp8_block_down_ignored),
    ("fp8_block_swiglu_expert", _fp8_block_weights_unquantized),
    ("fp8_block_expert_rows", _fp8_block_rows_ungated),
    ("fp8_block_expert_rows", _fp8_block_rows_no_shared),
]


@pytest.mark.parametrize("target,mutant", MUTATIONS,
                         ids=[f"{t}:{m.__name__}" for t, m in MUTATIONS])
def test_mutation_is_caught(monkeypatch, target, mutant):
    monkeypatch.setattr(O, target, mutant)
    caught = []
    for pin in PINS:
        try:
            pin(O)
        except Exception as exc:  # noqa: BLE001 - any failure counts as caught
            caught.append((pin.__name__, type(exc).__name__))
    assert caught, f"no pin caught the planted mistake in {target}"
