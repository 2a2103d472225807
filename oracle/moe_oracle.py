"""Float64 CPU oracle for the DeepSeekMoE layer forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The product path (the
CUDA library and its Python binding) never calls it, and it shares no code with
that path: no kernels, helpers, tables or constants.

What it computes, and where the pages say so
--------------------------------------------
Sources are the five pages about the deepseek-v3-jax project:

* "190行JAX复刻DeepSeek V3" (openai-hub.com), section "190行代码到底装进了什么":
  the DeepSeekMoE layer has 16 routed experts, each token picks 4, plus one
  always-on shared expert; the project runs *every* routed expert on *every*
  token and zeroes the experts that were not selected.
* Same page, section "最有价值的实验:无辅助损失均衡真的有效": after each training
  step an over-loaded expert's routing bias goes down and an idle one's goes
  up, with update speed gamma = 1e-3; the bias only changes *which* experts
  are selected, never the gate value of a selected expert.
* "DeepSeek V3 viết lại bằng 190 dòng JAX thuần" (lehuy.net), sections
  "Những gì có trong 190 dòng code" (bias pushes routing towards idle experts
  and changes which expert is chosen, not the expert weights) and
  "Những gì đã được đơn giản hóa" (dense MoE: every expert on every token,
  unselected ones zeroed; no sparse dispatch).

The pages print no formulas.  The readings below are the plain ones the text
supports (the DeepSeek-V3 technical report, which the pages summarise and list
as a source, uses the same):

1. affinity    s[t,e] = sigmoid(u[t,e]),  u = x @ W_r.T,  sigmoid(u) = 1/(1+exp(-u))
2. selection   the k experts with the largest biased score z = s + b; ties go to
               the lower expert index; slots ordered by descending z.  A NaN
               score ranks below every number.
3. gates       g[t,j] = s[t, idx[t,j]] / sum_j' s[t, idx[t,j']]   (unbiased s)
4. experts     SwiGLU:  E(x) = W_down (silu(W_gate x) * (W_up x)),
               silu(z) = z * sigmoid(z)
5. output      y[t] = shared(x[t]) + sum_j g[t,j] * E_{idx[t,j]}(x[t])
6. load        load[e] = #{(t,j) : idx[t,j] = e}
7. bias        b_e <- fp32(b_e - fp32(gamma) * sgn(load_e - mean_load)),
               mean_load = T*k/E, sgn(0) = 0, so that sgn(E*load_e - T*k) is an
               exact integer comparison.

8. sequence-wise balance loss (the pages keep the original report's small
               auxiliary loss with alpha = 1e-4 beside the bias; "DeepSeek V3
               viết lại bằng 190 dòng JAX thuần", section "Những gì có trong 190
               dòng code"; "190行JAX复刻DeepSeek V3", section "最有价值的实验"),
               per sequence of S consecutive tokens, as the report states it:
                 f_i  = E / (k S) * #{t in the sequence : i selected for t}
                 s'   = s[t,i] / sum_j s[t,j]        (unbiased affinities)
                 P_i  = (1/S) sum_t s'[t,i]
                 L    = alpha * sum_i f_i P_i
               "selected" is the layer's own selection (biased top-k); a last
               sequence shorter than S uses its own length.

9. backward    (the pages train with this layer: "DeepSeek V3 viết lại bằng 190
               dòng JAX thuần", section "Những gì có trong 190 dòng code")
               gradients of y for an output gradient dy by the chain rule;
               the selection is piecewise constant and carries no gradient,
               the gates g = s_sel / sum s_sel carry it to the selected
               affinities, through the sigmoid to W_r and x; the bias has no
               gradient (it moves by the sign rule).

10. fp8 gate/up (the official V3 trains its experts in FP8, which the
               re-creation leaves out: "190行JAX复刻DeepSeek V3", introduction;
               a B300-native option here, not on the pages): each row of
               W_gate, W_up and of the token matrix is quantized to e4m3 with
               one fp32 scale, scale = amax|row| / 448 (1 for a zero row or
               a row holding a NaN),
               code = e4m3(row / scale) rounded to nearest even; the layer is
               then the same layer on the dequantized values code * scale
               (routing on the unquantized tokens; W_down unquantized).

11. fp8 block-scaled experts (the official model's tile granularity; a
               B300-native option, not on the pages): every expert weight
               matrix is cut into 128 x 128 blocks (128 output rows x 128
               inputs) and every activation row into 1 x 128 blocks (the
               tokens for gate/up; for the down projection the hidden row H
               of each (token, expert) pair and of the shared expert).  A
               block with largest magnitude amax gets the scale 2^e, e the
               smallest integer with amax <= 448 * 2^e (e = 0 for a block of
               zeros or one whose maximum is not finite; e clamped to
               [-127, 127]); code = e4m3(v / 2^e), nearest, ties to even
               (NaN stays NaN, +-inf becomes +-448).  The named products run
               on the dequantized values code * 2^e.  H is quantized from its
               unrounded value (nothing rounds it to bf16 first).

``moe_forward_dense`` is the pages' own formulation (every expert on every
token, then masked).  ``moe_forward_sparse`` evaluates only the selected
experts; tests pin it to the dense formulation on small inputs, and it is the
form used for sampled rows of the large workloads.

Pinning: tests/test_oracle_pins.py (brute-force top-k over all subsets,
hand-derived closed forms in tests/golden/, bias invariance, textbook
reductions of the SwiGLU expert, permutation equivariance, dense/sparse
agreement) and tests/test_oracle_mutations.py (planted mistakes must fail a
pin).  Everything is float64 on the exact (bf16-rounded where the workload
stores bf16) input values; nothing is rounded except the fp32 bias result.
"""

from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------------
# 1. router affinity
# --------------------------------------------------------------------------
def sigmoid(u: np.ndarray) -> np.ndarray:
    """Logistic function 1/(1+exp(-u)) in float64 (reading 1 above)."""
    u = _f64(u)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-u))


def router_affinity(x, w_router) -> tuple[np.ndarray, np.ndarray]:
    """u = x W_r^T and s = sigmoid(u).

    x: [T, d], w_router: [E, d].  Returns (u, s), both [T, E] float64.
    Follows "190行JAX复刻DeepSeek V3", section "190行代码到底装进了什么"
    (a per-token, per-expert routing score) with the sigmoid reading.
    """
    u = _f64(x) @ _f64(w_router).T
    return u, sigmoid(u)


# --------------------------------------------------------------------------
# 2. biased top-k selection
# --------------------------------------------------------------------------
def biased_scores(s, bias) -> np.ndarray:
    """z = s + b (the bias enters selection only; section
    "最有价值的实验:无辅助损失均衡真的有效")."""
    return _f64(s) + _f64(bias)[None, :]


def select_topk(z: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest biased scores per row, ordered by (z desc,
    expert index asc).  NaN ranks below every number (treated as -inf).

    A stable sort on -z keeps equal keys in ascending index order, which is
    exactly the "ties go to the lower index" rule.
    """
    z = _f64(z)
    key = np.where(np.isnan(z), -np.inf, z)
    order = np.argsort(-key, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def topk_gap(z: np.ndarray, k: int) -> np.ndarray:
    """Per-row gap between the k-th and (k+1)-th largest biased score
    (float64).  A GPU selection may differ from the oracle's only where this
    gap is below the tie tolerance.  For k == E the gap is +inf."""
    z = _f64(z)
    key = np.where(np.isnan(z), -np.inf, z)
    srt = -np.sort(-key, axis=1)
    if k >= z.shape[1]:
        return np.full(z.shape[0], np.inf)
    return srt[:, k - 1] - srt[:, k]


# --------------------------------------------------------------------------
# 3. gates
# --------------------------------------------------------------------------
def gate_weights(s: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """g[t,j] = s[t, idx[t,j]] / sum_j' s[t, idx[t,j']]  (unbiased s)."""
    sel = np.take_along_axis(_f64(s), idx, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def route(x, w_router, bias, k: int) -> dict:
    """Router steps 1-3 for every token: u, s, z, idx, gates, gap."""
    u, s = router_affinity(x, w_router)
    z = biased_scores(s, bias)
    idx = select_topk(z, k)
    return {"u": u, "s": s, "z": z, "idx": idx,
            "gates": gate_weights(s, idx), "gap": topk_gap(z, k)}


# --------------------------------------------------------------------------
# 4. SwiGLU expert
# --------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z)."""
    z = _f64(z)
    return z * sigmoid(z)


def swiglu_expert(x, w_gate, w_up, w_down) -> np.ndarray:
    """E(x) = W_down (silu(W_gate x) * (W_up x)) applied to each row of x.

    x: [n, d]; w_gate, w_up: [h, d]; w_down: [d, h].  Returns [n, d].
    """
    x = _f64(x)
    a = x @ _f64(w_gate).T
    c = x @ _f64(w_up).T
    return (silu(a) * c) @ _f64(w_down).T


# --------------------------------------------------------------------------
# 5. layer output
# --------------------------------------------------------------------------
def moe_forward_dense(x, w_router, bias, experts, shared, k: int,
                      idx_override=None) -> dict:
    """The pages' formulation: every routed expert on every token, the
    unselected ones masked to zero, plus the shared expert.

    experts: (W_gate [E,h,d], W_up [E,h,d], W_down [E,d,h]);
    shared:  (W_gate [h,d],   W_up [h,d],   W_down [d,h]).
    idx_override (optional [T,k]) replaces the selection, e.g. to evaluate
    the output for a tolerated near-tie flip; gates follow from it.
    """
    r = route(x, w_router, bias, k)
    idx = r["idx"] if idx_override is None else np.asarray(idx_override)
    gates = gate_weights(r["s"], idx)
    T, E = r["s"].shape
    mask = np.zeros((T, E), dtype=F64)
    np.put_along_axis(mask, idx, gates, axis=1)
    wg, wu, wd = experts
    y = swiglu_expert(x, *shared)
    for e in range(E):
        y = y + mask[:, e:e + 1] * swiglu_expert(x, wg[e], wu[e], wd[e])
    out = dict(r)
    out.update({"idx": idx, "gates": gates, "y": y})
    return out


def moe_forward_sparse(x, w_router, bias, experts, shared, k: int,
                       idx_override=None) -> dict:
    """Same output as ``moe_forward_dense`` evaluating only the selected
    experts of each token (what a truly sparse layer computes)."""
    r = route(x, w_router, bias, k)
    idx = r["idx"] if idx_override is None else np.asarray(idx_override)
    gates = gate_weights(r["s"], idx)
    wg, wu, wd = experts
    y = swiglu_expert(x, *shared)
    for t in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            e = int(idx[t, j])
            y[t] += gates[t, j] * swiglu_expert(x[t:t + 1], wg[e], wu[e], wd[e])[0]
    out = dict(r)
    out.update({"idx": idx, "gates": gates, "y": y})
    return out


def expert_output_rows(x_rows, idx_rows, gate_rows, get_expert, shared):
    """Sparse output for a sample of rows, streaming one expert at a time.

    x_rows [n,d]; idx_rows [n,k]; gate_rows [n,k] (float64);
    get_expert(e) -> (W_gate [h,d], W_up [h,d], W_down [d,h]) as arrays.
    Used for the large workloads, whose weights do not fit a float64 copy in
    host memory: only the experts that the sampled rows selected are fetched.
    """
    x_rows = _f64(x_rows)
    y = swiglu_expert(x_rows, *shared)
    idx_rows = np.asarray(idx_rows)
    for e in np.unique(idx_rows):
        w = get_expert(int(e))
        tt, jj = np.nonzero(idx_rows == e)
        ye = swiglu_expert(x_rows[tt], *w)
        for n in range(len(tt)):
            y[tt[n]] += gate_rows[tt[n], jj[n]] * ye[n]
    return y


# --------------------------------------------------------------------------
# 6, 7. load counts and bias update
# --------------------------------------------------------------------------
def load_counts(idx: np.ndarray, n_experts: int) -> np.ndarray:
    """load[e] = number of (token, slot) pairs routed to expert e."""
    return np.bincount(np.asarray(idx).ravel(), minlength=n_experts).astype(np.int64)


def bias_update(bias, load, gamma: float, tk: int) -> np.ndarray:
    """b_e <- fp32(b_e - fp32(gamma) * sgn(load_e - TK/E)), sgn(0) = 0.

    sgn(load_e - TK/E) == sgn(E*load_e - TK) is taken on integers.  The
    subtraction is done in float64 on the float32 operands (exact, since both
    are float32 values whose exponents differ by far less than 29) and then
    rounded once to float32, which equals the IEEE float32 subtraction.
    """
    bias32 = np.asarray(bias, dtype=np.float32)
    load = np.asarray(load, dtype=np.int64)
    n_experts = load.shape[0]
    sgn = np.sign(n_experts * load - int(tk)).astype(F64)
    g32 = F64(np.float32(gamma))
    return (bias32.astype(F64) - g32 * sgn).astype(np.float32)


def route_and_update(x, w_router, bias, k: int, gamma: float) -> dict:
    """One route-only step: routing, load counts, updated bias."""
    r = route(x, w_router, bias, k)
    E = r["s"].shape[1]
    load = load_counts(r["idx"], E)
    r["load"] = load
    r["bias_new"] = bias_update(bias, load, gamma, r["idx"].size)
    return r


def sequence_balance_loss(s, idx, seq_len: int, alpha: float = 1e-4) -> np.ndarray:
    """Sequence-wise balance loss (reading 8 above), one value per sequence
    of ``seq_len`` consecutive tokens.  ``s`` [T, E] are the unbiased
    affinities, ``idx`` [T, k] the selected experts."""
    s = _f64(s)
    idx = np.asarray(idx)
    T, E = s.shape
    k = idx.shape[1]
    out = []
    for t0 in range(0, T, seq_len):
        t1 = min(T, t0 + seq_len)
        S = t1 - t0
        count = np.bincount(idx[t0:t1].ravel(), minlength=E).astype(F64)
        f = E / (k * S) * count
        s_norm = s[t0:t1] / s[t0:t1].sum(axis=1, keepdims=True)
        P = s_norm.sum(axis=0) / S
        out.append(alpha * float((f * P).sum()))
    return np.array(out, dtype=F64)


# --------------------------------------------------------------------------
# 9. backward of the layer
# --------------------------------------------------------------------------
def swiglu_expert_backward(x, w_gate, w_up, w_down, dy):
    """Gradients of E(x) = W_down (silu(W_gate x) * (W_up x)) for the output
    gradient dy [n, d]: (dx [n,d], dW_gate [h,d], dW_up [h,d], dW_down [d,h]).
    silu'(a) = sigmoid(a) (1 + a (1 - sigmoid(a)))."""
    x, dy = _f64(x), _f64(dy)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    a = x @ wg.T
    c = x @ wu.T
    sg = sigmoid(a)
    hmid = a * sg * c
    dw_down = dy.T @ hmid
    dh = dy @ wd
    da = dh * c * (sg * (1.0 + a * (1.0 - sg)))
    dc = dh * (a * sg)
    return da @ wg + dc @ wu, da.T @ x, dc.T @ x, dw_down


def moe_backward_dense(x, w_router, bias, experts, shared, k: int, dy,
                       idx_override=None) -> dict:
    """Gradients of ``moe_forward_dense``'s y for the output gradient dy
    [T, d] (reading 9): dx, dW_gate/dW_up [E,h,d], dW_down [E,d,h], the
    shared expert's three, and dW_router [E,d].  Also returns dG [T,E]
    (gradient of each gate, the dot of dy with the expert's output) and
    the forward's idx and gates."""
    fwd = moe_forward_dense(x, w_router, bias, experts, shared, k, idx_override)
    x, dy = _f64(x), _f64(dy)
    s, idx, gates = fwd["s"], fwd["idx"], fwd["gates"]
    T, E = s.shape
    wg, wu, wd = experts
    out = {"idx": idx, "gates": gates}
    dx, out["dsh_gate"], out["dsh_up"], out["dsh_down"] = swiglu_expert_backward(x, *shared, dy)
    mask = np.zeros((T, E), dtype=F64)
    np.put_along_axis(mask, idx, gates, axis=1)
    dG = np.zeros((T, E), dtype=F64)
    dwg = np.zeros(np.shape(wg), dtype=F64)
    dwu = np.zeros(np.shape(wu), dtype=F64)
    dwd = np.zeros(np.shape(wd), dtype=F64)
    for e in range(E):
        dG[:, e] = (dy * swiglu_expert(x, wg[e], wu[e], wd[e])).sum(axis=1)
        dxe, dwg[e], dwu[e], dwd[e] = swiglu_expert_backward(x, wg[e], wu[e], wd[e],
                                                             mask[:, e:e + 1] * dy)
        dx = dx + dxe
    # g_j = s_j / S over the selected experts: dL/ds_i = (dg_i - sum_j dg_j g_j) / S
    dg_sel = np.take_along_axis(dG, idx, axis=1)
    s_sel = np.take_along_axis(s, idx, axis=1)
    ds_sel = (dg_sel - (dg_sel * gates).sum(axis=1, keepdims=True)) / s_sel.sum(axis=1, keepdims=True)
    ds = np.zeros((T, E), dtype=F64)
    np.put_along_axis(ds, idx, ds_sel, axis=1)
    du = ds * s * (1.0 - s)
    out["dW_router"] = du.T @ x
    out["dx"] = dx + du @ _f64(w_router)
    out.update({"dW_gate": dwg, "dW_up": dwu, "dW_down": dwd, "dG": dG, "du": du})
    return out


def backward_token_rows(x_rows, w_router, bias, get_expert, shared, k: int, dy_rows,
                        idx_override=None) -> np.ndarray:
    """dx of a sample of tokens: reading 9 restricted to their rows (a token's
    dx depends only on its own routing and experts), streaming the experts
    they selected one at a time (get_expert(e) -> (W_gate, W_up, W_down)),
    for workloads whose weights do not fit a float64 copy."""
    x_rows, dy_rows = _f64(x_rows), _f64(dy_rows)
    r = route(x_rows, w_router, bias, k)
    idx = r["idx"] if idx_override is None else np.asarray(idx_override)
    s = r["s"]
    gates = gate_weights(s, idx)
    dx = swiglu_expert_backward(x_rows, *shared, dy_rows)[0]
    dg_sel = np.zeros(idx.shape, dtype=F64)
    for e in np.unique(idx):
        w = get_expert(int(e))
        tt, jj = np.nonzero(idx == e)
        dg_sel[tt, jj] = (dy_rows[tt] * swiglu_expert(x_rows[tt], *w)).sum(axis=1)
        dxe = swiglu_expert_backward(x_rows[tt], *w, gates[tt, jj][:, None] * dy_rows[tt])[0]
        np.add.at(dx, tt, dxe)
    s_sel = np.take_along_axis(s, idx, axis=1)
    ds_sel = (dg_sel - (dg_sel * gates).sum(axis=1, keepdims=True)) / s_sel.sum(axis=1, keepdims=True)
    du_sel = ds_sel * s_sel * (1.0 - s_sel)
    wr = _f64(w_router)
    for j in range(idx.shape[1]):
        dx += du_sel[:, j:j + 1] * wr[idx[:, j]]
    return dx


# --------------------------------------------------------------------------
# 10. fp8 (e4m3) per-row quantization
# --------------------------------------------------------------------------
def quantize_rows_e4m3(a):
    """Per-row e4m3 quantization (reading 10): returns (codes uint8 [..., n],
    scales fp32 [...], dequantized float64 [..., n]).  The rounding is
    PyTorch's float8_e4m3fn conversion (nearest, ties to even); the scale
    and the division are fp32 operations."""
    import torch
    t = torch.as_tensor(np.asarray(a, dtype=np.float32))
    amax = t.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (t / scale).to(torch.float8_e4m3fn)
    deq = q.to(torch.float64) * scale.to(torch.float64)
    return q.view(torch.uint8).numpy(), scale.squeeze(-1).numpy(), deq.numpy()


def fp8_gate_up_rows(x_rows, idx_rows, gate_rows, get_expert, shared):
    """Layer output for sampled rows with the gate/up products in e4m3
    (reading 10): the tokens and every row of W_gate and W_up replaced by
    their per-row dequantized values; W_down, the selection and the gates as
    in the unquantized layer (routing is done beforehand on the unquantized
    tokens and passed in).  Same arguments as expert_output_rows."""
    xq = quantize_rows_e4m3(x_rows)[2]

    def quantized(w):
        return quantize_rows_e4m3(w[0])[2], quantize_rows_e4m3(w[1])[2], _f64(w[2])

    return expert_output_rows(xq, idx_rows, gate_rows, lambda e: quantized(get_expert(e)),
                              quantized(shared))



# --------------------------------------------------------------------------
# 11. fp8 (e4m3) block-scaled quantization
# --------------------------------------------------------------------------
def e4m3_round(v):
    """Nearest e4m3 value of each element (ties to the even code), float64 in
    and out, written from the format: 3 mantissa bits, so a value in
    [2^k, 2^(k+1)) (k >= -6) sits on a grid of step 2^(k-3); below 2^-6 the
    subnormal grid has step 2^-9; the largest finite value is 448.  NaN
    stays NaN; magnitudes above 448 (infinities included) become 448."""
    v = np.asarray(v, dtype=F64)
    a = np.minimum(np.abs(v), 448.0)        # NaN stays NaN through every step below
    _, ex = np.frexp(a)                     # a = f * 2^ex, 0.5 <= f < 1
    step_exp = np.maximum(ex - 1, -6) - 3   # binade [2^k, 2^(k+1)) (k >= -6) has step 2^(k-3)
    q = np.rint(np.ldexp(a, -step_exp))     # exact scaling; rint rounds half to even
    r = np.minimum(np.ldexp(q, step_exp), 448.0)
    return np.copysign(r, v)


def e4m3_code(v):
    """Code bits (uint8) of values that are already e4m3 values (output of
    e4m3_round): sign, 4 exponent bits (bias 7), 3 mantissa bits; NaN 0x7f."""
    v = np.asarray(v, dtype=F64)
    codes = np.zeros(v.shape, dtype=np.uint8)
    nan = np.isnan(v)
    a = np.abs(np.where(nan, 0.0, v))
    sign = (np.signbit(v) & ~nan).astype(np.uint8) << 7
    _, ex = np.frexp(a)
    k = ex - 1
    normal = a >= 2.0 ** -6
    e_field = np.where(normal, k + 7, 0)
    mant = np.where(normal, np.ldexp(a, -k) - 1.0, np.ldexp(a, 6)) * 8.0
    codes = (sign | (e_field.astype(np.uint8) << 3) | np.rint(mant).astype(np.uint8))
    codes = np.where(a == 0, sign, codes).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), codes).astype(np.uint8)


def block_exponent(amax):
    """Exponent e of a block's scale 2^e (reading 11): the smallest integer
    with amax <= 448 * 2^e; 0 where amax is 0 or not finite; clamped to
    [-127, 127]."""
    amax = np.asarray(amax, dtype=F64)
    e = np.zeros(amax.shape, dtype=np.int64)
    ok = np.isfinite(amax) & (amax > 0)
    a = amax[ok]
    guess = np.ceil(np.log2(a / 448.0)).astype(np.int64)
    # settle the guess exactly against 448 * 2^e (exact in float64)
    guess = np.where(a > np.ldexp(448.0, guess), guess + 1, guess)
    guess = np.where(a <= np.ldexp(448.0, guess - 1), guess - 1, guess)
    e[ok] = np.clip(guess, -127, 127)
    return e


def quantize_blocks_e4m3(a, block_rows: int, codes: bool = True):
    """Block-scaled e4m3 quantization of a [R, C] (reading 11): blocks of
    block_rows x 128 (block_rows = 128 for weights, 1 for activation rows);
    R a multiple of block_rows, C a multiple of 128.  Returns (codes uint8
    [R, C] or None when ``codes`` is false, exponents int64 [R / block_rows,
    C / 128], dequantized float64 [R, C])."""
    a = np.asarray(a, dtype=F64)
    R, C = a.shape
    assert R % block_rows == 0 and C % 128 == 0
    blk = a.reshape(R // block_rows, block_rows, C // 128, 128)
    amax = np.max(np.abs(blk), axis=(1, 3))             # NaN if the block holds a NaN
    e = block_exponent(amax)
    scaled = blk * np.ldexp(1.0, -e)[:, None, :, None]  # exact: a power of two
    deq_codes = e4m3_round(scaled)
    bits = e4m3_code(deq_codes).reshape(R, C) if codes else None
    deq = (deq_codes * np.ldexp(1.0, e)[:, None, :, None]).reshape(R, C)
    return bits, e, deq


def fp8_block_swiglu_expert(x, w_gate, w_up, w_down, gate_up: bool, down: bool):
    """One expert under reading 11: gate/up on the block-dequantized tokens
    and weights if ``gate_up``; H (unrounded) and W_down block-dequantized
    before the down projection if ``down``."""
    x = _f64(x)
    if gate_up:
        xq = quantize_blocks_e4m3(x, 1, codes=False)[2]
        g = xq @ quantize_blocks_e4m3(w_gate, 128, codes=False)[2].T
        u = xq @ quantize_blocks_e4m3(w_up, 128, codes=False)[2].T
    else:
        g, u = x @ _f64(w_gate).T, x @ _f64(w_up).T
    hid = silu(g) * u
    if down:
        return (quantize_blocks_e4m3(hid, 1, codes=False)[2]
                @ quantize_blocks_e4m3(w_down, 128, codes=False)[2].T)
    return hid @ _f64(w_down).T


def fp8_block_expert_rows(x_rows, idx_rows, gate_rows, get_expert, shared, gate_up: bool,
                          down: bool):
    """Layer output for sampled rows under reading 11 (``gate_up``, ``down``:
    which products are block-scaled e4m3); arguments as expert_output_rows,
    the selection and gates coming from the unquantized routing."""
    x_rows = _f64(x_rows)
    y = fp8_block_swiglu_expert(x_rows, *shared, gate_up, down)
    idx_rows = np.asarray(idx_rows)
    for e in np.unique(idx_rows):
        tt, jj = np.nonzero(idx_rows == e)
        ye = fp8_block_swiglu_expert(x_rows[tt], *get_expert(int(e)), gate_up, down)
        y[tt] += gate_rows[tt, jj][:, None] * ye
    return y
