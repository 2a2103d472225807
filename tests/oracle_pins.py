"""Checks that pin the float64 oracle to things other than itself.

Each ``pin_*`` takes the oracle module and raises AssertionError when the
oracle disagrees with a value fixed by the pages or by mathematics:

* hand-derived closed forms (tests/golden/*.txt, each with its citation);
* brute force over every k-subset of experts with exact rational sums;
* invariants: k distinct experts per token, gates summing to one, gates
  unchanged by the bias, load counts summing to T*k;
* textbook reductions of the SwiGLU expert (identity weights reduce it to the
  elementwise silu(x)*x; zero up-projection gives zero);
* equivariances that catch index and transposition mistakes (permuting
  tokens, hidden units or experts);
* the pages' dense formulation against the sparse one.

tests/test_oracle_pins.py runs them on the real oracle, and
tests/test_oracle_mutations.py plants mistakes in the oracle and requires at
least one pin to fail for each.
"""

from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


def _logit(p):
    return math.log(p / (1.0 - p))


def _tiny_layer(rng, T, d, h, E):
    x = rng.standard_normal((T, d))
    w_r = rng.standard_normal((E, d)) / math.sqrt(d)
    b = rng.uniform(-0.05, 0.05, E)
    wg = rng.standard_normal((E, h, d)) / math.sqrt(d)
    wu = rng.standard_normal((E, h, d)) / math.sqrt(d)
    wd = rng.standard_normal((E, d, h)) / math.sqrt(h)
    sh = (rng.standard_normal((h, d)) / math.sqrt(d),
          rng.standard_normal((h, d)) / math.sqrt(d),
          rng.standard_normal((d, h)) / math.sqrt(h))
    return x, w_r, b, (wg, wu, wd), sh


# ---------------------------------------------------------------- routing
def pin_routing_golden(O):
    rows = _read_golden("routing_closed_form.txt")
    kv = {}
    p, idx, gates = {}, {}, {}
    for r in rows:
        key, *vals = r.split()
        if key == "p":
            p[int(vals[0])] = [float(v) for v in vals[1:]]
        elif key == "idx":
            idx[int(vals[0])] = [int(v) for v in vals[1:]]
        elif key == "gates":
            gates[int(vals[0])] = [float(Fraction(v)) for v in vals[1:]]
        else:
            kv[key] = vals
    E, k = int(kv["E"][0]), int(kv["k"][0])
    T = len(p)
    bias = np.array([float(v) for v in kv["bias"]])
    x = np.eye(T)
    w_r = np.array([[_logit(p[t][e]) for t in range(T)] for e in range(E)])
    r = O.route(x, w_r, bias, k)
    assert np.allclose(r["s"], np.array([p[t] for t in range(T)]), rtol=0, atol=1e-14)
    for t in range(T):
        assert list(r["idx"][t]) == idx[t], (t, r["idx"][t], idx[t])
        assert np.allclose(r["gates"][t], gates[t], rtol=0, atol=1e-14)
    load = O.load_counts(r["idx"], E)
    assert list(load) == [int(v) for v in kv["load"]]
    gamma = float(kv["gamma"][0])
    sign = np.array([int(v) for v in kv["sign"]], dtype=np.float32)
    b_new = O.bias_update(bias, load, gamma, T * k)
    # IEEE single-precision subtraction done by numpy's float32 ALU
    expect = np.float32(bias.astype(np.float32)) - np.float32(gamma) * sign
    assert b_new.dtype == np.float32
    assert np.array_equal(b_new, expect.astype(np.float32)), (b_new, expect)


def pin_topk_bruteforce(O):
    """The selected set maximises the exact sum of biased scores over all
    k-subsets; among equal sums the lexicographically smallest index set wins
    (ties go to the lower index).  Slots are ordered by descending score."""
    rng = np.random.default_rng(11)
    for trial in range(60):
        E = int(rng.integers(2, 9))
        k = int(rng.integers(1, min(E, 3) + 1))
        T = 6
        if trial % 3 == 0:   # many exact ties: multiples of 1/8
            z = rng.integers(0, 5, size=(T, E)) / 8.0
        else:
            z = rng.uniform(-1, 1, size=(T, E))
        if trial % 5 == 0:   # a few NaN scores rank below every number
            z[rng.random((T, E)) < 0.2] = np.nan
        idx = O.select_topk(z, k)
        assert idx.shape == (T, k)
        for t in range(T):
            vals = [(-math.inf if math.isnan(v) else Fraction(v)) for v in z[t]]

            def total(c):
                fin = [vals[i] for i in c if vals[i] != -math.inf]
                ninf = sum(1 for i in c if vals[i] == -math.inf)
                return (-ninf, sum(fin, Fraction(0)))
            best = max(itertools.combinations(range(E), k),
                       key=lambda c: (total(c), [-i for i in c]))
            assert sorted(idx[t].tolist()) == list(best), (z[t], idx[t], best)
            assert len(set(idx[t].tolist())) == k
            for j in range(k - 1):
                a, b = vals[idx[t, j]], vals[idx[t, j + 1]]
                assert a > b or (a == b and idx[t, j] < idx[t, j + 1])


def pin_gap(O):
    """The reported k-th/(k+1)-th gap is the margin that separates the
    selected set from the rest: nudging the best unselected score up by more
    than it changes the selection, by less does not."""
    rng = np.random.default_rng(5)
    z = rng.uniform(0, 1, size=(8, 7))
    k = 3
    gap = O.topk_gap(z, k)
    idx = O.select_topk(z, k)
    for t in range(8):
        rest = [e for e in range(7) if e not in idx[t]]
        e_best = max(rest, key=lambda e: z[t, e])
        assert gap[t] > 0
        assert abs(gap[t] - (min(z[t, idx[t]]) - z[t, e_best])) < 1e-15
        z2 = z.copy()
        z2[t, e_best] += 1.5 * gap[t]
        assert e_best in O.select_topk(z2, k)[t]
        z2[t, e_best] = z[t, e_best] + 0.5 * gap[t]
        assert e_best not in O.select_topk(z2, k)[t]


def pin_gate_invariants(O):
    rng = np.random.default_rng(3)
    x, w_r, b, _, _ = _tiny_layer(rng, 40, 16, 8, 12)
    k = 4
    r = O.route(x, w_r, b, k)
    s, g, idx = r["s"], r["gates"], r["idx"]
    assert np.all((s > 0) & (s < 1))
    # sigmoid(-u) = 1 - sigmoid(u); sigmoid(0) = 1/2
    r_neg = O.route(-x, w_r, b, k)
    assert np.allclose(r_neg["s"], 1.0 - s, rtol=0, atol=1e-15)
    assert np.allclose(g.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(g > 0)
    sel = np.take_along_axis(s, idx, axis=1)
    # g proportional to the unbiased affinity of the selected experts
    assert np.allclose(g / g[:, :1], sel / sel[:, :1], rtol=1e-12, atol=0)
    # a constant shift of every bias changes nothing
    r2 = O.route(x, w_r, b + 0.37, k)
    assert np.array_equal(r2["idx"], idx)
    assert np.allclose(r2["gates"], g, rtol=0, atol=1e-15)
    # a large bias on a chosen set forces exactly that set, and the gates
    # are that set's unbiased affinities normalised (bias invariance)
    S = [1, 5, 7, 10]
    b3 = b.copy()
    b3[S] += 100.0
    r3 = O.route(x, w_r, b3, k)
    for t in range(x.shape[0]):
        assert sorted(r3["idx"][t].tolist()) == S
        u = x[t] @ w_r[S].T
        sS = np.array([1.0 / (1.0 + math.exp(-v)) for v in u])
        order = [S.index(e) for e in r3["idx"][t]]
        assert np.allclose(r3["gates"][t], (sS / sS.sum())[order], rtol=0, atol=1e-14)
    # selecting every expert: gates are s / sum(s) over all experts
    rk = O.route(x, w_r, b, 12)
    Gfull = np.zeros_like(s)
    np.put_along_axis(Gfull, rk["idx"], rk["gates"], axis=1)
    assert np.allclose(Gfull, s / s.sum(axis=1, keepdims=True), rtol=0, atol=1e-15)


def pin_router_one_hot(O):
    """One-hot tokens read one router column: u[t,e] = W_r[e,t]."""
    rng = np.random.default_rng(9)
    w_r = rng.standard_normal((6, 4))
    u, s = O.router_affinity(np.eye(4), w_r)
    assert np.array_equal(u, w_r.T)
    assert np.allclose(s, [[1.0 / (1.0 + math.exp(-v)) for v in row] for row in w_r.T],
                       rtol=0, atol=1e-16)
    u2, _ = O.router_affinity(np.array([[2.0, 0, 0, -1.0]]), w_r)
    assert np.allclose(u2[0], 2.0 * w_r[:, 0] - w_r[:, 3], rtol=0, atol=1e-15)


def pin_load_counts(O):
    rng = np.random.default_rng(4)
    for E, k, T in [(16, 4, 50), (7, 7, 9), (5, 1, 1), (9, 2, 0)]:
        z = rng.uniform(0, 1, size=(T, E))
        idx = O.select_topk(z, k)
        load = O.load_counts(idx, E)
        assert load.shape == (E,) and load.sum() == T * k
        for e in range(E):
            assert load[e] == sum(int(v == e) for row in idx.tolist() for v in row)
    idx = np.array([[3, 0], [3, 1], [2, 3]])
    assert O.load_counts(idx, 5).tolist() == [1, 1, 1, 3, 0]


def pin_bias_update(O):
    g32 = np.float32(1e-3)
    # float32(1e-3) is 0.001000000047497451305389404296875 exactly
    assert float(g32) == 0.001000000047497451305389404296875
    b = np.array([0.0, 0.5, -0.25, 0.0078125], dtype=np.float32)
    # E = 4, TK = 8 -> mean 2: loads [4, 2, 1, 1] -> signs [+1, 0, -1, -1]
    out = O.bias_update(b, np.array([4, 2, 1, 1]), 1e-3, 8)
    expect = np.array([b[0] - g32, b[1], b[2] + g32, b[3] + g32], dtype=np.float32)
    assert out.dtype == np.float32 and np.array_equal(out, expect), (out, expect)
    assert out[0] == -g32 and out[1] == np.float32(0.5)
    # non-integer mean: E = 3, TK = 4 -> mean 4/3: loads [2, 1, 1] -> [+1, -1, -1]
    out = O.bias_update(np.zeros(3, np.float32), np.array([2, 1, 1]), 1e-3, 4)
    assert np.array_equal(out, np.array([-g32, g32, g32], dtype=np.float32))
    # balanced load leaves the bias unchanged (sign(0) = 0)
    bb = np.array([0.1, -0.2, 0.3], dtype=np.float32)
    assert np.array_equal(O.bias_update(bb, np.array([2, 2, 2]), 1e-3, 6), bb)
    # over many steps each bias moves by at most gamma per step (+ rounding)
    rng = np.random.default_rng(1)
    E = 8
    b0 = rng.uniform(-0.01, 0.01, E).astype(np.float32)
    bt = b0.copy()
    for step in range(50):
        load = rng.multinomial(32, np.ones(E) / E)
        bt = O.bias_update(bt, load, 1e-3, 32)
        assert np.all(np.abs(bt.astype(np.float64) - b0) <= (step + 1) * 1.0000001e-3 + 1e-8)


# ---------------------------------------------------------------- experts
def pin_swiglu_reductions(O):
    L3 = math.log(3.0)
    # identity weights: E(x) = silu(x) * x elementwise
    x = np.array([[L3, -L3, 0.0, 2.0]])
    I4 = np.eye(4)
    y = O.swiglu_expert(x, I4, I4, I4)
    sig = lambda v: 1.0 / (1.0 + math.exp(-v))  # noqa: E731
    expect = [0.75 * L3 * L3, 0.25 * L3 * L3, 0.0, 2.0 * sig(2.0) * 2.0]
    assert np.allclose(y[0], expect, rtol=1e-15, atol=1e-15)
    # gate row picks feature 0, up row picks feature 1, down writes to feature 2
    wg = np.array([[1.0, 0, 0, 0]])
    wu = np.array([[0, 1.0, 0, 0]])
    wd = np.array([[0.0], [0.0], [3.0], [0.0]])
    y = O.swiglu_expert(np.array([[L3, 2.0, 7.0, 9.0]]), wg, wu, wd)
    assert np.allclose(y[0], [0, 0, 3.0 * 0.75 * L3 * 2.0, 0], rtol=1e-15, atol=1e-15)
    # zero up projection gives zero; scaling down/up scales the output
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 6))
    wg, wu, wd = rng.standard_normal((3, 6)), rng.standard_normal((3, 6)), rng.standard_normal((6, 3))
    assert np.array_equal(O.swiglu_expert(x, wg, 0 * wu, wd), np.zeros((5, 6)))
    y = O.swiglu_expert(x, wg, wu, wd)
    assert np.allclose(O.swiglu_expert(x, wg, 2.5 * wu, wd), 2.5 * y, rtol=1e-13, atol=1e-14)
    assert np.allclose(O.swiglu_expert(x, wg, wu, -3 * wd), -3 * y, rtol=1e-13, atol=1e-14)
    # permuting hidden units (rows of W_gate, W_up, columns of W_down) is a no-op
    P = rng.permutation(3)
    assert np.allclose(O.swiglu_expert(x, wg[P], wu[P], wd[:, P]), y, rtol=1e-13, atol=1e-14)
    # permuting tokens permutes output rows
    Q = rng.permutation(5)
    assert np.allclose(O.swiglu_expert(x[Q], wg, wu, wd), y[Q], rtol=1e-13, atol=1e-14)
    # rectangular shapes: d = 6, h = 3 -> output [n, d]
    assert y.shape == (5, 6)
    # the gate path is not symmetric in gate/up: swapping them changes the result
    assert not np.allclose(O.swiglu_expert(x, wu, wg, wd), y)


def pin_scalar_layer_golden(O):
    rows = _read_golden("scalar_layer_closed_form.txt")
    L = math.log(3.0) ** 2
    data, cases = {}, []
    for r in rows:
        if r.startswith("case"):
            parts = [p.split() for p in r.split("|")]
            head = parts[0]
            cases.append({
                "k": int(head[2]), "b": [float(head[3]), float(head[4])],
                "idx": [int(v) for v in parts[1][1:]],
                "gates": [float(Fraction(v)) for v in parts[2][1:]],
                "y": float(Fraction(parts[3][1])) * L,
            })
        else:
            key, *vals = r.split()
            if key == "expert":
                data.setdefault("expert", {})[int(vals[0])] = [float(v) for v in vals[1:]]
            else:
                data[key] = [float(v) for v in vals]
    x = np.array([[data["x"][0]]])
    w_r = np.array([[data["w_router"][0]], [data["w_router"][1]]])
    ex = data["expert"]
    experts = (np.array([[[ex[e][0]]] for e in range(2)]),
               np.array([[[ex[e][1]]] for e in range(2)]),
               np.array([[[ex[e][2]]] for e in range(2)]))
    sh = data["shared"]
    shared = (np.array([[sh[0]]]), np.array([[sh[1]]]), np.array([[sh[2]]]))
    for c in cases:
        for fwd in (O.moe_forward_dense, O.moe_forward_sparse):
            out = fwd(x, w_r, np.array(c["b"]), experts, shared, c["k"])
            assert out["idx"][0].tolist() == c["idx"], (c, out["idx"])
            assert np.allclose(out["gates"][0], c["gates"], rtol=0, atol=1e-14)
            assert abs(out["y"][0, 0] - c["y"]) < 1e-13, (c, out["y"])


def pin_layer_reductions(O):
    rng = np.random.default_rng(8)
    x, w_r, b, (wg, wu, wd), sh = _tiny_layer(rng, 12, 6, 4, 5)
    # one expert selected from one: gate 1, y = shared(x) + expert(x)
    out = O.moe_forward_dense(x, w_r[:1], b[:1], (wg[:1], wu[:1], wd[:1]), sh, 1)
    assert np.allclose(out["gates"], 1.0, rtol=0, atol=0)
    ident = np.eye(6)
    out_id = O.moe_forward_dense(x, w_r[:1], b[:1], (ident[None, :, :], ident[None], ident[None]),
                                 (ident, ident, ident), 1)
    # both experts identity: y = 2 * silu(x) * x elementwise
    assert np.allclose(out_id["y"], 2 * x * x / (1 + np.exp(-x)), rtol=1e-14, atol=1e-14)
    # zero routed down-projections leave only the shared expert
    out0 = O.moe_forward_dense(x, w_r, b, (wg, wu, 0 * wd), sh, 2)
    only_shared = O.moe_forward_dense(x, w_r, b, (wg, wu, wd), (sh[0], sh[1], 0 * sh[2]), 2)
    full = O.moe_forward_dense(x, w_r, b, (wg, wu, wd), sh, 2)
    assert np.allclose(out0["y"] + only_shared["y"], full["y"], rtol=1e-13, atol=1e-14)
    # zero shared down-projection and all experts selected: y = sum_e s_e/sum(s) E_e(x)
    allk = O.moe_forward_dense(x, w_r, b, (wg, wu, wd), (sh[0], sh[1], 0 * sh[2]), 5)
    s = 1.0 / (1.0 + np.exp(-(x @ w_r.T)))
    ref = sum((s[:, e:e + 1] / s.sum(axis=1, keepdims=True)) * O.swiglu_expert(x, wg[e], wu[e], wd[e])
              for e in range(5))
    assert np.allclose(allk["y"], ref, rtol=1e-13, atol=1e-14)


def pin_equivariance(O):
    rng = np.random.default_rng(6)
    x, w_r, b, (wg, wu, wd), sh = _tiny_layer(rng, 10, 8, 6, 7)
    k = 3
    base = O.moe_forward_dense(x, w_r, b, (wg, wu, wd), sh, k)
    # permuting tokens permutes every per-token output
    Q = rng.permutation(10)
    o = O.moe_forward_dense(x[Q], w_r, b, (wg, wu, wd), sh, k)
    assert np.array_equal(o["idx"], base["idx"][Q])
    assert np.allclose(o["y"], base["y"][Q], rtol=1e-13, atol=1e-14)
    # relabelling experts (router rows, biases and weights together) leaves
    # y unchanged and relabels the selection
    P = rng.permutation(7)
    o = O.moe_forward_dense(x, w_r[P], b[P], (wg[P], wu[P], wd[P]), sh, k)
    inv = np.argsort(P)
    assert np.array_equal(P[o["idx"]], base["idx"])
    assert np.array_equal(inv[base["idx"]], o["idx"])
    assert np.allclose(o["y"], base["y"], rtol=1e-13, atol=1e-14)
    # duplicated router rows with equal bias tie exactly; the lower index wins
    w2 = w_r.copy()
    w2[4] = w2[2]
    b2 = b.copy()
    b2[4] = b2[2]
    b2[2] += 50.0
    b2[4] += 50.0
    r = O.route(x, w2, b2, 1)
    assert np.all(r["idx"][:, 0] == 2)


def pin_dense_sparse_agree(O):
    rng = np.random.default_rng(7)
    for (T, d, h, E, k) in [(9, 8, 4, 6, 2), (5, 4, 8, 3, 3), (7, 6, 6, 8, 1)]:
        x, w_r, b, ex, sh = _tiny_layer(rng, T, d, h, E)
        dn = O.moe_forward_dense(x, w_r, b, ex, sh, k)
        sp = O.moe_forward_sparse(x, w_r, b, ex, sh, k)
        assert np.array_equal(dn["idx"], sp["idx"])
        rel = np.linalg.norm(dn["y"] - sp["y"]) / np.linalg.norm(dn["y"])
        assert rel < 1e-12, rel
        rows = O.expert_output_rows(x, dn["idx"], dn["gates"],
                                    lambda e: (ex[0][e], ex[1][e], ex[2][e]), sh)
        assert np.linalg.norm(rows - dn["y"]) / np.linalg.norm(dn["y"]) < 1e-12


def pin_route_and_update(O):
    rng = np.random.default_rng(12)
    x, w_r, b, _, _ = _tiny_layer(rng, 30, 8, 4, 6)
    r = O.route_and_update(x, w_r, b.astype(np.float32), 2, 1e-3)
    assert r["load"].sum() == 60
    over = r["load"] * 6 > 60
    under = r["load"] * 6 < 60
    bb = b.astype(np.float32)
    assert np.all(r["bias_new"][over] < bb[over])
    assert np.all(r["bias_new"][under] > bb[under])


def pin_balance_loss_golden(O):
    """Hand-derived sequence-wise balance losses (tests/golden)."""
    alpha = 1e-4
    for row in _read_golden("balance_loss_closed_form.txt"):
        parts = row.split()
        E, k, S = int(parts[1]), int(parts[2]), int(parts[3])
        toks, want = parts[4:-1], float(parts[-1])
        s = np.array([[float(v) for v in t.split("|")[0].split(",")] for t in toks])
        idx = np.array([[int(v) for v in t.split("|")[1].split(",")] for t in toks])
        assert s.shape == (S, E) and idx.shape == (S, k)
        got = O.sequence_balance_loss(s, idx, S, alpha)
        assert got.shape == (1,)
        assert abs(got[0] - want * alpha) <= 1e-15, (parts[0], got[0], want * alpha)


def pin_balance_loss_closed_forms(O):
    """Uniform affinities and perfectly balanced selection give exactly
    alpha per sequence; full collapse onto one expert gives alpha * E; a
    short last sequence uses its own length; the loss ignores per-token
    scaling of s and relabelling of the experts."""
    alpha = 1e-4
    E, k, S = 8, 2, 8
    T = 2 * S
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)])
    s = np.full((T, E), 0.37)
    L = O.sequence_balance_loss(s, idx, S, alpha)
    assert L.shape == (2,) and np.allclose(L, alpha, rtol=0, atol=1e-18)
    # collapse: every token picks expert 3 and all its affinity is there
    s1 = np.zeros((5, E))
    s1[:, 3] = 0.9
    L1 = O.sequence_balance_loss(s1, np.full((5, 1), 3), 5, alpha)
    assert abs(L1[0] - alpha * E) <= 1e-18
    # T = 10 with S = 8: the second sequence has 2 tokens, each balanced
    idx2 = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(8)] + [[0, 1], [2, 3]])
    s2 = np.full((10, E), 0.5)
    L2 = O.sequence_balance_loss(s2, idx2, 8, alpha)
    # second sequence: counts 1 for experts 0..3 -> f = 8/(2*2) = 2 there,
    # P = 1/8 everywhere -> L = alpha * 4 * 2 / 8 = alpha
    assert L2.shape == (2,) and np.allclose(L2, alpha, rtol=0, atol=1e-18)
    rng = np.random.default_rng(21)
    s3 = rng.uniform(0.05, 0.95, size=(24, 6))
    idx3 = np.stack([rng.choice(6, size=2, replace=False) for _ in range(24)])
    base = O.sequence_balance_loss(s3, idx3, 8, alpha)
    scaled = O.sequence_balance_loss(s3 * rng.uniform(0.5, 2.0, size=(24, 1)), idx3, 8, alpha)
    assert np.allclose(base, scaled, rtol=1e-12, atol=0)
    perm = rng.permutation(6)  # expert e becomes perm[e]
    s_p = np.empty_like(s3)
    s_p[:, perm] = s3
    assert np.allclose(O.sequence_balance_loss(s_p, perm[idx3], 8, alpha), base, rtol=1e-12, atol=0)


def _backward_case(seed, T=6, d=5, h=4, E=5, k=2):
    """Tiny layer whose top-k gaps are wide enough that the finite
    differences below never change the selection."""
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, d))
    w_r = rng.normal(size=(E, d))
    b = np.linspace(0.3, -0.3, E)
    ex = (rng.normal(size=(E, h, d)), rng.normal(size=(E, h, d)), rng.normal(size=(E, d, h)))
    sh = (rng.normal(size=(h, d)), rng.normal(size=(h, d)), rng.normal(size=(d, h)))
    return x, w_r, b, ex, sh, rng.normal(size=(T, d))


def pin_backward_finite_differences(O):
    """Every gradient entry against a central difference of the forward
    oracle's <dy, y>, in float64 (step 1e-6)."""
    x, w_r, b, ex, sh, dy = _backward_case(31)
    k, eps = 2, 1e-6
    assert O.topk_gap(O.route(x, w_r, b, k)["z"], k).min() > 1e-3
    g = O.moe_backward_dense(x, w_r, b, ex, sh, k, dy)

    def loss(x_, w_r_, ex_, sh_):
        return float((dy * O.moe_forward_dense(x_, w_r_, b, ex_, sh_, k)["y"]).sum())

    def check(arr, grad, place):
        worst = 0.0
        for i in np.ndindex(arr.shape):
            hi, lo = arr.copy(), arr.copy()
            hi[i] += eps
            lo[i] -= eps
            fd = (loss(*place(hi)) - loss(*place(lo))) / (2 * eps)
            worst = max(worst, abs(fd - grad[i]) / (1.0 + abs(grad[i])))
        assert worst < 1e-6, worst

    check(x, g["dx"], lambda a: (a, w_r, ex, sh))
    check(w_r, g["dW_router"], lambda a: (x, a, ex, sh))
    for j, name in enumerate(["dW_gate", "dW_up", "dW_down"]):
        check(ex[j], g[name], lambda a, j=j: (x, w_r, tuple(a if m == j else ex[m] for m in range(3)), sh))
    for j, name in enumerate(["dsh_gate", "dsh_up", "dsh_down"]):
        check(sh[j], g[name], lambda a, j=j: (x, w_r, ex, tuple(a if m == j else sh[m] for m in range(3))))


def pin_backward_special_cases(O):
    """One routed expert (gate identically 1): the router gets no gradient.
    Gates are invariant to scaling the selected affinities together, so
    sum_j s_j dL/ds_j = 0 over each token's selection.  Zero routed weights:
    only the shared expert carries dx, and no gate has a gradient."""
    x, w_r, b, ex, sh, dy = _backward_case(32, E=1, k=1)
    g = O.moe_backward_dense(x, w_r, b, ex, sh, 1, dy)
    assert np.array_equal(g["dW_router"], np.zeros_like(w_r))
    x, w_r, b, ex, sh, dy = _backward_case(33, E=6, k=3)
    g = O.moe_backward_dense(x, w_r, b, ex, sh, 3, dy)
    s = O.route(x, w_r, b, 3)["s"]
    ds = g["du"] / (s * (1.0 - s))
    s_sel = np.take_along_axis(s, g["idx"], axis=1)
    ds_sel = np.take_along_axis(ds, g["idx"], axis=1)
    assert np.abs((s_sel * ds_sel).sum(axis=1)).max() < 1e-12 * (1 + np.abs(ds_sel).max())
    zero = tuple(np.zeros_like(w) for w in ex)
    g0 = O.moe_backward_dense(x, w_r, b, zero, sh, 3, dy)
    dx_sh = O.swiglu_expert_backward(x, *sh, dy)[0]
    assert np.allclose(g0["dx"], dx_sh, rtol=1e-13, atol=1e-13)
    assert np.array_equal(g0["dW_router"], np.zeros_like(w_r))


def pin_backward_rows_agree(O):
    """The per-token-rows backward gives the dense backward's dx rows."""
    x, w_r, b, ex, sh, dy = _backward_case(34, T=9, E=6, k=3)
    full = O.moe_backward_dense(x, w_r, b, ex, sh, 3, dy)
    rows = np.array([0, 4, 8])
    got = O.backward_token_rows(x[rows], w_r, b, lambda e: (ex[0][e], ex[1][e], ex[2][e]), sh, 3,
                                dy[rows])
    assert np.allclose(got, full["dx"][rows], rtol=1e-12, atol=1e-12)


def _e4m3_values():
    """Every finite e4m3 value, from the format's definition (1 sign, 4
    exponent bits with bias 7, 3 mantissa bits; exponent field 0 is
    subnormal; code 0x7f / 0xff is NaN)."""
    vals = []
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        sgn = -1.0 if c >> 7 else 1.0
        e, m = (c >> 3) & 15, c & 7
        mag = math.ldexp(1 + m / 8, e - 7) if e else math.ldexp(m / 8, -6)
        vals.append((c, sgn * mag))
    return vals


def pin_quantize_e4m3(O):
    """Per-row e4m3 quantization: a row already on the e4m3 grid with
    maximum 448 is kept exactly with scale 1 and the format's own codes;
    scaling a row by a power of two scales only its scale; the largest
    magnitude maps to +-448; a zero row gets scale 1 and zero codes; the
    error of every normal value is at most 2^-4 of it."""
    grid = _e4m3_values()
    codes = np.array([c for c, _ in grid], dtype=np.uint8)
    vals = np.array([v for _, v in grid])
    q, sc, deq = O.quantize_rows_e4m3(vals[None, :])
    assert sc[0] == 1.0 and np.array_equal(q[0], codes) and np.array_equal(deq[0], vals)
    rng = np.random.default_rng(41)
    row = rng.normal(size=(3, 200)).astype(np.float32)
    q1, s1, _ = O.quantize_rows_e4m3(row)
    q2, s2, _ = O.quantize_rows_e4m3(row * np.float32(2.0 ** 7))
    assert np.array_equal(q1, q2) and np.array_equal(s2, s1 * np.float32(2.0 ** 7))
    top = np.abs(row).argmax(axis=1)
    assert set(q1[np.arange(3), top].tolist()) <= {0x7E, 0xFE}
    qz, sz, dz = O.quantize_rows_e4m3(np.zeros((1, 64), dtype=np.float32))
    assert sz[0] == 1.0 and not qz.any() and not dz.any()
    _, s3, d3 = O.quantize_rows_e4m3(row)
    normal = np.abs(row) >= (2.0 ** -6) * s3[:, None]
    assert np.all(np.abs(d3 - row)[normal] <= 2.0 ** -4 * np.abs(row)[normal])


def _fp8_case(seed, exact):
    """A small layer whose gate/up weights are on the e4m3 grid times a power
    of two with each row's maximum at 448 times that power (so per-row
    quantization keeps them exactly); tokens on that grid too if ``exact``."""
    rng = np.random.default_rng(seed)
    grid = np.array([v for _, v in _e4m3_values() if abs(v) <= 448.0])

    def on_grid(shape):
        a = rng.choice(grid, size=shape)
        a[..., 0] = 448.0 * rng.choice([-1.0, 1.0], size=shape[:-1])  # row max 448
        return a * 2.0 ** rng.integers(-12, -6, size=shape[:-1])[..., None]

    T, d, h, E, k = 5, 16, 8, 4, 2
    x = on_grid((T, d)) if exact else rng.normal(size=(T, d)).astype(np.float32).astype(np.float64)
    experts = [(on_grid((h, d)), on_grid((h, d)), rng.normal(size=(d, h)) * 0.1) for _ in range(E)]
    shared = (on_grid((h, d)), on_grid((h, d)), rng.normal(size=(d, h)) * 0.1)
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)])
    gates = rng.uniform(0.1, 1.0, size=(T, k))
    return x, idx, gates, experts, shared


def pin_fp8_gate_up(O):
    """The fp8 gate/up layer: with tokens and gate/up weights that per-row
    e4m3 quantization keeps exactly, it IS the unquantized layer; with
    weights kept exactly, it is the unquantized layer on the tokens'
    dequantized values; the down projection is never quantized."""
    x, idx, gates, ex, sh = _fp8_case(43, exact=True)
    got = O.fp8_gate_up_rows(x, idx, gates, lambda e: ex[e], sh)
    ref = O.expert_output_rows(x, idx, gates, lambda e: ex[e], sh)
    assert np.array_equal(got, ref)
    x, idx, gates, ex, sh = _fp8_case(44, exact=False)
    xq = O.quantize_rows_e4m3(x)[2]
    assert not np.array_equal(xq, x)
    got = O.fp8_gate_up_rows(x, idx, gates, lambda e: ex[e], sh)
    ref = O.expert_output_rows(xq, idx, gates, lambda e: ex[e], sh)
    assert np.allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    # a W_down off the e4m3 grid (normal values) enters unrounded
    sh2 = (sh[0], sh[1], sh[2] * 1.0001)
    ref2 = O.expert_output_rows(xq, idx, gates, lambda e: ex[e], sh2)
    got2 = O.fp8_gate_up_rows(x, idx, gates, lambda e: ex[e], sh2)
    assert np.allclose(got2, ref2, rtol=0, atol=1e-12 * np.abs(ref2).max())


def pin_e4m3_round(O):
    """e4m3 rounding written from the format: every finite e4m3 value is kept
    with the format's own code; the midpoint of two neighbours goes to the
    one with the even code; fp32 values agree with PyTorch's float8_e4m3fn
    conversion (a separate implementation); NaN stays NaN, infinities and
    magnitudes above 448 become +-448."""
    grid = _e4m3_values()
    codes = np.array([c for c, _ in grid], dtype=np.uint8)
    vals = np.array([v for _, v in grid])
    assert np.array_equal(O.e4m3_round(vals), vals)
    assert np.array_equal(O.e4m3_code(vals[vals != 0]), codes[vals != 0])
    pos = sorted({v for _, v in grid if v >= 0})
    code_of = {v: c for c, v in grid if v >= 0 and not (v == 0 and c)}
    for lo, hi in zip(pos[:-1], pos[1:]):
        even = lo if code_of[lo] % 2 == 0 else hi
        assert O.e4m3_round(np.array([(lo + hi) / 2]))[0] == even, (lo, hi)
        assert O.e4m3_round(np.array([-(lo + hi) / 2]))[0] == -even
    import torch
    rng = np.random.default_rng(47)
    v = (rng.normal(size=20000) * np.exp2(rng.integers(-14, 8, size=20000))).astype(np.float32)
    v = np.clip(v, -448, 448).astype(np.float64)
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn)
    assert np.array_equal(O.e4m3_round(v), ref.to(torch.float64).numpy())
    assert np.array_equal(O.e4m3_code(O.e4m3_round(v)), ref.view(torch.uint8).numpy())
    sp = O.e4m3_round(np.array([np.nan, np.inf, -np.inf, 1e6, -500.0]))
    assert np.isnan(sp[0]) and list(sp[1:]) == [448.0, -448.0, 448.0, -448.0]


def pin_block_exponent(O):
    """The block scale exponent: 448 * 2^(e-1) < amax <= 448 * 2^e, checked by
    brute force over e; exact boundaries; 0 for zero or non-finite blocks;
    clamped to the UE8M0 range [-127, 127]."""
    rng = np.random.default_rng(48)
    amax = np.abs(rng.normal(size=4000)) * np.exp2(rng.integers(-60, 60, size=4000))
    e = O.block_exponent(amax)
    for a, ee in zip(amax, e):
        cand = [k for k in range(-130, 130) if a <= 448.0 * 2.0 ** k]
        assert ee == min(cand), (a, ee)
    edge = np.array([448.0, 448.0 * (1 + 2.0 ** -52), 224.0, 224.0 * (1 + 2.0 ** -52), 1.0,
                     448.0 * 2.0 ** -20, 0.0, np.inf, np.nan, 1e-45, 2.0 ** 140])
    assert list(O.block_exponent(edge)) == [0, 1, -1, 0, -8, -20, 0, 0, 0, -127, 127]


def _block_grid_matrix(rng, R, C, br, lo=-9, hi=-3):
    """A matrix on the block grid: every br x 128 block is e4m3 values times
    2^e_block with one element of magnitude in (224, 448], so block
    quantization keeps it exactly with exponents e_block."""
    grid = np.array([v for _, v in _e4m3_values() if abs(v) <= 448.0])
    nb_r, nb_c = R // br, C // 128
    e = rng.integers(lo, hi, size=(nb_r, nb_c))
    a = rng.choice(grid[np.abs(grid) < 224], size=(nb_r, br, nb_c, 128))
    a[:, 0, :, 0] = rng.choice([-448.0, 320.0, 240.0, -256.0], size=(nb_r, nb_c))
    a = a * np.ldexp(1.0, e)[:, None, :, None]
    return a.reshape(R, C), e


def pin_quantize_blocks(O):
    """Block quantization: a matrix on the block grid is kept exactly with
    its exponents; blocks are independent (changing one block changes only
    its own codes and exponent); scaling one block by 2^j shifts its
    exponent by j and keeps its codes; the error of every normal value is at
    most 2^-4 of it; a block with a NaN gets exponent 0 and a NaN code only
    where the NaN is."""
    rng = np.random.default_rng(49)
    for br in (128, 1):
        R = 256 if br == 128 else 6
        a, e = _block_grid_matrix(rng, R, 384, br)
        q, eq, deq = O.quantize_blocks_e4m3(a, br)
        assert np.array_equal(deq, a) and np.array_equal(eq, e)
        b = a.copy()
        b[:br, 128:256] *= 2.0 ** 5
        b[br:2 * br, 256:384] = rng.normal(size=(br, 128))
        qb, eb, _ = O.quantize_blocks_e4m3(b, br)
        assert eb[0, 1] == e[0, 1] + 5 and np.array_equal(qb[:br, 128:256], q[:br, 128:256])
        same = np.ones_like(q, dtype=bool)
        same[br:2 * br, 256:384] = False
        assert np.array_equal(qb[same], q[same])
        diff_e = np.ones_like(e, dtype=bool)
        diff_e[0, 1] = diff_e[1, 2] = False
        assert np.array_equal(eb[diff_e], e[diff_e])
    x = rng.normal(size=(5, 256)) * np.exp2(rng.integers(-8, 8, size=(5, 1)))
    _, ex, dx = O.quantize_blocks_e4m3(x, 1)
    scale = np.repeat(np.ldexp(1.0, ex), 128, axis=1)
    normal = np.abs(x) >= 2.0 ** -6 * scale
    assert np.all(np.abs(dx - x)[normal] <= 2.0 ** -4 * np.abs(x)[normal])
    assert np.all(np.abs(dx - x)[~normal] <= 2.0 ** -10 * scale[~normal])
    y = x.copy()
    y[2, 130] = np.nan
    qy, ey, dy = O.quantize_blocks_e4m3(y, 1)
    assert ey[2, 1] == 0 and qy[2, 130] == 0x7F and np.isnan(dy[2, 130])
    assert np.isfinite(np.delete(dy[2], 130)).all()


def _nearest_e4m3_times(v, e):
    """Brute force: the e4m3 grid value times 2^e nearest to v, ties to the
    even code (independent of the oracle's rounding arithmetic)."""
    grid = _e4m3_values()
    best = None
    for c, g in grid:
        w = g * 2.0 ** e
        d = abs(w - v)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c, w)
    return best[2]


def _brute_block_quant(a, br):
    """Block quantization by brute force: each br x 128 block's exponent by
    search over e, each element the nearest grid value times 2^e (ties to
    the even code)."""
    grid = _e4m3_values()
    gv = np.array([g for _, g in grid])
    gc = np.array([c for c, _ in grid])
    out = np.empty_like(a)
    for r0 in range(0, a.shape[0], br):
        for c0 in range(0, a.shape[1], 128):
            blk = a[r0:r0 + br, c0:c0 + 128]
            amax = np.abs(blk).max()
            e = min(kk for kk in range(-130, 130) if amax <= 448.0 * 2.0 ** kk)
            cand = gv * 2.0 ** e
            dist = np.abs(blk[..., None] - cand)
            best = dist.min(axis=-1, keepdims=True)
            ties = dist == best
            pick = np.where(ties & (gc % 2 == 0), 0, 1) + np.where(ties, 0, 2)
            out[r0:r0 + br, c0:c0 + 128] = cand[np.argmin(pick, axis=-1)]
    return out


def pin_fp8_block_layer(O):
    """The block-scaled layer: with tokens and weights on the block grid the
    gate/up products are exact (the layer IS the unquantized layer when the
    down projection is not quantized); with the down projection quantized,
    each hidden row's 128-unit blocks are rounded by brute force to the
    nearest grid point at the block's exponent, from the unrounded H; the
    shared expert and the gates enter as in the unquantized layer."""
    rng = np.random.default_rng(50)
    T, d, h, E, k = 3, 256, 256, 3, 2
    x, _ = _block_grid_matrix(rng, T, d, 1)
    ex = [(_block_grid_matrix(rng, h, d, 128)[0], _block_grid_matrix(rng, h, d, 128)[0],
           _block_grid_matrix(rng, d, h, 128)[0]) for _ in range(E)]
    sh = (_block_grid_matrix(rng, h, d, 128)[0], _block_grid_matrix(rng, h, d, 128)[0],
          rng.normal(size=(d, h)) * 0.05)
    idx = np.array([[0, 2], [1, 0], [2, 1]])
    gates = rng.uniform(0.2, 1.0, size=(T, k))
    got = O.fp8_block_expert_rows(x, idx, gates, lambda e: ex[e], sh, gate_up=True, down=False)
    ref = O.expert_output_rows(x, idx, gates, lambda e: ex[e], sh)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13 * np.abs(ref).max())
    # the down projection: H from the exact gate/up products, never rounded
    wg, wu, wd = ex[1]
    hid = O.silu(x @ wg.T) * (x @ wu.T)
    hq = np.empty_like(hid)
    for r in range(T):
        for b in range(h // 128):
            seg = hid[r, 128 * b:128 * (b + 1)]
            amax = np.abs(seg).max()
            e = min(kk for kk in range(-130, 130) if amax <= 448.0 * 2.0 ** kk)
            hq[r, 128 * b:128 * (b + 1)] = [_nearest_e4m3_times(v, e) for v in seg]
    y_ref = hq @ wd.T  # wd is on the block grid: kept exactly
    y = O.fp8_block_swiglu_expert(x, wg, wu, wd, gate_up=True, down=True)
    assert np.allclose(y, y_ref, rtol=1e-13, atol=1e-13 * np.abs(y_ref).max())
    assert not np.allclose(y, hid @ wd.T, rtol=1e-6)
    # neither product quantized: the textbook expert
    assert np.array_equal(O.fp8_block_swiglu_expert(x, wg, wu, wd, gate_up=False, down=False),
                          O.swiglu_expert(x, wg, wu, wd))
    # operands off the grid: every operand block-quantized by brute force
    xr = rng.normal(size=(2, 128))
    wr = [rng.normal(size=(128, 128)) * 0.09 for _ in range(3)]
    qx = _brute_block_quant(xr, 1)
    qw = [_brute_block_quant(w, 128) for w in wr]
    hid = O.silu(qx @ qw[0].T) * (qx @ qw[1].T)
    y_ref = _brute_block_quant(hid, 1) @ qw[2].T
    y = O.fp8_block_swiglu_expert(xr, *wr, gate_up=True, down=True)
    assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-12 * np.abs(y_ref).max())


PINS = [
    pin_routing_golden,
    pin_topk_bruteforce,
    pin_gap,
    pin_gate_invariants,
    pin_router_one_hot,
    pin_load_counts,
    pin_bias_update,
    pin_swiglu_reductions,
    pin_scalar_layer_golden,
    pin_layer_reductions,
    pin_equivariance,
    pin_dense_sparse_agree,
    pin_route_and_update,
    pin_balance_loss_golden,
    pin_balance_loss_closed_forms,
    pin_backward_finite_differences,
    pin_backward_special_cases,
    pin_backward_rows_agree,
    pin_quantize_e4m3,
    pin_fp8_gate_up,
    pin_e4m3_round,
    pin_block_exponent,
    pin_quantize_blocks,
    pin_fp8_block_layer,
]
