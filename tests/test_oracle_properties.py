"""Properties of the float64 oracle over random small problems (hypothesis).

Each property is fixed by the definitions, not by the oracle itself: the
selection against brute force over all k-subsets, the gates' normalisation
and proportionality, the bias's effect on selection only, dense against
sparse evaluation, the bias step's bound, and the e4m3 quantization's error
bound.  Shapes stay tiny so the suite runs in seconds.
"""
import itertools

import numpy as np
from hypothesis import given, settings
from hypothesis import strategies as st

from oracle import moe_oracle as O

SETTINGS = settings(max_examples=40, deadline=None)


@st.composite
def routing_case(draw):
    T = draw(st.integers(1, 6))
    d = draw(st.integers(1, 8))
    E = draw(st.integers(1, 7))
    k = draw(st.integers(1, E))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, d))
    w = rng.normal(size=(E, d)) / np.sqrt(d)
    b = rng.uniform(-0.05, 0.05, size=E)
    return x, w, b, k


@SETTINGS
@given(routing_case())
def test_selection_is_the_best_k_subset(case):
    x, w, b, k = case
    r = O.route(x, w, b, k)
    z = O.biased_scores(r["s"], b)
    E = w.shape[0]
    for t in range(x.shape[0]):
        best = max(itertools.combinations(range(E), k),
                   key=lambda c: (sum(z[t, list(c)]), [-e for e in c]))
        assert sorted(r["idx"][t].tolist()) == sorted(best)
        # slots in descending biased score
        zs = z[t, r["idx"][t]]
        assert np.all(np.diff(zs) <= 0)


@SETTINGS
@given(routing_case())
def test_gates_normalised_proportional_and_bias_free(case):
    x, w, b, k = case
    r = O.route(x, w, b, k)
    g = r["gates"]
    assert np.allclose(g.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    sel = np.take_along_axis(r["s"], r["idx"], axis=1)
    assert np.allclose(g * sel.sum(axis=1, keepdims=True), sel, rtol=1e-12, atol=0)
    # a bias shift common to every expert changes neither the selection nor
    # the gates; the bias never enters the gate values
    r2 = O.route(x, w, b + 0.25, k)
    assert np.array_equal(r2["idx"], r["idx"]) and np.allclose(r2["gates"], g, rtol=0, atol=0)


@SETTINGS
@given(routing_case(), st.integers(1, 6), st.integers(0, 2**31 - 1))
def test_dense_equals_sparse(case, h, seed):
    x, w, b, k = case
    rng = np.random.default_rng(seed)
    d, E = x.shape[1], w.shape[0]
    ex = (rng.normal(size=(E, h, d)), rng.normal(size=(E, h, d)), rng.normal(size=(E, d, h)))
    sh = (rng.normal(size=(h, d)), rng.normal(size=(h, d)), rng.normal(size=(d, h)))
    yd = O.moe_forward_dense(x, w, b, ex, sh, k)["y"]
    ys = O.moe_forward_sparse(x, w, b, ex, sh, k)["y"]
    assert np.allclose(yd, ys, rtol=1e-12, atol=1e-12 * np.abs(yd).max())


@SETTINGS
@given(st.integers(1, 64), st.integers(1, 8), st.integers(0, 2**31 - 1))
def test_bias_step_moves_each_bias_by_at_most_gamma(E, k, seed):
    k = min(k, E)
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 50))
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)])
    load = O.load_counts(idx, E)
    assert load.sum() == T * k
    b = rng.uniform(-1, 1, size=E).astype(np.float32)
    gamma = np.float32(1e-3)
    b2 = O.bias_update(b, load, 1e-3, T * k)
    step = np.abs(b2.astype(np.float64) - b.astype(np.float64))
    # one fp32 step of gamma, rounded once: at most gamma plus half an ulp of
    # the result (which can be larger than b's ulp when |b| is small)
    mag = np.maximum(np.abs(b), np.abs(b2)).astype(np.float32)
    assert np.all(step <= float(gamma) + np.spacing(mag).astype(np.float64))
    over = E * load > T * k
    assert np.all(b2[over] <= b[over]) and np.all(b2[E * load < T * k] >= b[E * load < T * k])
    assert np.array_equal(b2[E * load == T * k], b[E * load == T * k])


@SETTINGS
@given(st.integers(1, 5), st.integers(1, 40), st.integers(-20, 20), st.integers(0, 2**31 - 1))
def test_e4m3_rows_within_the_format_bound(rows, cols, exp, seed):
    rng = np.random.default_rng(seed)
    a = (rng.normal(size=(rows, cols)) * 2.0 ** exp).astype(np.float32)
    codes, scales, deq = O.quantize_rows_e4m3(a)
    assert codes.shape == a.shape and scales.shape == (rows,)
    amax = np.abs(a).max(axis=1)
    nz = amax > 0
    # the row maximum maps to +-448 (codes 0x7e / 0xfe)
    top = np.abs(a).argmax(axis=1)
    assert set((codes[np.arange(rows), top][nz] & 0x7F).tolist()) <= {0x7E}
    # normal values within 2^-4 relative; subnormal ones within half the
    # subnormal spacing, 2^-10 of the row's scale
    err = np.abs(deq - a)
    normal = np.abs(a) >= 2.0 ** -6 * scales[:, None]
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(a)[normal])
    sub = np.broadcast_to(2.0 ** -10 * scales[:, None].astype(np.float64), a.shape)
    assert np.all(err[~normal] <= sub[~normal] * (1 + 1e-6))
