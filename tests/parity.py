"""Comparison of the CUDA path's outputs with the float64 oracle.

Acceptance rules (the layer's stated tolerances):
* routing: the selected expert SET of every token equals the oracle's; a
  different set is tolerated only where the oracle's k-th vs (k+1)-th biased
  score gap is below 1e-6, and then the GPU's set must itself be a top-k set
  within that tolerance.  Slots must be in descending biased-score order
  (adjacent slots may swap only within 1e-6).
* load counts: exactly bincount(GPU selection), and equal to the oracle's
  counts wherever no tolerated flip occurred.
* updated bias: bit-exact against the oracle fed the GPU's load counts.
* outputs: fp32 workloads rel L2 <= 1e-5; bf16 workloads rel L2 <= 1e-2 and
  max |diff| <= 5e-2 * rms(y_ref), against the oracle evaluated on the
  GPU's (validated) selection.
* gates: fp32 absolute 1e-6 (fp32 workloads) / 1e-5 (bf16 workloads).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O

GAP_TOL = 1e-6
TOL = {
    "f32": dict(rel_l2=1e-5, max_abs_rms=None, gate_atol=1e-6),
    "bf16": dict(rel_l2=1e-2, max_abs_rms=5e-2, gate_atol=1e-5),
}


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def npi(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").numpy().astype(np.int64)


def check_routing(gpu_idx: np.ndarray, gpu_gates: np.ndarray, ref: dict, gate_atol: float,
                  rows=None) -> int:
    """Returns the number of tolerated flips.  ``ref`` is oracle.route(...)."""
    T, k = gpu_idx.shape
    rows = np.arange(T) if rows is None else np.asarray(rows)
    z, s = ref["z"][rows], ref["s"][rows]
    E = z.shape[1]
    assert ((gpu_idx >= 0) & (gpu_idx < E)).all(), "expert index out of range"
    srt = np.sort(gpu_idx, axis=1)
    assert (np.diff(srt, axis=1) > 0).all() if k > 1 else True, "repeated expert in a token"
    ref_set = np.sort(ref["idx"][rows], axis=1)
    flipped = np.nonzero((srt != ref_set).any(axis=1))[0]
    if len(flipped):
        assert (ref["gap"][rows][flipped] < GAP_TOL).all(), \
            f"selection differs at tokens {rows[flipped][:8]} with gaps {ref['gap'][rows][flipped][:8]}"
    key = np.where(np.isnan(z), -np.inf, z)
    zsel = np.take_along_axis(key, gpu_idx, axis=1)
    rest = key.copy()
    np.put_along_axis(rest, gpu_idx, -np.inf, axis=1)
    if k < E:
        ok = zsel.min(axis=1) >= rest.max(axis=1) - GAP_TOL
        assert ok.all(), f"GPU selection is not a top-k set at tokens {rows[~ok][:8]}"
    if k > 1:
        d = zsel[:, :-1] - zsel[:, 1:]
        assert (np.nan_to_num(d, nan=0.0) >= -GAP_TOL).all(), "slots not in descending score order"
    g_ref = O.gate_weights(s, gpu_idx)
    fin = np.isfinite(g_ref)
    assert np.array_equal(fin, np.isfinite(gpu_gates)), "NaN pattern of gates differs"
    err = np.abs(gpu_gates[fin] - g_ref[fin]).max() if fin.any() else 0.0
    assert err <= gate_atol, f"gate error {err}"
    return len(flipped)


def check_load(gpu_load: np.ndarray, gpu_idx: np.ndarray, ref_idx: np.ndarray, E: int,
               n_flips: int):
    assert np.array_equal(gpu_load, np.bincount(gpu_idx.ravel(), minlength=E))
    if n_flips == 0:
        assert np.array_equal(gpu_load, O.load_counts(ref_idx, E))


def check_output(y_gpu: np.ndarray, y_ref: np.ndarray, dtype: str,
                 max_abs_rms: float | None = None) -> dict:
    tol = dict(TOL[dtype])
    if max_abs_rms is not None:
        tol["max_abs_rms"] = max_abs_rms
    fin = np.isfinite(y_ref).all(axis=1)
    assert np.array_equal(np.isfinite(y_gpu).all(axis=1), fin), "NaN rows differ"
    a, b = y_gpu[fin], y_ref[fin]
    diff = a - b
    nref = np.linalg.norm(b)
    rel = np.linalg.norm(diff) / nref if nref > 0 else np.linalg.norm(diff)
    rms = np.sqrt(np.mean(b * b)) if b.size else 0.0
    mx = np.abs(diff).max() if diff.size else 0.0
    assert rel <= tol["rel_l2"], f"rel L2 {rel:.3e} > {tol['rel_l2']}"
    if tol["max_abs_rms"] is not None:
        assert mx <= tol["max_abs_rms"] * rms, f"max abs {mx:.3e} > {tol['max_abs_rms']} * rms {rms:.3e}"
    return {"rel_l2": float(rel), "max_abs": float(mx), "rms": float(rms)}
