"""The expert epilogue's silu (the gate/up products' SwiGLU) against
float64: z / (1 + e^-z) on a grid over every range the pre-activations take,
plus the special values."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_fwd_b300 import moe as M

pytestmark = pytest.mark.gpu


def _silu64(z):
    with np.errstate(over="ignore", invalid="ignore"):
        return z / (1.0 + np.exp(-z))


def test_silu_accuracy():
    z = np.concatenate([np.linspace(-20.0, 20.0, 400001), np.linspace(-87.0, 88.0, 100001),
                        -np.geomspace(1e-30, 86.9, 20001), np.geomspace(1e-30, 1e4, 20001)])
    zt = torch.from_numpy(z.astype(np.float32)).cuda()
    out = torch.empty_like(zt)
    M.moe_selftest_silu(zt, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref = _silu64(zt.cpu().numpy().astype(np.float64))
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-300)
    small = np.abs(z) <= 20
    # the fast exponential's argument rounding grows with |z|
    assert rel[small].max() < 2e-6, float(rel[small].max())
    assert rel.max() < 2e-5, float(rel.max())


def test_silu_special_values():
    z = torch.tensor([0.0, -0.0, 1e-30, -1e-30, 88.0, -87.5, -200.0, float("inf"),
                      float("-inf"), float("nan")], device="cuda")
    out = torch.empty_like(z)
    M.moe_selftest_silu(z, out)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert o[0] == 0 and o[1] == 0
    assert abs(o[2] - 0.5e-30) <= 1e-36 and abs(o[3] + 0.5e-30) <= 1e-36
    assert o[4] == np.float32(88.0)
    assert o[5] == 0 and np.signbit(o[5]) and o[6] == 0
    assert o[7] == np.inf
    assert np.isnan(o[8]) and np.isnan(o[9])
