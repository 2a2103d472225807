"""MoeLayer's argument checks: a tensor whose data pointer reaches the library
must have exactly the shape, dtype and device the call reads, and be
contiguous; anything else raises before a launch (host-side, no GPU)."""
import pytest
import torch

from sparse_moe_layer_fwd_b300 import layer as L
from sparse_moe_layer_fwd_b300.layer import MoeLayer

CPU = torch.device("cpu")


def test_exact_tensor_passes():
    L._check("x", torch.zeros(4, 8, dtype=torch.bfloat16), (4, 8), torch.bfloat16, CPU)
    L._check("x", torch.zeros(0, 8), (0, 8), torch.float32, CPU)


@pytest.mark.parametrize("t,why", [
    (torch.zeros(4, 9, dtype=torch.bfloat16), "shape"),
    (torch.zeros(3, 8, dtype=torch.bfloat16), "shape"),
    (torch.zeros(32, dtype=torch.bfloat16), "shape"),
    (torch.zeros(4, 8, dtype=torch.float32), "dtype"),
    (torch.zeros(8, 4, dtype=torch.bfloat16).t(), "contiguous"),
    (torch.zeros(4, 16, dtype=torch.bfloat16)[:, ::2], "contiguous"),
])
def test_mismatch_raises(t, why):
    with pytest.raises(ValueError, match=why if why == "contiguous" else "expected"):
        L._check("x", t, (4, 8), torch.bfloat16, CPU)


def test_wrong_device_raises():
    t = torch.empty(4, 8, dtype=torch.bfloat16, device="meta")
    with pytest.raises(ValueError, match="on cpu"):
        L._check("x", t, (4, 8), torch.bfloat16, CPU)


def test_not_a_tensor_raises():
    with pytest.raises(TypeError):
        L._check("x", 12345, (4, 8), torch.bfloat16, CPU)


def test_layer_refuses_host_weights():
    E, d = 8, 64
    with pytest.raises(ValueError, match="CUDA"):
        MoeLayer(torch.zeros(E, d), torch.zeros(E), None, None, None, None, None, None,
                 T=4, k=2, dtype="bf16", flags=0)
