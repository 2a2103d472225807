"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic, so both the CUDA path and the float64 oracle can be fed
from it.  Every workload is named by what it is, with its sizes:

=================  =====  ====  ====  ===  ==  =====  ====  ======================
name               T      d     h     E    k   dtype  seed  notes
=================  =====  ====  ====  ===  ==  =====  ====  ======================
tiny_fp32          256    256   128   16   4   f32    0     b ~ U(-0.01, 0.01)
mini_bf16          8192   384   384   16   4   bf16   1     b = 0
bias_dynamics      256    256   128   16   4   f32    2     200 route+update steps
v3_prefill         8192   7168  2048  256  8   bf16   3     b ~ U(-0.01, 0.01)
v3_decode          128    7168  2048  256  8   bf16   4     b = 0, balanced
v3_decode_zipf     128    7168  2048  256  8   bf16   4     Zipf(1.2) router skew
v3_prefill_32exp.  1024   7168  2048  32   8   bf16   3     profiling-size prefill
v3_decode_32exp.   16     7168  2048  32   8   bf16   4     profiling-size decode
=================  =====  ====  ====  ===  ==  =====  ====  ======================

Distributions: x ~ N(0,1); W_gate, W_up ~ N(0, 1/d); W_down ~ N(0, 1/h);
router W_r ~ N(0, 1/d) in fp32.  bf16 tensors are drawn in fp32 and rounded to
nearest-even bf16; the oracle reads back the rounded values.

Router skew (bias_dynamics, v3_decode_zipf) is put into the inputs, not into
the method: the last input feature is the constant 1 (x[:, d-1] = 1) and the
router's last column carries a per-expert offset c_e (W_r[e, d-1] = c_e), so
every token's router logit for expert e is shifted by c_e.  bias_dynamics
draws c_e ~ N(0, 1); v3_decode_zipf uses c_e = -1.2 * ln(r_e) with r a seeded
permutation of 1..E, i.e. logit offsets proportional to the log of Zipf(1.2)
weights.

Draw order for one workload: x, W_r, (skew offsets), b, then per routed expert
W_gate, W_up, W_down, then the shared expert's W_gate, W_up, W_down.  Small
workloads are drawn with a CPU ``torch.Generator`` (identical on every
machine); the DeepSeek-V3-sized ones are drawn on the GPU with a CUDA
generator (22.5 GB of weights) and the oracle reads back the bytes it needs.
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    h: int
    E: int
    k: int
    dtype: str          # "f32" or "bf16"
    seed: int
    bias: str = "zero"  # "zero" or "uniform"
    skew: str = "none"  # "none", "normal" or "zipf"
    steps: int = 1
    route_only: bool = False

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def weight_bytes(self) -> int:
        el = 4 if self.dtype == "f32" else 2
        return (self.E + 1) * 3 * self.h * self.d * el

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_fp32", 256, 256, 128, 16, 4, "f32", 0, bias="uniform"),
        Workload("mini_bf16", 8192, 384, 384, 16, 4, "bf16", 1, bias="zero"),
        Workload("bias_dynamics", 256, 256, 128, 16, 4, "f32", 2, bias="zero",
                 skew="normal", steps=200, route_only=True),
        # the "small" configuration of the JAX re-creation: 8 routed experts,
        # top-2, 128-token context (32 sequences); width as the mini model
        Workload("small_bf16", 4096, 384, 384, 8, 2, "bf16", 5, bias="uniform"),
        Workload("v3_prefill", 8192, 7168, 2048, 256, 8, "bf16", 3, bias="uniform"),
        Workload("v3_decode", 128, 7168, 2048, 256, 8, "bf16", 4, bias="zero"),
        Workload("v3_decode_zipf", 128, 7168, 2048, 256, 8, "bf16", 4, bias="zero",
                 skew="zipf"),
        # V3 expert shapes with 32 experts and ~256 tokens per expert: the
        # prefill GEMM regime on 2.9 GB of weights, for profiler captures
        Workload("v3_prefill_32experts", 1024, 7168, 2048, 32, 8, "bf16", 3, bias="uniform"),
        # the decode regime (about 4 tokens per expert) on the same 32
        # experts' weights, for profiler captures of the decode GEMMs
        Workload("v3_decode_32experts", 16, 7168, 2048, 32, 8, "bf16", 4, bias="zero"),
        # V3 prefill's token volume (8192 tokens, top-8, 940 MB of permuted
        # rows, more than L2 holds) on 16 experts' weights (1.5 GB): the
        # dispatch and combine at full size with a few GB on the device, for
        # profiler captures of those kernels
        Workload("v3_prefill_16experts", 8192, 7168, 2048, 16, 8, "bf16", 3, bias="uniform"),
    ]
}


def _gen(seed: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, gen, device, dtype):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def draw_x(wl: Workload, gen: torch.Generator, device: str) -> torch.Tensor:
    """One batch of tokens x [T, d] (constant last feature under skew)."""
    x = _normal((wl.T, wl.d), 1.0, gen, device, wl.torch_dtype)
    if wl.skew != "none":
        x[:, wl.d - 1] = 1.0
    return x


def _skew_offsets(wl: Workload, gen: torch.Generator, device: str) -> torch.Tensor:
    if wl.skew == "normal":
        return torch.randn((wl.E,), generator=gen, device=device, dtype=torch.float32)
    if wl.skew == "zipf":
        r = torch.randperm(wl.E, generator=gen, device=device).to(torch.float64) + 1.0
        return (-1.2 * torch.log(r)).to(torch.float32)
    raise ValueError(wl.skew)


def make_inputs(wl: Workload, device: str = "cpu", gen_device: str | None = None,
                experts: bool = True) -> dict:
    """All inputs of one workload as torch tensors on ``device``.

    Keys: x [T,d], w_router [E,d] f32, bias [E] f32, w_gate [E,h,d],
    w_up [E,h,d], w_down [E,d,h], sh_gate [h,d], sh_up [h,d], sh_down [d,h],
    and "gen" (the generator, positioned after the draws, which
    ``next_x`` continues for multi-step workloads).  With experts=False only
    the routing inputs are drawn (the expert weights come last in the draw
    order, so x, W_r and b are the same either way).
    """
    if gen_device is None:
        gen_device = "cpu" if wl.weight_bytes < (1 << 28) else device
    gen = _gen(wl.seed, gen_device)
    dt = wl.torch_dtype
    x = draw_x(wl, gen, gen_device)
    w_router = _normal((wl.E, wl.d), 1.0 / math.sqrt(wl.d), gen, gen_device, torch.float32)
    if wl.skew != "none":
        w_router[:, wl.d - 1] = _skew_offsets(wl, gen, gen_device)
    if wl.bias == "uniform":
        bias = (torch.rand((wl.E,), generator=gen, device=gen_device) * 0.02 - 0.01)
    else:
        bias = torch.zeros((wl.E,), device=gen_device)
    bias = bias.to(torch.float32)

    out = {
        "x": x.to(device),
        "w_router": w_router.to(device),
        "bias": bias.to(device),
        "gen": gen,
        "gen_device": gen_device,
    }
    if not experts:
        return out
    w_gate = torch.empty((wl.E, wl.h, wl.d), dtype=dt, device=device)
    w_up = torch.empty((wl.E, wl.h, wl.d), dtype=dt, device=device)
    w_down = torch.empty((wl.E, wl.d, wl.h), dtype=dt, device=device)
    sg, sd = 1.0 / math.sqrt(wl.d), 1.0 / math.sqrt(wl.h)
    for e in range(wl.E):
        w_gate[e] = _normal((wl.h, wl.d), sg, gen, gen_device, dt).to(device)
        w_up[e] = _normal((wl.h, wl.d), sg, gen, gen_device, dt).to(device)
        w_down[e] = _normal((wl.d, wl.h), sd, gen, gen_device, dt).to(device)
    out["w_gate"], out["w_up"], out["w_down"] = w_gate, w_up, w_down
    out["sh_gate"] = _normal((wl.h, wl.d), sg, gen, gen_device, dt).to(device)
    out["sh_up"] = _normal((wl.h, wl.d), sg, gen, gen_device, dt).to(device)
    out["sh_down"] = _normal((wl.d, wl.h), sd, gen, gen_device, dt).to(device)
    return out


def next_x(wl: Workload, inputs: dict, device: str) -> torch.Tensor:
    """A fresh token batch from the workload's generator stream (the
    bias-dynamics run draws one per step)."""
    return draw_x(wl, inputs["gen"], inputs["gen_device"]).to(device)


def custom(T, d, h, E, k, dtype="bf16", seed=0, bias="uniform", skew="none",
           name=None) -> Workload:
    """A workload with arbitrary sizes (edge cases, ragged tails)."""
    return Workload(name or f"custom_T{T}_d{d}_h{h}_E{E}_k{k}_{dtype}",
                    T, d, h, E, k, dtype, seed, bias=bias, skew=skew)


def fingerprint(inputs: dict, weight_row_stride: int = 64) -> dict:
    """SHA-256 of a workload's inputs as they sit in memory: every byte of x,
    W_r and b, and every ``weight_row_stride``-th row of each expert weight
    matrix (the V3 weights are 22.5 GB; a strided sample keeps this fast).
    Returns {"sha256": hex digest, "scope": what was hashed}."""
    import hashlib
    h = hashlib.sha256()

    def add(t):
        h.update(t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes())

    for name in ("x", "w_router", "bias"):
        add(inputs[name])
    have_w = "w_gate" in inputs
    if have_w:
        for name in ("w_gate", "w_up", "w_down", "sh_gate", "sh_up", "sh_down"):
            w = inputs[name]
            add(w.reshape(-1, w.shape[-1])[::weight_row_stride])
    scope = "x, W_r, b in full" + (
        f"; every {weight_row_stride}th row of each expert weight matrix" if have_w else "")
    return {"sha256": h.hexdigest(), "scope": scope}
