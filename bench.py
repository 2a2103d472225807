"""MoE-layer forward throughput on B300 (tokens/s) and roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one forward pass of the whole layer (router, top-k, load counts,
dispatch, both expert GEMMs with the shared expert, combine) over one batch
of the workload, through the C ABI of libmoe.so.  Inputs are synthetic and
seeded (sparse_moe_layer_fwd_b300.inputs) and resident in device memory when
the timed region starts.  The default workload is the DeepSeek-V3-shaped
prefill layer (T = 8192, d = 7168, h = 2048, 256 routed experts, top-8, one
shared expert): 22.5 GB of expert weights, far larger than the 126 MB L2, so
no L2 flush is needed between steps.  Workloads whose inputs L2 could hold
(the mini-model layer, the routing-only pass) get a 252 MB write before every
step, outside the per-step CUDA-event spans that then give the time.

Per-phase device times come from CUDA events that the library records on the
launching stream between phases (moe_forward_profiled).  `roofline` is for
the dominant kernel (expert GEMM 1: gate/up + SwiGLU, shared expert
included): algorithmic FLOPs (prefill) or bytes (decode) per launch divided
by its mean event-timed duration, against MEASURED_PEAKS.json.

With N > 1 (torchrun, one process per GPU) every rank runs an independent
replica on its own batch (the layer forward has no cross-replica exchange):
weak scaling, value = all ranks' tokens / the slowest rank's time.

--impl reference times the float64 CPU oracle on the host cores on bounded
samples of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (fwd, bf16) at 1 B300; % of tensor-core or HBM roofline"
def tc_router(wl):
    """The library routes bf16 tokens over 96 experts or more on the tensor
    cores (router weights split into three bf16 terms), else on CUDA cores."""
    return wl.dtype == "bf16" and wl.E >= 96 and wl.T > 0


def kernels_per_step(wl, route_only, fp8=False):
    """Kernels one forward launches: router (weight split + MMA, or FFMA
    logits), top-k, block ranks, scan [, token quantization (fp8), permute,
    GEMM 1, GEMM 2, combine]."""
    n = (2 if tc_router(wl) else 1) + 3
    return n if route_only else n + 4 + int(fp8)

# DRAM traffic of expert GEMM 1 per launch (dram__bytes_read.sum +
# dram__bytes_write.sum).  Counters beyond the kernel time are captured on
# the 32-expert V3-width cases (2.9 GB of weights, one kernel, two launches;
# prefill: 256 tokens per expert, decode: 4) and scaled to a full launch of
# the same regime by the ratio of the two cases' algorithmic bytes (weights
# of the touched experts plus token rows, which the traffic follows); keyed
# to the hash of the GEMM sources at capture time and reported as null once
# those sources change.
NCU_TRAFFIC = {
    # profiles/k_expert_tc2_v3_prefill_32experts_full.md ("DRAM counters of
    # the current sources"): GEMM 1 read + written bytes on that case
    "bf16": {"sha": "dd10e8a46ce0f545", "case": "v3_prefill_32experts",
             "bytes": 2.176548352e9 + 0.033965824e9},
    ":fp8blk": {"sha": "dd10e8a46ce0f545", "case": "v3_prefill_32experts",
                "bytes": 1.043218432e9 + 0.018627072e9},
    # profiles/k_expert_tc_v3_decode_32experts_full.md: the one-SM kernel
    "bf16:decode": {"sha": "dd10e8a46ce0f545", "case": "v3_decode_32experts",
                    "bytes": 1.939902e9 + 0.003503104e9},
}


def _traffic_for(wl, load, fp8=False, fp8_blk=False):
    """GEMM 1's DRAM bytes per launch of this workload, from the capture of
    its regime: null if none matches the current sources, or if the
    workload's tokens per expert are more than twice or less than half the
    captured case's (the share of weight rows re-read from L2 would differ)."""
    regime = "" if wl.T * wl.k / wl.E >= 96 else ":decode"
    cap = NCU_TRAFFIC.get((":fp8blk" if fp8_blk else ":fp8" if fp8 else "bf16") + regime)
    if not cap or cap.get("sha") != _kernel_sha():
        return None
    small = I_WORKLOADS()[cap["case"]]
    ratio = (wl.T * wl.k / wl.E) / (small.T * small.k / small.E)
    if not 0.5 <= ratio <= 2.0:
        return None
    return _scaled_traffic(cap, wl, load, fp8, fp8_blk)


def _scaled_traffic(cap, wl, load, fp8, fp8_blk):
    """A small-case capture scaled to this workload's launch."""
    if not cap:
        return None
    small = I_WORKLOADS()[cap["case"]]
    sload = np.full(small.E, small.T * small.k // small.E)
    return cap["bytes"] * (_algorithmic(wl, load, fp8, fp8_blk)[2] /
                           _algorithmic(small, sload, fp8, fp8_blk)[2])


def I_WORKLOADS():
    from sparse_moe_layer_fwd_b300 import inputs as I
    return I.WORKLOADS


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "sm_max_mhz": d.get("sm_max_mhz", 2032.0), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "sm_max_mhz": 2032.0, "source": "fallback"}


def _code_lines(text):
    """Source lines with // comments and blank lines removed."""
    out = []
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            out.append(code)
    return "\n".join(out)


def _kernel_sha(read=None):
    """SHA-256 (16 hex digits) of the expert GEMM sources, comments ignored."""
    if read is None:
        def read(f):
            with open(os.path.join(ROOT, "sparse_moe_layer_fwd_b300", "csrc", f)) as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in ("ptx.cuh", "experts_tc.cuh", "experts_tc2.cuh", "moe.cu"):
        h.update(_code_lines(read(f)).encode())
    return h.hexdigest()[:16]


SMI_LAG_S = 0.15


def _kernel_clocks(M, reset_first=False):
    """Mean SM clock (MHz) of each tensor-core kernel class since the last
    reset, from the kernels' own cycle and %globaltimer counters."""
    rec = M.moe_sm_clock_record(reset=reset_first)
    return {n: round(v["mhz"], 1) for n, v in rec.items() if v["mhz"]}


def _note_inband_cap(clocks):
    """Mark a window whose tensor-core kernels ran more than 5% below the
    maximum SM clock by their own counters, whatever nvidia-smi showed."""
    mhz = [v for v in (clocks.get("kernel_sm_mhz") or {}).values() if v]
    if mhz and clocks.get("sm_max_mhz") and min(mhz) < 0.95 * clocks["sm_max_mhz"]:
        clocks["inband_below_max"] = (f"tensor-core kernels at {min(mhz):.0f}-{max(mhz):.0f} MHz "
                                      f"by their own cycle counters (board power cap)")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a window."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                except ValueError:
                    continue
                rows.append((ts, parts))
        os.unlink(self.file.name)
        self.rows = rows
        # nvidia-smi reports a clock change about 0.1 s after the kernels see
        # it (a power-capped V3 prefill run: the step times rose at 58 ms of
        # load, the first sample showing the lower clock came at 173 ms), so
        # the window reaches SMI_LAG_S past the end of the timed region
        inside = ([p for ts, p in rows if t0 - 0.05 <= ts <= t1 + SMI_LAG_S]
                  or [p for _, p in rows[-5:]])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm = []
        mx = None
        for p in inside:
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                pass
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(inside)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(elapsed_ms: float, tokens_per_rank: int, world_size: int, device="cpu"):
    """Whole-job throughput of independent replicas: the slowest rank's time
    (max over ranks) and all ranks' tokens.  Returns (max_ms, tokens/s)."""
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    if world_size > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    max_ms = float(t.item())
    return max_ms, world_size * tokens_per_rank / (max_ms / 1e3)


L2_BYTES = 126 * 2**20


def _working_set_bytes(wl, route_only):
    """Bytes one step reads from its resident inputs: tokens and router, and
    (full layer) every expert's weights."""
    el = 2 if wl.dtype == "bf16" else 4
    b = wl.T * wl.d * el + wl.E * wl.d * 4
    if not route_only:
        b += (wl.E + 1) * 3 * wl.d * wl.h * el
    return b


def _algorithmic(wl, load, fp8=False, fp8_blk=False):
    """FLOPs and bytes of the two expert GEMMs for one launch each (fp8: a
    GEMM reads one-byte codes of weights and tokens, plus row scales, or
    one exponent byte per 128 x 128 weight block and per 1 x 128 token or
    hidden block)."""
    TK, T, d, h = wl.T * wl.k, wl.T, wl.d, wl.h
    rows = TK + T
    fl1 = 4.0 * rows * d * h
    fl2 = 2.0 * rows * d * h
    touched = int((load > 0).sum()) + 1  # + shared expert
    if fp8_blk:
        by1 = touched * 2 * h * d * (1 + 1 / 16384) + rows * d * (1 + 1 / 128) + rows * h * (1 + 1 / 128)
        by2 = touched * d * h * (1 + 1 / 16384) + rows * h * (1 + 1 / 128) + TK * d * 2 + T * d * 4
        return fl1, fl2, by1, by2, touched - 1
    if fp8:
        by1 = touched * 2 * h * (d + 4) + rows * (d + 4) + rows * h * 2
    else:
        by1 = touched * 2 * h * d * 2 + rows * d * 2 + rows * h * 2
    by2 = touched * d * h * 2 + rows * h * 2 + TK * d * 2 + T * d * 4
    return fl1, fl2, by1, by2, touched - 1


def cpu_oracle_sample(wl, inp, n_tokens, seed=0):
    """Run the float64 oracle on n_tokens tokens of the workload: routing,
    shared expert and each token's k routed experts, streaming expert
    weights from device memory one at a time.  Returns seconds."""
    from oracle import moe_oracle as O
    rows = np.sort(np.random.default_rng(seed).choice(wl.T, n_tokens, replace=False))
    f64 = lambda t: t.detach().to("cpu").to(torch.float64).numpy()  # noqa: E731
    x = f64(inp["x"][torch.from_numpy(rows).to(inp["x"].device)])
    wr, b = f64(inp["w_router"]), f64(inp["bias"])
    t0 = time.perf_counter()
    r = O.route(x, wr, b, wl.k)
    sh = (f64(inp["sh_gate"]), f64(inp["sh_up"]), f64(inp["sh_down"]))
    O.expert_output_rows(x, r["idx"], r["gates"],
                         lambda e: (f64(inp["w_gate"][e]), f64(inp["w_up"][e]), f64(inp["w_down"][e])),
                         sh)
    return time.perf_counter() - t0


def cpu_baseline_layer(wl, inp, n_rows=512, seed=0):
    """The float64 oracle on the host cores, as the layer's measurement plan
    asks: routing of all T tokens, then the outputs of n_rows seeded rows
    (all rows when T <= n_rows), experts streamed from device memory one at
    a time.  Returns the cpu_baseline object: value = sampled rows per second
    of the whole layer (their share of the routing time plus their outputs)."""
    from oracle import moe_oracle as O
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    f64 = lambda t: t.detach().to("cpu").to(torch.float64).numpy()  # noqa: E731
    x = f64(inp["x"])
    wr, b = f64(inp["w_router"]), f64(inp["bias"])
    t0 = time.perf_counter()
    r = O.route(x, wr, b, wl.k)
    t_route = time.perf_counter() - t0
    n = min(n_rows, wl.T)
    rows = (np.sort(np.random.default_rng(seed).choice(wl.T, n, replace=False))
            if n < wl.T else np.arange(wl.T))
    sh_dev = (inp["sh_gate"], inp["sh_up"], inp["sh_down"])
    t1 = time.perf_counter()
    sh = tuple(f64(w) for w in sh_dev)
    O.expert_output_rows(x[rows], r["idx"][rows], r["gates"][rows],
                         lambda e: (f64(inp["w_gate"][e]), f64(inp["w_up"][e]), f64(inp["w_down"][e])),
                         sh)
    t_out = time.perf_counter() - t1
    per_row = t_route / wl.T + t_out / n
    return {"value": 1.0 / per_row, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "routing_tokens_per_s": wl.T / t_route, "output_rows_per_s": n / t_out,
            "sample": (f"float64 oracle on {wl.name}: routing of all {wl.T} tokens, then the "
                       f"outputs of {n} seeded rows (shared expert and their {wl.k} routed "
                       f"experts, weights streamed from device memory one expert at a time); "
                       f"value = 1 / (routing time per token + output time per row)")}


def run_reference(args, wl):
    ws, rank, local = _dist()
    if rank != 0:
        return
    from sparse_moe_layer_fwd_b300 import inputs as I
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = I.make_inputs(wl, device=dev)
    n = args.ref_tokens
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    for i in range(args.warmup):
        cpu_oracle_sample(wl, inp, n, seed=1000 + i)
    times = [cpu_oracle_sample(wl, inp, n, seed=i) for i in range(args.steps)]
    total = sum(times)
    value = n * args.steps / total
    sample = (f"{n} tokens per step of {wl.name}: float64 routing of those tokens, shared "
              f"expert and their {wl.k} routed experts, expert weights streamed from device memory")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "h": wl.h, "E": wl.E, "k": wl.k},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _timed_forward(M, layer, x, stream, steps, flush, sampler_index=None, trace=None):
    """`steps` forward passes back to back on `stream` with per-phase events
    (moe_forward_profiled); flush: a buffer written before every step
    (outside the per-step spans).  Returns (loop ms, per-step ms list, mean
    phase ms array, clocks or None).  trace: a dict that receives each
    step's start (ms from the first) and phase times, and the raw clock
    samples (s from the start)."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(M.N_PHASE_EVENTS)]
          for _ in range(steps)]
    for row in ev:  # torch creates the CUDA event on its first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(sampler_index) if sampler_index is not None else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    M.moe_sm_clock_record(reset=True)
    t_host0 = time.time()
    start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        M.moe_forward_profiled(layer.desc, x, layer.w_router, layer.bias, layer.experts,
                               layer.shared, layer.y, layer.topk_idx, layer.gates,
                               layer.load_counts, layer.workspace, layer.ws_bytes, stream, ev[i])
    end.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    clocks = sampler.stop(t_host0, t_host1) if sampler else None
    if clocks is not None:
        clocks["kernel_sm_mhz"] = _kernel_clocks(M)
        _note_inband_cap(clocks)
    if M.moe_last_error() != M.MOE_OK:
        raise RuntimeError("device error word set during the timed region")
    per_step = [ev[i][0].elapsed_time(ev[i][-1]) for i in range(steps)]
    loop_ms = start.elapsed_time(end) if flush is None else sum(per_step)
    phase_ms = np.zeros(len(M.PHASES))
    for i in range(steps):
        for p in range(len(M.PHASES)):
            phase_ms[p] += ev[i][p].elapsed_time(ev[i][p + 1])
    if trace is not None:
        trace["phases"] = list(M.PHASES)
        trace["steps"] = [[start.elapsed_time(ev[i][0])] +
                          [ev[i][p].elapsed_time(ev[i][p + 1]) for p in range(len(M.PHASES))]
                          for i in range(steps)]
        if sampler is not None:
            trace["smi_fields"] = ClockSampler.FIELDS
            trace["smi"] = [[round(ts - t_host0, 3)] + p[1:] for ts, p in sampler.rows]
    return loop_ms, per_step, phase_ms / steps, clocks


# Dense bf16 tensor-core rate per SM clock: 4096 multiply-adds per clock
# per SM (a stand-alone CTA-pair MMA loop reaches it for N >= 128; the
# nominal 2.25 PFLOP/s dense bf16 is this rate at about 1.86 GHz), 148 SMs.
BF16_TFLOPS_PER_MHZ = 2 * 4096 * 148 / 1e6


def _tensor_peak(peaks, clocks, fp8=False, slot="gate_up"):
    """Denominator of a tensor-core roofline: the measured burst bf16 figure
    (times the nominal fp8/bf16 ratio 2 for e4m3 products).  Beside it, not
    in its place: the tensor pipe's peak at the clock the kernel ran at --
    its in-band mean SM clock over the timed region (kernel cycles / kernel
    ns) times the per-clock rate.  Back-to-back V3 prefill steps reach the
    board's power cap within about 60 ms, after which the SM clock settles
    near 1.1-1.3 GHz; the burst figure itself (a single 8192^3 product) implies
    at least 1808.6 / 1.212 = 1492 MHz."""
    mult = 2.0 if fp8 else 1.0
    peak = mult * peaks["bf16_tflops"]
    kind = (f"{'2 x ' if fp8 else ''}{peaks['source']} bf16 burst"
            + (" (nominal fp8/bf16 ratio)" if fp8 else ""))
    at_clock = None
    mhz = ((clocks or {}).get("kernel_sm_mhz") or {}).get(slot)
    if mhz:
        at_clock = {"sm_mhz": mhz, "peak_tflops": mult * BF16_TFLOPS_PER_MHZ * mhz}
    return peak, kind, at_clock


def _decode_line(M, I, MoeLayer, name, args, peaks, local):
    """One V3 decode workload (T = 128) timed as the main line is, reported
    against the HBM roofline: the layer's algorithmic bytes (touched routed
    experts + the shared expert, all three matrices; router weights; tokens
    in and out) per step over the step time, and expert GEMM 1 alone."""
    wl = I.WORKLOADS[name]
    inp = I.make_inputs(wl, device="cuda")
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype)
    stream = torch.cuda.current_stream()
    x = inp["x"]
    for _ in range(args.warmup):
        layer.forward(x, stream)
    torch.cuda.synchronize()
    if M.moe_last_error() != M.MOE_OK:
        raise RuntimeError("device error word set during warm-up")
    load = layer.load_counts.cpu().numpy()
    loop_ms, per_step, phase_ms, clocks = _timed_forward(M, layer, x, stream, args.steps, None,
                                                         local)
    touched = int((load > 0).sum())
    expert_bytes = 3 * wl.d * wl.h * 2
    layer_bytes = ((touched + 1) * expert_bytes + wl.E * wl.d * 4 + 2 * wl.T * wl.d * 2)
    ms = loop_ms / args.steps
    fl1, fl2, by1, by2, _ = _algorithmic(wl, load)
    g1 = by1 / (phase_ms[2] / 1e3) / 1e9
    layer_gbs = layer_bytes / (ms / 1e3) / 1e9
    out = {"workload": name, "T": wl.T, "value": wl.T / (ms / 1e3), "unit": "tokens/s",
           "ms_per_step": ms, "ms_per_step_median": statistics.median(per_step),
           "touched_experts": touched,
           "layer_bytes_per_step": layer_bytes, "layer_gbs": layer_gbs,
           "frac": layer_gbs / peaks["hbm_gbs"],
           "gemm1_gbs": g1, "gemm1_frac": g1 / peaks["hbm_gbs"],
           "gemm1_traffic": _traffic_for(wl, load), "gemm1_bytes": by1,
           "peak": peaks["hbm_gbs"], "peak_kind": f"{peaks['source']} HBM copy bandwidth",
           "phase_ms": {n: float(v) for n, v in zip(M.PHASES, phase_ms)},
           "gpu_launches": kernels_per_step(wl, False) * args.steps,
           "clocks": clocks}
    del layer, inp
    torch.cuda.empty_cache()
    return out


def run_ours(args, wl):
    from sparse_moe_layer_fwd_b300 import inputs as I
    from sparse_moe_layer_fwd_b300 import moe as M
    from sparse_moe_layer_fwd_b300.layer import MoeLayer

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    wl_rank = wl.with_(seed=wl.seed + 1000 * rank) if ws > 1 else wl
    route_only = args.route_only or wl.route_only
    inp = I.make_inputs(wl_rank, device="cuda", experts=not route_only)
    fp8 = bool(args.fp8) and not route_only
    fp8_blk = fp8 and args.fp8 == "block"
    base_flags = (M.MOE_FP8_BLOCK if fp8_blk else M.MOE_FP8_GATE_UP) if fp8 else 0
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_ROUTE_ONLY if route_only else base_flags)
    stream = torch.cuda.current_stream()
    x = inp["x"]
    fingerprint = I.fingerprint(inp) if rank == 0 else None

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    # warm-up
    for _ in range(args.warmup):
        layer.forward(x, stream)
    torch.cuda.synchronize()
    if M.moe_last_error() != M.MOE_OK:
        raise RuntimeError("device error word set during warm-up")
    load = layer.load_counts.cpu().numpy()

    # A working set that L2 could hold is evicted before every timed step by
    # writing a buffer of twice the L2 size (outside the per-step event
    # spans, which then give the time); larger ones stream from HBM anyway.
    ws_bytes = _working_set_bytes(wl, route_only)
    flush = (torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
             if ws_bytes < 4 * L2_BYTES else None)
    l2_note = (f"L2 flushed before each step ({2 * L2_BYTES >> 20} MB write outside the timed "
               f"spans; working set {ws_bytes / 1e6:.0f} MB)" if flush is not None else
               f"inputs larger than L2 ({ws_bytes / 1e9:.1f} GB read per step)")

    # timed region: per-step phase events on the launching stream
    barrier()
    trace = {} if args.trace and rank == 0 else None
    local_ms, per_step, phase_ms, clocks = _timed_forward(
        M, layer, x, stream, args.steps, flush, local if rank == 0 else None, trace)
    if trace is not None:
        with open(args.trace, "w") as f:
            json.dump({"workload": wl.name, "kernel_sm_mhz": (clocks or {}).get("kernel_sm_mhz"),
                       **trace}, f)
    barrier()
    elapsed_ms, value = aggregate(local_ms, wl.T * args.steps, ws, "cuda")
    median_ms = statistics.median(per_step)

    # optional: the same steps replayed from one captured CUDA graph (no host
    # launches; the step is timed around each replay, L2 flushed as above)
    graph = None
    if args.graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.forward(x, torch.cuda.current_stream())
        torch.cuda.synchronize()
        ge = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            ge[i][0].record(stream)
            g.replay()
            ge[i][1].record(stream)
        torch.cuda.synchronize()
        if M.moe_last_error() != M.MOE_OK:
            raise RuntimeError("device error word set during the graph replays")
        g_ms, g_value = aggregate(sum(a.elapsed_time(b) for a, b in ge), wl.T * args.steps, ws,
                                  "cuda")
        graph = {"value": g_value, "unit": "tokens/s", "ms_per_step": g_ms / args.steps}
        del g

    # end to end through the host-buffer entry point (pinned x in, y out).
    # Inputs larger than L2: two layers on two streams, as a serving loop
    # would run them, so one step's copies overlap the other's kernels (each
    # step still copies its own x in and its own y out inside the timed
    # region).  Working sets L2 could hold: one stream, L2 flushed per step.
    e2e = None
    if not args.no_e2e:
        nlay = 1 if flush is not None else 2
        flags_e = M.MOE_ROUTE_ONLY if route_only else base_flags
        hls = [MoeLayer.from_inputs(inp, wl.k, wl.dtype, flags_e, host_io=True)
               for _ in range(nlay)]
        streams = [stream] + [torch.cuda.Stream() for _ in range(nlay - 1)]
        x_hosts = [x.cpu().pin_memory() for _ in range(nlay)]
        y_hosts = [torch.empty_like(x_hosts[0]).pin_memory() for _ in range(nlay)]
        for j in range(nlay):
            for _ in range(2):
                hls[j].forward_host_io(x_hosts[j], y_hosts[j], streams[j])
        torch.cuda.synchronize()
        barrier()
        if flush is None:
            s0 = torch.cuda.Event(enable_timing=True)
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(nlay)]
            s0.record(streams[0])
            for j in range(1, nlay):
                streams[j].wait_event(s0)
            for i in range(args.steps):
                j = i % nlay
                hls[j].forward_host_io(x_hosts[j], y_hosts[j], streams[j])
            for j in range(nlay):
                ends[j].record(streams[j])
            torch.cuda.synchronize()
            e_local = max(s0.elapsed_time(e) for e in ends)
        else:
            s2 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            e2 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            for i in range(args.steps):
                flush.zero_()
                s2[i].record(stream)
                hls[0].forward_host_io(x_hosts[0], y_hosts[0], stream)
                e2[i].record(stream)
            torch.cuda.synchronize()
            e_local = sum(s2[i].elapsed_time(e2[i]) for i in range(args.steps))
        if M.moe_last_error() != M.MOE_OK:
            raise RuntimeError("device error word set during the end-to-end run")
        e2e_ms, e2e_value = aggregate(e_local, wl.T * args.steps, ws, "cuda")
        nb = x_hosts[0].numel() * x_hosts[0].element_size()
        e2e = {"value": e2e_value, "unit": "tokens/s",
               "h2d_bytes_per_step": nb, "d2h_bytes_per_step": 0 if route_only else nb,
               "ms_per_step": e2e_ms / args.steps, "streams": nlay}
        del hls

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peaks = _peaks()
    meta = {"torch": torch.__version__, "inputs": fingerprint}
    if route_only:
        rflops = 2.0 * wl.T * wl.E * wl.d
        ach = rflops / (phase_ms[0] / 1e3) / 1e12
        if tc_router(wl):
            # three bf16 MMAs per fp32-exact product: the peak for the
            # algorithmic FLOPs is a third of the dense bf16 peak
            rpeak, rbound = peaks["bf16_tflops"] / 3.0, "tensor"
            rkind = f"{peaks['source']} bf16 burst / 3 (router weights as three bf16 terms)"
            rkernel = "k_router_split + k_router_tc + k_router_topk (router phase)"
        else:
            # fp32 FFMA on CUDA cores: 148 SMs x 128 lanes x 2 FLOP x max clock
            rpeak, rbound = 148 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12, "alu"
            rkind = "148 SMs x 128 FP32 lanes x 2 FLOP x max SM clock"
            rkernel = "k_router_logits (fp32 FFMA) + k_router_topk (router phase)"
        line = {
            "metric": METRIC + " [routing only]", "value": wl.T * args.steps / (elapsed_ms / 1e3),
            "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "ms_per_step_median": median_ms,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 router, bf16 x" if wl.dtype == "bf16" else "f32",
            "data": "synthetic (seeded N(0,1) tokens, N(0,1/d) router)",
            "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k,
                       "route_only": True, "l2": l2_note},
            "roofline": {"bound": rbound, "kernel": rkernel,
                         "achieved": ach, "peak": rpeak, "unit": "TFLOP/s",
                         "frac": ach / rpeak, "traffic": None, "peak_kind": rkind,
                         "flops_per_launch": rflops, "ms_per_launch": phase_ms[0]},
            "phase_ms": {n: float(v) for n, v in zip(M.PHASES, phase_ms)},
            "e2e": e2e, "gpu_launches": kernels_per_step(wl, True) * args.steps,
            **({"cuda_graph": graph} if graph else {}),
            "clocks": clocks, **meta,
        }
        print(json.dumps(line), flush=True)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    fl1, fl2, by1, by2, touched = _algorithmic(wl, load, fp8, fp8_blk)
    g1_s, g2_s = phase_ms[2] / 1e3, phase_ms[3] / 1e3
    prefill_like = wl.T * wl.k / wl.E >= 96
    sha = _kernel_sha()
    traffic = _traffic_for(wl, load, fp8, fp8_blk)  # GEMM 1
    if prefill_like:
        ach = fl1 / g1_s / 1e12
        peak, kind, clk1 = _tensor_peak(peaks, clocks, fp8)
        roof = {"bound": "tensor",
                "kernel": ("k_expert_tc2 (GEMM 1 on e4m3 codes: gate/up + SwiGLU, CTA pairs)"
                           if fp8 else "k_expert_tc2 (GEMM 1: gate/up + SwiGLU, CTA pairs)"),
                "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "traffic": traffic, "peak_kind": kind,
                "flops_per_launch": fl1, "ms_per_launch": phase_ms[2]}
        if clk1 is not None:
            roof["at_kernel_clock"] = {**clk1, "frac": ach / clk1["peak_tflops"]}
        both = (fl1 + fl2) / (g1_s + g2_s) / 1e12
        layer_roof = {"expert_gemms_tflops": both, "frac": both / peak,
                      "gemm2_tflops": fl2 / g2_s / 1e12, "gemm2_frac": fl2 / g2_s / 1e12 / peak,
                      "gemm2_gbs": by2 / g2_s / 1e9}
        _, _, clk2 = _tensor_peak(peaks, clocks, fp8, "down")
        if clk1 is not None and clk2 is not None:
            # both products at their own clocks: FLOPs over what the tensor
            # pipe could do in each product's time at that product's clock
            layer_roof["frac_at_kernel_clock"] = (fl1 + fl2) / 1e12 / (
                g1_s * clk1["peak_tflops"] + g2_s * clk2["peak_tflops"])
            layer_roof["gemm2_frac_at_kernel_clock"] = fl2 / 1e12 / (g2_s * clk2["peak_tflops"])
    else:
        ach = by1 / g1_s / 1e9
        roof = {"bound": "hbm",
                "kernel": ("k_expert_tc2 (GEMM 1 on e4m3 codes, CTA pairs)" if fp8 else
                           "k_expert_tc (GEMM 1: gate/up + SwiGLU, one SM)"),
                "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": traffic,
                "peak_kind": f"{peaks['source']} copy bandwidth",
                "bytes_per_launch": by1, "ms_per_launch": phase_ms[2]}
        both = (by1 + by2) / (g1_s + g2_s) / 1e9
        layer_roof = {"expert_gemms_gbs": both, "frac": both / peaks["hbm_gbs"]}
    layer_roof["touched_experts"] = touched

    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline_layer(wl, inp, n_rows=args.cpu_rows)

    # the V3 decode layer (balanced and Zipf-skewed routing), measured in the
    # same process after the main workload, against the HBM roofline
    decode = None
    if wl.name == "v3_prefill" and not fp8 and not args.no_decode and ws == 1:
        del layer
        inp = None
        torch.cuda.empty_cache()
        decode = [_decode_line(M, I, MoeLayer, n, args, peaks, local)
                  for n in ("v3_decode", "v3_decode_zipf")]

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "ms_per_step_median": median_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 experts (128x128 weight / 1x128 activation block scales)" if fp8_blk else
                  "e4m3 gate/up (per-row scales), bf16 down" if fp8 else "bf16"),
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
        "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "h": wl.h, "E": wl.E, "k": wl.k,
                   "shared_experts": 1, "parallelism": f"replicas x{ws}",
                   "l2": l2_note, **({"fp8": args.fp8} if fp8 else {})},
        "roofline": roof, "roofline_layer": layer_roof,
        "phase_ms": {n: float(v) for n, v in zip(M.PHASES, phase_ms)},
        "cpu_baseline": cpu, "e2e": e2e, **({"cuda_graph": graph} if graph else {}),
        "gpu_launches": kernels_per_step(wl, False, fp8) * args.steps,
        **({"decode": decode} if decode else {}),
        "clocks": clocks, "kernel_sha": sha, **meta,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# Short names of the five benchmark workloads (--config C3 is --workload v3_prefill).
CONFIGS = {"C0": "tiny_fp32", "C1": "mini_bf16", "C2": "bias_dynamics", "C3": "v3_prefill",
           "C4": "v3_decode", "C4z": "v3_decode_zipf"}


def run_train(args, wl):
    """Training step: forward (with the backward's buffers) and backward for
    a fixed output gradient, timed together; reports tokens/s of the step,
    the two phases, and the backward's GEMM FLOPs against the burst bf16
    peak (12 d h FLOP per routed pair or shared-expert token: dH, dX and the
    three weight gradients; the recomputed gate/up products are not counted)."""
    from sparse_moe_layer_fwd_b300 import inputs as I
    from sparse_moe_layer_fwd_b300 import moe as M
    from sparse_moe_layer_fwd_b300.layer import MoeLayer

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    inp = I.make_inputs(wl.with_(seed=wl.seed + 1000 * rank) if ws > 1 else wl, device="cuda")
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype,
                                 M.MOE_TRAINING | (M.MOE_GRAD_BF16 if args.grad_bf16 else 0))
    gen = torch.Generator(device="cuda").manual_seed(wl.seed + 7)
    dy = torch.randn((wl.T, wl.d), generator=gen, device="cuda").to(inp["x"].dtype)
    x = inp["x"]
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        layer.forward(x, stream)
        layer.backward(x, dy, stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for row in ev:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    M.moe_sm_clock_record(reset=True)
    t0 = time.time()
    for i in range(args.steps):
        ev[i][0].record(stream)
        layer.forward(x, stream)
        ev[i][1].record(stream)
        layer.backward(x, dy, stream)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop(t0, time.time()) if sampler else None
    if clocks is not None:
        clocks["kernel_sm_mhz"] = _kernel_clocks(M)
        _note_inband_cap(clocks)
    if M.moe_last_error() != M.MOE_OK:
        raise RuntimeError("device error word set")
    fwd = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps))
    bwd = sum(ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps))
    elapsed_ms, value = aggregate(fwd + bwd, wl.T * args.steps, ws, "cuda")
    if rank != 0:
        return
    peaks = _peaks()
    rows = wl.T * wl.k + wl.T
    bflops = 12.0 * rows * wl.d * wl.h
    bwd_ms = bwd / args.steps
    peak, kind, clkb = _tensor_peak(peaks, clocks, slot="backward")
    ach = bflops / (bwd_ms / 1e3) / 1e12
    line = {
        "metric": METRIC + " [training step: forward + backward]", "value": value,
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (bf16 weight gradients)" if args.grad_bf16 else "bf16 (fp32 weight gradients)",
        "data": "synthetic (seeded N(0,1) tokens and output gradient, N(0,1/fan_in) weights)",
        "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "h": wl.h, "E": wl.E, "k": wl.k,
                   "l2": "inputs larger than L2"},
        "phase_ms": {"forward": fwd / args.steps, "backward": bwd_ms},
        # forward kernels, then the backward's 12 (tables, dY rows, gaps, du,
        # dH, SwiGLU gradient, dX, three weight gradients, dW_r, dx)
        "gpu_launches": (kernels_per_step(wl, False) + 12) * args.steps,
        "roofline": {"bound": "tensor", "kernel": "backward (dH, dX, weight-gradient GEMMs)",
                     "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                     "traffic": None, "peak_kind": f"{kind}; 12 d h FLOP per row",
                     "flops_per_launch": bflops, "ms_per_launch": bwd_ms,
                     **({"at_kernel_clock": {**clkb, "frac": ach / clkb["peak_tflops"]}}
                        if clkb else {})},
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_bias_dynamics(args, wl):
    """Route + bias update per step on a fresh batch each step (the
    bias-balancing run); reports ms per step and the per-expert load share
    at the first and last timed step."""
    from sparse_moe_layer_fwd_b300 import inputs as I
    from sparse_moe_layer_fwd_b300 import moe as M
    from sparse_moe_layer_fwd_b300.layer import MoeLayer

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    inp = I.make_inputs(wl.with_(seed=wl.seed + 1000 * rank) if ws > 1 else wl, device="cuda",
                        experts=False)
    n = args.warmup + args.steps
    xs = [inp["x"]] + [I.next_x(wl, inp, "cuda") for _ in range(n - 1)]
    b0 = inp["bias"].clone()
    layer = MoeLayer.from_inputs(inp, wl.k, wl.dtype, M.MOE_ROUTE_ONLY)
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    shares = []
    for i in range(n):
        flush.zero_()
        ev[i][0].record(stream)
        layer.forward(xs[i], stream)
        layer.bias_update(1e-3, stream)
        ev[i][1].record(stream)
        if i in (args.warmup, n - 1):
            shares.append((layer.load_counts.float() / (wl.T * wl.k)).cpu())
    torch.cuda.synchronize()
    if M.moe_last_error() != M.MOE_OK:
        raise RuntimeError("device error word set")
    local_ms = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(args.warmup, n))
    elapsed_ms, value = aggregate(local_ms, wl.T * args.steps, ws, "cuda")
    layer.bias.copy_(b0)
    if rank == 0:
        line = {
            "metric": METRIC + " [bias dynamics: route + bias update per step]", "value": value,
            "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if wl.dtype == "f32" else "f32 router, bf16 x",
            "data": "synthetic (seeded N(0,1) tokens per step, router offsets N(0,1))",
            "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k,
                       "l2": "L2 flushed before each step (252 MB write outside the timed spans)"},
            "roofline": None,
            "load_share": {"first_step": [float(shares[0].min()), float(shares[0].max())],
                           "last_step": [float(shares[-1].min()), float(shares[-1].max())],
                           "uniform": 1.0 / wl.E},
            "gpu_launches": kernels_per_step(wl, True) * args.steps + args.steps,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="v3_prefill")
    ap.add_argument("--config", choices=sorted(CONFIGS),
                    help="a configuration by its short name (sets --workload)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=4)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=512,
                    help="output rows the CPU oracle computes for cpu_baseline")
    ap.add_argument("--trace", default=None,
                    help="write the main workload's per-step phase times and raw clock "
                         "samples to this JSON file")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the V3 decode runs that follow the V3 prefill line")
    ap.add_argument("--train", action="store_true",
                    help="time a training step: forward and backward")
    ap.add_argument("--grad-bf16", action="store_true",
                    help="with --train: weight gradients written in bf16 (MOE_GRAD_BF16)")
    ap.add_argument("--fp8", nargs="?", const="gate_up", choices=["gate_up", "block"],
                    help="expert products on e4m3 codes: gate/up only with per-row scales "
                         "(MOE_FP8_GATE_UP, the default), or both with 128x128 / 1x128 "
                         "block scales (MOE_FP8_BLOCK)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the forward replayed from a captured CUDA graph")
    ap.add_argument("--route-only", action="store_true",
                    help="time the routing pass only (router, top-k, load counts)")
    args = ap.parse_args()
    if args.impl == "ours" and args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, _, _ = _dist()
    if args.gpus != ws:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={ws}: launch N > 1 with torchrun")
    from sparse_moe_layer_fwd_b300 import inputs as I
    wl = I.WORKLOADS[CONFIGS[args.config] if args.config else args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.train:
        run_train(args, wl)
    elif wl.steps > 1:
        run_bias_dynamics(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
