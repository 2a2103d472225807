"""bench.py's DRAM-traffic figures: a small-case capture scaled to a full
launch of the same regime, and null once the GEMM sources have changed."""
import numpy as np

import bench
from sparse_moe_layer_fwd_b300 import inputs as I


def _balanced(wl):
    return np.full(wl.E, wl.T * wl.k // wl.E)


def test_capture_case_reproduces_its_own_bytes():
    for key, cap in bench.NCU_TRAFFIC.items():
        if cap["sha"] != bench._kernel_sha():
            continue
        wl = I.WORKLOADS[cap["case"]]
        fp8_blk = key.startswith(":fp8blk")
        got = bench._traffic_for(wl, _balanced(wl), fp8_blk=fp8_blk)
        assert abs(got - cap["bytes"]) <= 1e-9 * cap["bytes"]


def test_regimes_do_not_mix():
    pre, dec = I.WORKLOADS["v3_prefill"], I.WORKLOADS["v3_decode"]
    lp = _balanced(pre)
    ld = np.zeros(dec.E, dtype=np.int64)
    ld[:250] = 1
    tp, td = bench._traffic_for(pre, lp), bench._traffic_for(dec, ld)
    if bench.NCU_TRAFFIC["bf16"]["sha"] == bench._kernel_sha():
        # prefill follows the prefill capture's excess over its algorithmic bytes
        ratio = tp / bench._algorithmic(pre, lp)[2]
        small = I.WORKLOADS["v3_prefill_32experts"]
        assert abs(ratio - bench.NCU_TRAFFIC["bf16"]["bytes"] /
                   bench._algorithmic(small, _balanced(small))[2]) < 1e-12
    if bench.NCU_TRAFFIC["bf16:decode"]["sha"] == bench._kernel_sha():
        small = I.WORKLOADS["v3_decode_32experts"]
        ratio = td / bench._algorithmic(dec, ld)[2]
        assert abs(ratio - bench.NCU_TRAFFIC["bf16:decode"]["bytes"] /
                   bench._algorithmic(small, _balanced(small))[2]) < 1e-12


def test_stale_capture_reports_null(monkeypatch):
    monkeypatch.setattr(bench, "_kernel_sha", lambda read=None: "0" * 16)
    for name in ("v3_prefill", "v3_decode"):
        wl = I.WORKLOADS[name]
        assert bench._traffic_for(wl, _balanced(wl)) is None
    # no capture of the per-row FP8 mode: null whatever the sources
    wl = I.WORKLOADS["v3_prefill"]
    assert bench._traffic_for(wl, _balanced(wl), fp8=True) is None


def test_other_tokens_per_expert_reports_null():
    # 4096 tokens per expert against the capture's 256: L2 reuse differs
    wl = I.WORKLOADS["v3_prefill_16experts"]
    assert bench._traffic_for(wl, _balanced(wl)) is None
