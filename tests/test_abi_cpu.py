"""The C ABI without a GPU: the library loads, exports every function the
header declares, sizes workspaces, and rejects bad arguments on the host
before anything is launched (the fake pointers below are never touched)."""
import ctypes
import subprocess

import pytest
import torch

from sparse_moe_layer_fwd_b300 import moe as M

FAKE = 1 << 40  # 16-byte aligned, never dereferenced


def test_library_exports_every_header_function():
    names = M.header_functions()
    assert set(names) == {
        "moe_workspace_size", "moe_forward", "moe_host_io_extra_bytes", "moe_forward_host_io",
        "moe_bias_update", "moe_last_error", "moe_error_string", "moe_workspace_regions",
        "moe_forward_profiled", "moe_route_noalloc", "moe_seq_balance_loss", "moe_backward",
        "moe_e4m3_packed_bytes", "moe_quantize_rows_e4m3", "moe_selftest_timeout",
        "moe_e4m3_block_packed_bytes", "moe_quantize_blocks_e4m3", "moe_sm_clock_record",
        "moe_selftest_silu"}
    lib = ctypes.CDLL(M.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", M.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(names), exported ^ set(names)


def test_error_strings():
    for code in [0, *M.ERRORS]:
        assert M.moe_error_string(code) and M.moe_error_string(code) != "unknown error"
    assert M.moe_error_string(12345) == "unknown error"


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(d=0), dict(h=0), dict(E=0), dict(E=1025), dict(k=0), dict(k=33, E=64),
    dict(k=9, E=8), dict(d=96), dict(h=100), dict(dtype=7), dict(flags=8), dict(flags=16),
    dict(flags=32), dict(flags=64),
])
def test_invalid_desc_has_no_workspace(bad):
    kw = dict(T=64, d=256, h=128, E=16, k=4, dtype="f32", flags=0)
    dtype = kw.pop("dtype")
    if "dtype" in bad:
        d = M.MoeDesc(kw["T"], kw["d"], kw["h"], kw["E"], kw["k"], bad["dtype"], 0)
    else:
        kw.update({k: v for k, v in bad.items()})
        d = M.make_desc(kw["T"], kw["d"], kw["h"], kw["E"], kw["k"], dtype, kw["flags"])
    assert M.moe_workspace_size(d) == 0
    assert M.moe_host_io_extra_bytes(d) == 0
    rc = M.moe_forward(d, FAKE, FAKE, FAKE, M.make_experts(FAKE, FAKE, FAKE),
                       M.make_experts(FAKE, FAKE, FAKE), FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40,
                       check=False)
    assert rc in (M.ERR_CODE["MOE_ERR_SHAPE"], M.ERR_CODE["MOE_ERR_DTYPE"])


def test_tensor_core_path_needs_multiples_of_128():
    assert M.moe_workspace_size(M.make_desc(64, 192, 128, 8, 2, "bf16")) == 0
    assert M.moe_workspace_size(M.make_desc(64, 192, 128, 8, 2, "bf16",
                                            M.MOE_SIMT_EXPERTS)) > 0
    assert M.moe_workspace_size(M.make_desc(64, 192, 128, 8, 2, "f32")) > 0
    # the CUDA-core cross-check flag is for bf16 only
    assert M.moe_workspace_size(M.make_desc(64, 256, 128, 8, 2, "f32", M.MOE_SIMT_EXPERTS)) == 0


def _args(desc, **over):
    a = dict(x=FAKE, w_router=FAKE, bias=FAKE, experts=M.make_experts(FAKE, FAKE, FAKE),
             shared=M.make_experts(FAKE, FAKE, FAKE), y=FAKE, topk_idx=FAKE, gates=FAKE,
             load_counts=FAKE, workspace=FAKE, ws_bytes=M.moe_workspace_size(desc))
    a.update(over)
    return a


def _call(desc, **over):
    a = _args(desc, **over)
    return M.moe_forward(desc, a["x"], a["w_router"], a["bias"], a["experts"], a["shared"],
                         a["y"], a["topk_idx"], a["gates"], a["load_counts"], a["workspace"],
                         a["ws_bytes"], check=False)


def test_argument_errors_are_found_on_the_host():
    d = M.make_desc(64, 256, 128, 16, 4, "bf16")
    E = M.ERR_CODE
    assert _call(d, x=None) == E["MOE_ERR_NULL"]
    assert _call(d, y=None) == E["MOE_ERR_NULL"]
    assert _call(d, workspace=None) == E["MOE_ERR_NULL"]
    assert _call(d, experts=M.make_experts(FAKE, None, FAKE)) == E["MOE_ERR_NULL"]
    assert _call(d, experts=None) == E["MOE_ERR_NULL"]
    assert _call(d, x=FAKE + 8) == E["MOE_ERR_ALIGN"]
    assert _call(d, shared=M.make_experts(FAKE, FAKE, FAKE + 2)) == E["MOE_ERR_ALIGN"]
    assert _call(d, ws_bytes=M.moe_workspace_size(d) - 1) == E["MOE_ERR_WORKSPACE"]
    # route-only needs neither y nor expert weights
    r = M.make_desc(64, 256, 128, 16, 4, "bf16", M.MOE_ROUTE_ONLY)
    rc = _call(r, y=None, experts=None, shared=None)
    assert rc != E["MOE_ERR_NULL"]
    # bias update arguments
    assert M.moe_bias_update(None, FAKE, 1e-3, 16, 64, check=False) == E["MOE_ERR_NULL"]
    assert M.moe_bias_update(FAKE, FAKE, 1e-3, 0, 64, check=False) == E["MOE_ERR_SHAPE"]
    assert M.moe_bias_update(FAKE, FAKE, 1e-3, 16, -1, check=False) == E["MOE_ERR_SHAPE"]
    # backward arguments: needs the training flag (bf16 tensor-core path only)
    fk = M.make_experts(FAKE, FAKE, FAKE)
    gk = M.make_grads(FAKE, FAKE, FAKE)
    dt = M.make_desc(64, 256, 128, 16, 4, "bf16", M.MOE_TRAINING)
    wst = M.moe_workspace_size(dt)
    bw = lambda desc=dt, **o: M.moe_backward(  # noqa: E731
        desc, o.get("x", FAKE), FAKE, fk, fk, FAKE, FAKE, o.get("dy", FAKE), FAKE,
        o.get("dexp", gk), gk, FAKE, FAKE, o.get("ws_bytes", wst), check=False)
    assert wst > M.moe_workspace_size(d)
    assert bw(desc=d) == E["MOE_ERR_DTYPE"]
    assert M.moe_workspace_size(M.make_desc(64, 256, 128, 16, 4, "f32", M.MOE_TRAINING)) == 0
    assert bw(dy=None) == E["MOE_ERR_NULL"]
    assert bw(dexp=M.make_grads(FAKE, None, FAKE)) == E["MOE_ERR_NULL"]
    assert bw(x=FAKE + 4) == E["MOE_ERR_ALIGN"]
    assert bw(ws_bytes=wst - 1) == E["MOE_ERR_WORKSPACE"]
    # balance-loss arguments
    ws = M.moe_workspace_size(d)
    bl = lambda **o: M.moe_seq_balance_loss(  # noqa: E731
        o.get("desc", d), o.get("seq_len", 16), 1e-4, o.get("idx", FAKE), o.get("ws", FAKE),
        o.get("ws_bytes", ws), o.get("loss", FAKE), check=False)
    assert bl(seq_len=0) == E["MOE_ERR_SHAPE"]
    assert bl(idx=None) == E["MOE_ERR_NULL"]
    assert bl(loss=None) == E["MOE_ERR_NULL"]
    assert bl(ws_bytes=ws - 1) == E["MOE_ERR_WORKSPACE"]
    assert bl(ws=FAKE + 4) == E["MOE_ERR_ALIGN"]
    assert bl(desc=M.make_desc(0, 256, 128, 16, 4, "bf16"), idx=None) == M.MOE_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_valid_call_without_gpu_reports_device_error():
    d = M.make_desc(64, 256, 128, 16, 4, "f32")
    assert _call(d) == M.ERR_CODE["MOE_ERR_DEVICE"]
    assert M.moe_bias_update(FAKE, FAKE, 1e-3, 16, 64, check=False) == M.ERR_CODE["MOE_ERR_DEVICE"]
    assert M.moe_seq_balance_loss(d, 16, 1e-4, FAKE, FAKE, M.moe_workspace_size(d), FAKE,
                                  check=False) == M.ERR_CODE["MOE_ERR_DEVICE"]


@pytest.mark.parametrize("shape", [
    (256, 256, 128, 16, 4, "f32"), (8192, 384, 384, 16, 4, "bf16"),
    (8192, 7168, 2048, 256, 8, "bf16"), (128, 7168, 2048, 256, 8, "bf16"), (0, 256, 128, 16, 4, "bf16"),
    (1, 128, 128, 1, 1, "bf16"),
])
def test_workspace_regions_are_disjoint_and_aligned(shape):
    T, d, h, E, k, dt = shape
    desc = M.make_desc(T, d, h, E, k, dt)
    total = M.moe_workspace_size(desc)
    regs = M.moe_workspace_regions(desc)
    assert total > 0 and len(regs) == 12
    spans = sorted(regs.values())
    for (o1, b1), (o2, _) in zip(spans, spans[1:]):
        assert o1 % 256 == 0 and o1 + b1 <= o2
    assert spans[-1][0] + spans[-1][1] <= total
    el = 4 if dt == "f32" else 2
    assert regs["x_perm"][1] == T * k * d * el
    assert regs["h"][1] == (T * k + T) * h * el
    # the routed rows, then the shared expert's rows
    assert regs["y_perm"][1] == (T * k + T) * d * el
    assert regs["x_q"][1] == 0 and regs["h_q"][1] == 0
    # the tensor-core router (bf16 tokens, 96 experts or more) keeps the
    # router weights as three bf16 terms, expert rows padded to 256
    tc_router = dt == "bf16" and E >= 96 and T > 0
    assert regs["router_w3"][1] == (3 * ((E + 255) // 256 * 256) * d * 2 if tc_router else 0)
    ro = M.make_desc(T, d, h, E, k, dt, M.MOE_ROUTE_ONLY)
    assert M.moe_workspace_size(ro) <= total and len(M.moe_workspace_regions(ro)) == 5
    assert M.moe_host_io_extra_bytes(desc) >= 2 * T * d * el


@pytest.mark.parametrize("F", [M.MOE_FP8_GATE_UP, M.MOE_FP8_BLOCK])
def test_fp8_flags(F):
    # bf16 tensor-core forward only; the two fp8 modes do not combine; flag
    # 16 is not a flag
    for bad in (("f32", F), ("bf16", F | M.MOE_SIMT_EXPERTS), ("bf16", F | M.MOE_ROUTE_ONLY),
                ("bf16", F | M.MOE_TRAINING), ("bf16", M.MOE_FP8_GATE_UP | M.MOE_FP8_BLOCK),
                ("bf16", F | 16)):
        assert M.moe_workspace_size(M.make_desc(64, 256, 128, 16, 4, bad[0], bad[1])) == 0
    T, d, h, E, k = 300, 7168, 2048, 256, 8
    desc = M.make_desc(T, d, h, E, k, "bf16", F)
    regs = M.moe_workspace_regions(desc)
    assert len(regs) == 12
    R = T * k + T
    # the gathered token rows hold one-byte codes in both modes
    assert regs["x_perm"][1] == T * k * d
    if F == M.MOE_FP8_GATE_UP:
        # x_q: the tokens' codes, then their row scales; H in bf16
        assert regs["x_q"][1] == (T * d + 255) // 256 * 256 + 4 * T
        assert regs["h_q"][1] == 0 and regs["h"][1] == R * h * 2
    else:
        # x_q: codes, then exponent words [ceil(d / 512)][T]; h_q likewise for
        # the hidden rows, which are never held in bf16
        assert regs["x_q"][1] == (T * d + 255) // 256 * 256 + 4 * T * ((d // 128 + 3) // 4)
        assert regs["h_q"][1] == (R * h + 255) // 256 * 256 + 4 * R * ((h // 128 + 3) // 4)
        assert regs["h"][1] == 0
    assert regs["x_q"][0] % 256 == 0 and regs["h_q"][0] % 256 == 0


def test_block_packed_layout_and_argument_errors():
    assert M.moe_e4m3_block_packed_bytes(128, 640) == 128 * 640 + 4 * 2
    assert M.moe_e4m3_block_packed_bytes(256, 7168) == 256 * 7168 + 2 * 14 * 4
    for rows, cols in ((100, 128), (128, 100), (0, 128), (-128, 128), (128, 0)):
        expect = (256 * 0 + 0) if rows == 0 and cols == 128 else 0
        assert M.moe_e4m3_block_packed_bytes(rows, cols) == expect
    E = M.ERR_CODE
    q = lambda a=FAKE, rows=128, cols=128, out=FAKE: M.moe_quantize_blocks_e4m3(  # noqa: E731
        a, rows, cols, out, check=False)
    assert q(cols=100) == E["MOE_ERR_SHAPE"] and q(rows=64) == E["MOE_ERR_SHAPE"]
    assert q(a=None) == E["MOE_ERR_NULL"] and q(out=None) == E["MOE_ERR_NULL"]
    assert q(out=FAKE + 8) == E["MOE_ERR_ALIGN"]
    assert q(rows=0, a=None) == M.MOE_OK


def test_e4m3_packed_layout_and_argument_errors():
    assert M.moe_e4m3_packed_bytes(10, 24) == 256 + 40
    assert M.moe_e4m3_packed_bytes(256, 7168) == 256 * 7168 + 1024
    assert M.moe_e4m3_packed_bytes(0, 128) == 0
    assert M.moe_e4m3_packed_bytes(-1, 128) == 0 and M.moe_e4m3_packed_bytes(4, 0) == 0
    E = M.ERR_CODE
    q = lambda a=FAKE, rows=4, cols=128, out=FAKE: M.moe_quantize_rows_e4m3(  # noqa: E731
        a, rows, cols, out, check=False)
    assert q(cols=100) == E["MOE_ERR_SHAPE"]
    assert q(rows=-1) == E["MOE_ERR_SHAPE"]
    assert q(a=None) == E["MOE_ERR_NULL"] and q(out=None) == E["MOE_ERR_NULL"]
    assert q(out=FAKE + 8) == E["MOE_ERR_ALIGN"]
    assert q(rows=0, a=None) == M.MOE_OK


def test_selftest_timeout_arguments():
    E = M.ERR_CODE
    assert M.moe_selftest_timeout(0, check=False) == E["MOE_ERR_SHAPE"]
    assert M.moe_selftest_timeout(10001, check=False) == E["MOE_ERR_SHAPE"]
    if not torch.cuda.is_available():
        assert M.moe_selftest_timeout(100, check=False) == E["MOE_ERR_DEVICE"]


def test_static_scratch_size_matches_the_header():
    """The binding's copy of MOE_STATIC_SCRATCH_BYTES is the header's value."""
    import re
    text = open(M.HEADER_PATH).read()
    m = re.search(r"#define\s+MOE_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "MOE_STATIC_SCRATCH_BYTES not found in moe.h"
    assert M.MOE_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_noalloc_rejects_problems_larger_than_its_array():
    """The size check comes before anything touches a device: fake pointers
    and no GPU are enough."""
    # 65536 tokens x 256 experts: the fp32 router logits alone take 64 MiB
    big = M.make_desc(65536, 128, 128, 256, 1, "bf16")
    need = M.moe_workspace_size(M.make_desc(65536, 128, 128, 256, 1, "bf16", M.MOE_ROUTE_ONLY))
    assert M.moe_workspace_size(big) > 0  # a valid problem ...
    assert need > M.MOE_STATIC_SCRATCH_BYTES  # ... whose routing scratch does not fit
    rc = M.moe_route_noalloc(big, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, check=False)
    assert rc == M.ERR_CODE["MOE_ERR_WORKSPACE"]
    assert M.library().moe_route_noalloc(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                         None) == M.ERR_CODE["MOE_ERR_NULL"]


def test_clock_record_slots_match_the_header():
    """The binding's slot count and order are the header's MOE_CLOCK_*."""
    import re
    text = open(M.HEADER_PATH).read()
    slots = {m.group(1): int(m.group(2))
             for m in re.finditer(r"#define\s+MOE_CLOCK_(\w+)\s+(\d+)", text)}
    assert slots.pop("SLOTS") == M.MOE_CLOCK_SLOTS == len(M.CLOCK_SLOT_NAMES)
    assert sorted(slots.values()) == list(range(M.MOE_CLOCK_SLOTS))
    for name, idx in slots.items():
        assert M.CLOCK_SLOT_NAMES[idx] == {"GATE_UP": "gate_up", "DOWN": "down",
                                           "BWD": "backward", "ROUTER": "router"}[name]


def test_clock_record_arguments():
    assert M.library().moe_sm_clock_record(None, 0) == M.ERR_CODE["MOE_ERR_NULL"]


@pytest.mark.parametrize("E", [34, 98, 256])
def test_group_table_holds_every_scheduler_counter(E):
    """The group table: seven per-group arrays (7 E + 12 ints) and then the
    schedulers' tile counters, of which the backward uses next[2..7] -- the
    region must hold all of them even where its size is a multiple of the
    256-byte region alignment (E = 34 mod 64 with the old size)."""
    regs = M.moe_workspace_regions(M.make_desc(64, 128, 128, E, 2, "bf16", M.MOE_TRAINING))
    assert regs["groups"][1] >= (7 * E + 12 + 8) * 4


def test_selftest_silu_arguments():
    E = M.ERR_CODE
    lib = M.library()
    assert lib.moe_selftest_silu(None, None, -1, None) == E["MOE_ERR_SHAPE"]
    assert lib.moe_selftest_silu(None, None, 0, None) == M.MOE_OK
    assert lib.moe_selftest_silu(None, FAKE, 4, None) == E["MOE_ERR_NULL"]
    if not torch.cuda.is_available():
        assert lib.moe_selftest_silu(FAKE, FAKE, 4, None) == E["MOE_ERR_DEVICE"]
