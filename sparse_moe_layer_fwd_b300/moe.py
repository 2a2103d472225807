"""ctypes binding of libmoe.so: the same entry points as include/moe.h.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Pointers may be given as ints or as torch tensors (their
``data_ptr()`` is passed); streams as ints, ``torch.cuda.Stream`` objects or
None (the legacy default stream).  A non-zero return code raises
``MoeError``.  Importing this module fails loudly if libmoe.so has not been
built: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "moe.h")

MOE_F32, MOE_BF16 = 0, 1
MOE_ROUTE_ONLY, MOE_SIMT_EXPERTS, MOE_TRAINING, MOE_FP8_GATE_UP = 1, 2, 4, 8
MOE_FP8_BLOCK = 32
MOE_GRAD_BF16 = 64
MOE_OK = 0
MOE_STATIC_SCRATCH_BYTES = 32 << 20
ERRORS = {
    -1: "MOE_ERR_NULL", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_ALIGN", -4: "MOE_ERR_WORKSPACE",
    -5: "MOE_ERR_DTYPE", -6: "MOE_ERR_LAUNCH", -7: "MOE_ERR_DEVICE_TIMEOUT", -8: "MOE_ERR_DEVICE",
}
ERR_CODE = {v: k for k, v in ERRORS.items()}


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({moe_error_string(code)})")


class MoeDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("h", ctypes.c_int),
                ("E", ctypes.c_int), ("k", ctypes.c_int), ("dtype", ctypes.c_int),
                ("flags", ctypes.c_uint)]


class MoeExpertW(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p)]


class MoeExpertGrad(ctypes.Structure):
    _fields_ = [("d_gate", ctypes.c_void_p), ("d_up", ctypes.c_void_p),
                ("d_down", ctypes.c_void_p)]


class MoeRegion(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 16), ("offset", ctypes.c_size_t),
                ("bytes", ctypes.c_size_t)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is not built ({LIB_PATH}); run "
                          "`python -m sparse_moe_layer_fwd_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, S, I, U = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint
    dp, ep = ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeExpertW)
    lib.moe_workspace_size.argtypes, lib.moe_workspace_size.restype = [dp], S
    lib.moe_host_io_extra_bytes.argtypes, lib.moe_host_io_extra_bytes.restype = [dp], S
    fwd_args = [dp, P, P, P, ep, ep, P, P, P, P, P, S, P]
    lib.moe_forward.argtypes, lib.moe_forward.restype = fwd_args, I
    lib.moe_forward_host_io.argtypes, lib.moe_forward_host_io.restype = fwd_args, I
    lib.moe_forward_profiled.argtypes = fwd_args + [ctypes.POINTER(P)]
    lib.moe_forward_profiled.restype = I
    lib.moe_bias_update.argtypes = [P, P, ctypes.c_float, I, I, P]
    lib.moe_bias_update.restype = I
    gp = ctypes.POINTER(MoeExpertGrad)
    lib.moe_backward.argtypes = [dp, P, P, ep, ep, P, P, P, P, gp, gp, P, P, S, P]
    lib.moe_backward.restype = I
    lib.moe_seq_balance_loss.argtypes = [dp, I, ctypes.c_float, P, P, S, P, P]
    lib.moe_seq_balance_loss.restype = I
    lib.moe_last_error.argtypes, lib.moe_last_error.restype = [], I
    lib.moe_sm_clock_record.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), I]
    lib.moe_sm_clock_record.restype = I
    lib.moe_error_string.argtypes, lib.moe_error_string.restype = [I], ctypes.c_char_p
    lib.moe_workspace_regions.argtypes = [dp, ctypes.POINTER(MoeRegion), I]
    lib.moe_workspace_regions.restype = I
    lib.moe_route_noalloc.argtypes = [dp, P, P, P, P, P, P, P]
    lib.moe_route_noalloc.restype = I
    lib.moe_selftest_timeout.argtypes, lib.moe_selftest_timeout.restype = [U, P], I
    lib.moe_selftest_silu.argtypes, lib.moe_selftest_silu.restype = [P, P, I, P], I
    lib.moe_e4m3_packed_bytes.argtypes = [ctypes.c_longlong, I]
    lib.moe_e4m3_packed_bytes.restype = S
    lib.moe_quantize_rows_e4m3.argtypes = [P, ctypes.c_longlong, I, P, P]
    lib.moe_quantize_rows_e4m3.restype = I
    lib.moe_e4m3_block_packed_bytes.argtypes = [ctypes.c_longlong, I]
    lib.moe_e4m3_block_packed_bytes.restype = S
    lib.moe_quantize_blocks_e4m3.argtypes = [P, ctypes.c_longlong, I, P, P]
    lib.moe_quantize_blocks_e4m3.restype = I
    del U
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def header_functions(path: str = HEADER_PATH) -> list[str]:
    """Names of the functions that include/moe.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*MOE_API\s+(?:size_t|int|const char\*)\s+(moe_\w+)\s*\(", text, re.M)))


def _ptr(v) -> int | None:
    if v is None:
        return None
    if isinstance(v, int):
        return v
    return int(v.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def make_desc(T, d, h, E, k, dtype="bf16", flags=0) -> MoeDesc:
    dt = {"f32": MOE_F32, "bf16": MOE_BF16, MOE_F32: MOE_F32, MOE_BF16: MOE_BF16}[dtype]
    return MoeDesc(int(T), int(d), int(h), int(E), int(k), dt, int(flags))


def make_experts(w_gate, w_up, w_down) -> MoeExpertW:
    return MoeExpertW(_ptr(w_gate), _ptr(w_up), _ptr(w_down))


def make_grads(d_gate, d_up, d_down) -> MoeExpertGrad:
    return MoeExpertGrad(_ptr(d_gate), _ptr(d_up), _ptr(d_down))


def _check(rc: int, where: str) -> int:
    if rc != MOE_OK:
        raise MoeError(rc, where)
    return rc


def moe_workspace_size(desc: MoeDesc) -> int:
    return int(_lib.moe_workspace_size(ctypes.byref(desc)))


def moe_host_io_extra_bytes(desc: MoeDesc) -> int:
    return int(_lib.moe_host_io_extra_bytes(ctypes.byref(desc)))


def moe_forward(desc, x, w_router, bias, experts, shared, y, topk_idx, gates, load_counts,
                workspace, ws_bytes, stream=None, check=True) -> int:
    rc = _lib.moe_forward(ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(bias),
                          ctypes.byref(experts) if experts is not None else None,
                          ctypes.byref(shared) if shared is not None else None,
                          _ptr(y), _ptr(topk_idx), _ptr(gates), _ptr(load_counts),
                          _ptr(workspace), int(ws_bytes), _stream(stream))
    return _check(rc, "moe_forward") if check else rc


N_PHASE_EVENTS = 6
PHASES = ("router", "dispatch", "gemm_gate_up", "gemm_down", "combine")


def moe_forward_profiled(desc, x, w_router, bias, experts, shared, y, topk_idx, gates,
                         load_counts, workspace, ws_bytes, stream, events, check=True) -> int:
    """``events``: N_PHASE_EVENTS torch.cuda.Event objects (or raw handles)."""
    handles = (ctypes.c_void_p * N_PHASE_EVENTS)(
        *[e if isinstance(e, int) else int(e.cuda_event) for e in events])
    rc = _lib.moe_forward_profiled(ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(bias),
                                   ctypes.byref(experts) if experts is not None else None,
                                   ctypes.byref(shared) if shared is not None else None,
                                   _ptr(y), _ptr(topk_idx), _ptr(gates), _ptr(load_counts),
                                   _ptr(workspace), int(ws_bytes), _stream(stream), handles)
    return _check(rc, "moe_forward_profiled") if check else rc


def moe_forward_host_io(desc, x_host, w_router, bias, experts, shared, y_host, topk_idx, gates,
                        load_counts, workspace, ws_bytes, stream=None, check=True) -> int:
    rc = _lib.moe_forward_host_io(ctypes.byref(desc), _ptr(x_host), _ptr(w_router), _ptr(bias),
                                  ctypes.byref(experts) if experts is not None else None,
                                  ctypes.byref(shared) if shared is not None else None,
                                  _ptr(y_host), _ptr(topk_idx), _ptr(gates), _ptr(load_counts),
                                  _ptr(workspace), int(ws_bytes), _stream(stream))
    return _check(rc, "moe_forward_host_io") if check else rc


def moe_bias_update(load_counts, bias, gamma, E, TK, stream=None, check=True) -> int:
    rc = _lib.moe_bias_update(_ptr(load_counts), _ptr(bias), ctypes.c_float(gamma), int(E),
                              int(TK), _stream(stream))
    return _check(rc, "moe_bias_update") if check else rc


def moe_backward(desc, x, w_router, experts, shared, topk_idx, gates, dy, dx, d_experts, d_shared,
                 d_router, workspace, ws_bytes, stream=None, check=True) -> int:
    rc = _lib.moe_backward(ctypes.byref(desc), _ptr(x), _ptr(w_router),
                           ctypes.byref(experts) if experts is not None else None,
                           ctypes.byref(shared) if shared is not None else None,
                           _ptr(topk_idx), _ptr(gates), _ptr(dy), _ptr(dx),
                           ctypes.byref(d_experts) if d_experts is not None else None,
                           ctypes.byref(d_shared) if d_shared is not None else None,
                           _ptr(d_router), _ptr(workspace), int(ws_bytes), _stream(stream))
    return _check(rc, "moe_backward") if check else rc


def moe_seq_balance_loss(desc, seq_len, alpha, topk_idx, workspace, ws_bytes, loss, stream=None,
                         check=True) -> int:
    rc = _lib.moe_seq_balance_loss(ctypes.byref(desc), int(seq_len), ctypes.c_float(alpha),
                                   _ptr(topk_idx), _ptr(workspace), int(ws_bytes), _ptr(loss),
                                   _stream(stream))
    return _check(rc, "moe_seq_balance_loss") if check else rc


def moe_last_error() -> int:
    return int(_lib.moe_last_error())


MOE_CLOCK_SLOTS = 4
CLOCK_SLOT_NAMES = ("gate_up", "down", "backward", "router")


def moe_sm_clock_record(reset: bool = False, check=True) -> dict:
    """Mean SM clock (MHz) each tensor-core kernel class ran at since the
    last reset, from the kernels' in-band cycle and wall-time counters:
    {slot name: {"cycles", "ns", "mhz"}}.  Synchronise first."""
    buf = (ctypes.c_ulonglong * (2 * MOE_CLOCK_SLOTS))()
    rc = _lib.moe_sm_clock_record(buf, 1 if reset else 0)
    if check:
        _check(rc, "moe_sm_clock_record")
    out = {}
    for i, n in enumerate(CLOCK_SLOT_NAMES):
        cyc, ns = int(buf[2 * i]), int(buf[2 * i + 1])
        out[n] = {"cycles": cyc, "ns": ns, "mhz": (1e3 * cyc / ns) if ns else None}
    return out


def moe_error_string(code: int) -> str:
    return _lib.moe_error_string(int(code)).decode()


def moe_workspace_regions(desc: MoeDesc) -> dict:
    regs = (MoeRegion * 16)()
    n = _lib.moe_workspace_regions(ctypes.byref(desc), regs, 16)
    if n < 0:
        raise MoeError(n, "moe_workspace_regions")
    return {regs[i].name.decode(): (int(regs[i].offset), int(regs[i].bytes)) for i in range(n)}


def moe_route_noalloc(desc, x, w_router, bias, topk_idx, gates, load_counts, stream=None,
                      check=True) -> int:
    """Route-only pass (router, top-k, gates, load counts) whose scratch is
    the library's static device array, for callers that must not allocate
    device memory or hand over a workspace.  Same outputs as moe_forward with
    MOE_ROUTE_ONLY; descs needing more than MOE_STATIC_SCRATCH_BYTES of
    scratch are rejected (MOE_ERR_WORKSPACE).  Calls share the array: do not
    let two of them overlap on the GPU."""
    rc = _lib.moe_route_noalloc(ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(bias),
                                _ptr(topk_idx), _ptr(gates), _ptr(load_counts), _stream(stream))
    return _check(rc, "moe_route_noalloc") if check else rc


def moe_e4m3_packed_bytes(rows: int, cols: int) -> int:
    """Bytes of a packed e4m3 matrix: codes [rows, cols], then fp32 scales
    [rows] from the next multiple of 256 bytes."""
    return int(_lib.moe_e4m3_packed_bytes(int(rows), int(cols)))


def e4m3_scale_offset(rows: int, cols: int) -> int:
    return (rows * cols + 255) // 256 * 256


def moe_quantize_rows_e4m3(a, rows, cols, packed, stream=None, check=True) -> int:
    """Per-row e4m3 quantization of the bf16 matrix a [rows, cols] into the
    packed buffer (moe_e4m3_packed_bytes(rows, cols) bytes)."""
    rc = _lib.moe_quantize_rows_e4m3(_ptr(a), int(rows), int(cols), _ptr(packed),
                                     _stream(stream))
    return _check(rc, "moe_quantize_rows_e4m3") if check else rc


def moe_e4m3_block_packed_bytes(rows: int, cols: int) -> int:
    """Bytes of a block-quantized e4m3 matrix: codes [rows, cols], then the
    exponent words [rows / 128][ceil(cols / 512)] from the next multiple of
    256 bytes (0 unless rows and cols are multiples of 128)."""
    return int(_lib.moe_e4m3_block_packed_bytes(int(rows), int(cols)))


def e4m3_block_words(cols: int) -> int:
    """Exponent words per block row (or per activation row): four 128-wide
    blocks per word."""
    return (cols // 128 + 3) // 4


def moe_quantize_blocks_e4m3(a, rows, cols, packed, stream=None, check=True) -> int:
    """Block-scaled e4m3 quantization (128 x 128 blocks) of the bf16 matrix
    a [rows, cols] into the packed buffer (moe_e4m3_block_packed_bytes)."""
    rc = _lib.moe_quantize_blocks_e4m3(_ptr(a), int(rows), int(cols), _ptr(packed),
                                       _stream(stream))
    return _check(rc, "moe_quantize_blocks_e4m3") if check else rc


def moe_selftest_timeout(limit_ms: int, stream=None, check=True) -> int:
    """Enqueue a kernel whose one bounded wait runs out after limit_ms; after
    a synchronise, moe_last_error() reports MOE_ERR_DEVICE_TIMEOUT."""
    rc = _lib.moe_selftest_timeout(int(limit_ms), _stream(stream))
    return _check(rc, "moe_selftest_timeout") if check else rc


def moe_selftest_silu(z, out, stream=None, check=True) -> int:
    """The expert epilogue's silu applied to the fp32 device tensor z -> out."""
    rc = _lib.moe_selftest_silu(_ptr(z), _ptr(out), int(z.numel()), _stream(stream))
    return _check(rc, "moe_selftest_silu") if check else rc
