"""Device buffers for one MoE layer and calls through the C ABI.

PyTorch provides the device memory and the stream; every step of the layer
runs in libmoe.so.  ``MoeLayer`` owns the outputs and the workspace for one
problem size and re-uses them on every call.
"""
from __future__ import annotations

import torch

from . import moe as M


def _check(name, t, shape, dtype, device):
    """Raise unless t is a contiguous tensor of exactly this shape and dtype
    on this device: the library reads and writes exactly that many elements
    from its data pointer, so anything else would be read past its end (or,
    off the GPU, not be device memory at all)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    shape = tuple(int(n) for n in shape)
    if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous {dtype} tensor of shape {shape}, got "
                         f"{t.dtype} {tuple(t.shape)}"
                         + ("" if t.is_contiguous() else " (not contiguous)"))
    if t.device != device:
        raise ValueError(f"{name}: expected a tensor on {device}, got one on {t.device}")


class MoeLayer:
    def __init__(self, w_router, bias, w_gate, w_up, w_down, sh_gate, sh_up, sh_down, *,
                 T: int, k: int, dtype: str, flags: int = 0, host_io: bool = False):
        self.E, self.d = w_router.shape
        self.h = w_gate.shape[1] if w_gate is not None else 128
        self.T, self.k, self.dtype, self.flags = T, k, dtype, flags
        dev = w_router.device
        if dev.type != "cuda":
            raise ValueError(f"w_router: expected a CUDA tensor, got one on {dev}")
        E, d, h = self.E, self.d, self.h
        tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        _check("w_router", w_router, (E, d), torch.float32, dev)
        _check("bias", bias, (E,), torch.float32, dev)
        if w_gate is not None:
            for name, t, shape in (("w_gate", w_gate, (E, h, d)), ("w_up", w_up, (E, h, d)),
                                   ("w_down", w_down, (E, d, h)), ("sh_gate", sh_gate, (h, d)),
                                   ("sh_up", sh_up, (h, d)), ("sh_down", sh_down, (d, h))):
                _check(name, t, shape, tdt, dev)
        self.desc = M.make_desc(T, self.d, self.h, self.E, k, dtype, flags)
        self.w_router, self.bias = w_router, bias
        self._keep = (w_gate, w_up, w_down, sh_gate, sh_up, sh_down)
        have_w = w_gate is not None
        # fp8 modes: the weights they name as packed e4m3 matrices (codes +
        # row scales, or codes + block exponents), quantized once here
        self.packed = {}
        if have_w and flags & M.MOE_FP8_GATE_UP:
            self.packed.update({"w_gate": self.quantize(w_gate), "w_up": self.quantize(w_up),
                                "sh_gate": self.quantize(sh_gate), "sh_up": self.quantize(sh_up)})
            w_gate, w_up = self.packed["w_gate"], self.packed["w_up"]
            sh_gate, sh_up = self.packed["sh_gate"], self.packed["sh_up"]
        if have_w and flags & M.MOE_FP8_BLOCK:
            qb = self.quantize_blocks
            self.packed.update({"w_gate": qb(w_gate), "w_up": qb(w_up), "w_down": qb(w_down),
                                "sh_gate": qb(sh_gate), "sh_up": qb(sh_up),
                                "sh_down": qb(sh_down)})
            w_gate, w_up, w_down = self.packed["w_gate"], self.packed["w_up"], self.packed["w_down"]
            sh_gate, sh_up, sh_down = (self.packed["sh_gate"], self.packed["sh_up"],
                                       self.packed["sh_down"])
        self.experts = M.make_experts(w_gate, w_up, w_down) if have_w else None
        self.shared = M.make_experts(sh_gate, sh_up, sh_down) if have_w else None
        self._tdt = tdt
        self.ws_bytes = M.moe_workspace_size(self.desc)
        if self.ws_bytes == 0:
            raise M.MoeError(M.ERR_CODE["MOE_ERR_SHAPE"], "moe_workspace_size")
        if host_io:
            self.ws_bytes += M.moe_host_io_extra_bytes(self.desc)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        route_only = bool(flags & M.MOE_ROUTE_ONLY)
        self.y = None if (route_only or host_io) else torch.empty((T, self.d), dtype=tdt, device=dev)
        self.topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.gates = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.load_counts = torch.empty((self.E,), dtype=torch.int32, device=dev)
        self.regions = M.moe_workspace_regions(self.desc)

    @staticmethod
    def quantize(w: torch.Tensor, stream=None) -> torch.Tensor:
        """Packed per-row e4m3 copy of a bf16 weight tensor (rows = all but the
        last dimension): codes, then fp32 scales from a 256-byte boundary."""
        cols = w.shape[-1]
        rows = w.numel() // cols
        out = torch.empty(M.moe_e4m3_packed_bytes(rows, cols), dtype=torch.uint8,
                          device=w.device)
        if stream is None:
            stream = torch.cuda.current_stream(w.device)
        M.moe_quantize_rows_e4m3(w.contiguous(), rows, cols, out, stream)
        return out

    @staticmethod
    def quantize_blocks(w: torch.Tensor, stream=None) -> torch.Tensor:
        """Packed block-scaled e4m3 copy (128 x 128 blocks) of a bf16 weight
        tensor (rows = all but the last dimension): codes, then exponent
        words from a 256-byte boundary."""
        cols = w.shape[-1]
        rows = w.numel() // cols
        out = torch.empty(M.moe_e4m3_block_packed_bytes(rows, cols), dtype=torch.uint8,
                          device=w.device)
        if stream is None:
            stream = torch.cuda.current_stream(w.device)
        M.moe_quantize_blocks_e4m3(w.contiguous(), rows, cols, out, stream)
        return out

    @staticmethod
    def unpack_blocks(packed: torch.Tensor, rows: int, cols: int, act_rows: bool = False):
        """(codes uint8 [rows, cols], exponents uint8 [row blocks, cols / 128])
        of a packed block matrix; act_rows: an activation layout (one block
        row per row, words [ceil(cols / 512)][rows])."""
        so = M.e4m3_scale_offset(rows, cols)
        wpr = M.e4m3_block_words(cols)
        codes = packed[:rows * cols].view(rows, cols)
        nb = cols // 128
        if act_rows:
            w = packed[so:so + 4 * wpr * rows].view(wpr, rows, 4)
            ex = w.permute(1, 0, 2).reshape(rows, 4 * wpr)[:, :nb]
        else:
            w = packed[so:so + 4 * wpr * (rows // 128)].view(rows // 128, 4 * wpr)
            ex = w[:, :nb]
        return codes, ex

    @staticmethod
    def unpack(packed: torch.Tensor, rows: int, cols: int):
        """(codes uint8 [rows, cols], scales fp32 [rows]) views of a packed matrix."""
        so = M.e4m3_scale_offset(rows, cols)
        return (packed[:rows * cols].view(rows, cols),
                packed[so:so + 4 * rows].view(torch.float32))

    @classmethod
    def from_inputs(cls, inp: dict, k: int, dtype: str, flags: int = 0, T: int | None = None,
                    host_io: bool = False) -> "MoeLayer":
        T = inp["x"].shape[0] if T is None else T
        return cls(inp["w_router"], inp["bias"], inp.get("w_gate"), inp.get("w_up"),
                   inp.get("w_down"), inp.get("sh_gate"), inp.get("sh_up"), inp.get("sh_down"),
                   T=T, k=k, dtype=dtype, flags=flags, host_io=host_io)

    def forward(self, x, stream=None):
        _check("x", x, (self.T, self.d), self._tdt, self.workspace.device)
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        M.moe_forward(self.desc, x, self.w_router, self.bias, self.experts, self.shared, self.y,
                      self.topk_idx, self.gates, self.load_counts, self.workspace, self.ws_bytes,
                      stream)
        return self.y

    def forward_host_io(self, x_host, y_host, stream=None):
        cpu = torch.device("cpu")
        _check("x_host", x_host, (self.T, self.d), self._tdt, cpu)
        _check("y_host", y_host, (self.T, self.d), self._tdt, cpu)
        if stream is None:
            stream = torch.cuda.current_stream(self.workspace.device)
        M.moe_forward_host_io(self.desc, x_host, self.w_router, self.bias, self.experts,
                              self.shared, y_host, self.topk_idx, self.gates, self.load_counts,
                              self.workspace, self.ws_bytes, stream)
        return y_host

    def bias_update(self, gamma: float = 1e-3, stream=None):
        if stream is None:
            stream = torch.cuda.current_stream(self.workspace.device)
        M.moe_bias_update(self.load_counts, self.bias, gamma, self.E, self.T * self.k, stream)

    def backward(self, x, dy, stream=None) -> dict:
        """Gradients for the output gradient dy, after forward(x) on this layer
        (built with MOE_TRAINING): dx, the expert and shared-expert weight
        gradients (fp32, or bf16 with MOE_GRAD_BF16) and the router's."""
        _check("x", x, (self.T, self.d), self._tdt, self.workspace.device)
        _check("dy", dy, (self.T, self.d), self._tdt, self.workspace.device)
        if stream is None:
            stream = torch.cuda.current_stream(self.workspace.device)
        wg, wu, wd, sg, su, sd = self._keep
        f32 = dict(dtype=torch.float32, device=self.workspace.device)
        wdt = dict(dtype=torch.bfloat16 if self.flags & M.MOE_GRAD_BF16 else torch.float32,
                   device=self.workspace.device)
        g = {"dx": torch.empty_like(dy), "dW_gate": torch.empty(wg.shape, **wdt),
             "dW_up": torch.empty(wu.shape, **wdt), "dW_down": torch.empty(wd.shape, **wdt),
             "dsh_gate": torch.empty(sg.shape, **wdt), "dsh_up": torch.empty(su.shape, **wdt),
             "dsh_down": torch.empty(sd.shape, **wdt),
             "dW_router": torch.empty(self.w_router.shape, **f32)}
        M.moe_backward(self.desc, x, self.w_router, self.experts, self.shared, self.topk_idx,
                       self.gates, dy, g["dx"],
                       M.make_grads(g["dW_gate"], g["dW_up"], g["dW_down"]),
                       M.make_grads(g["dsh_gate"], g["dsh_up"], g["dsh_down"]),
                       g["dW_router"], self.workspace, self.ws_bytes, stream)
        return g

    def balance_loss(self, seq_len: int, alpha: float = 1e-4, stream=None) -> torch.Tensor:
        """Per-sequence balance loss of the routing of the last forward."""
        if stream is None:
            stream = torch.cuda.current_stream(self.workspace.device)
        out = torch.empty(((self.T + seq_len - 1) // seq_len,), dtype=torch.float32,
                          device=self.workspace.device)
        M.moe_seq_balance_loss(self.desc, seq_len, alpha, self.topk_idx, self.workspace,
                               self.ws_bytes, out, stream)
        return out

    def region(self, name: str, dtype: torch.dtype, shape) -> torch.Tensor:
        """A view of a named workspace region (for inspecting intermediates)."""
        off, nbytes = self.regions[name]
        el = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        assert n * el <= nbytes, (name, shape, nbytes)
        return self.workspace[off:off + n * el].view(dtype).view(*shape)
