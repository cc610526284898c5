"""Python binding of libbeam_moe.so, the sm_103a forward pass of Beam's
Mixture-of-Experts block (sigmoid router with selection bias and
group-limited top-k, dispatch, SwiGLU experts, combine).

Argument marshalling only: every function here checks tensor dtypes, shapes
and devices, then calls the C entry point of the same name in
``include/beam_moe.h`` with raw device pointers and the current CUDA stream.
Every step of the computation runs in the library's kernels; there is no
fallback, and importing this package fails if the library is missing.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbeam_moe.so")

MOE_OK = 0
MOE_W_BF16, MOE_W_NVFP4, MOE_W_FP8, MOE_W_NVFP4_A4 = 0, 1, 2, 3
MOE_OP_ROUTE, MOE_OP_PERMUTE, MOE_OP_EXPERTS, MOE_OP_FORWARD = 0, 1, 2, 3
MOE_DEV_TIMEOUT, MOE_DEV_BAD_INDEX = 0x1, 0x2
MOE_LAYOUT_ROWMAJOR, MOE_LAYOUT_TILED = 0, 1

EXPORTED = ("moe_version", "moe_status_string", "moe_check_dims", "moe_workspace_size",
            "moe_workspace_init", "moe_workspace_status", "moe_route", "moe_route_logits",
            "moe_permute",
            "moe_experts_swiglu", "moe_combine", "moe_forward", "moe_bias_update",
            "moe_quantize_nvfp4", "moe_pack_bf16", "moe_pack_nvfp4", "moe_pack_fp8",
            "moe_permute_noalloc")


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int),
                ("n_group", ctypes.c_int), ("topk_group", ctypes.c_int), ("top_k", ctypes.c_int),
                ("I", ctypes.c_int), ("routed_scale", ctypes.c_float)]


class MoeExperts(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int),
                ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("g_gate", ctypes.c_void_p), ("g_up", ctypes.c_void_p), ("g_down", ctypes.c_void_p),
                ("x_global", ctypes.c_float), ("h_global", ctypes.c_float),
                ("layout", ctypes.c_int)]


_P, _I, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_DP = ctypes.POINTER(MoeDims)
_sig = {
    "moe_version": ([], _I),
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_check_dims": ([_DP], _I),
    "moe_workspace_size": ([_DP, _I, _I], _S),
    "moe_workspace_init": ([_P, _P], _I),
    "moe_workspace_status": ([_P, _P, ctypes.POINTER(ctypes.c_uint32)], _I),
    "moe_route": ([_DP, _P, _P, _P, _P, _P, _P, _S, _P], _I),
    "moe_route_logits": ([_DP, _P, _P, _P, _P, _P, _P, _P, _S, _P], _I),
    "moe_permute": ([_DP, _P, _P, _P, _P, _P, _P, _P, _S, _P], _I),
    "moe_experts_swiglu": ([_DP, ctypes.POINTER(MoeExperts), _P, _P, _P, _P, _P, _P, _S, _P], _I),
    "moe_combine": ([_DP, _P, _P, _P, _P], _I),
    "moe_forward": ([_DP, _P, _P, _P, ctypes.POINTER(MoeExperts), _P, _P, _P, _P, _S, _P], _I),
    "moe_quantize_nvfp4": ([_I, _I, _P, ctypes.c_float, _P, _P, _P], _I),
    "moe_pack_bf16": ([_I, _I, _I, _P, _P, _P], _I),
    "moe_pack_nvfp4": ([_I, _I, _I, _P, _P, _P, _P], _I),
    "moe_pack_fp8": ([_I, _I, _I, _P, _P, _P], _I),
    "moe_bias_update": ([_DP, _P, _P, ctypes.c_double, _I, _I, ctypes.POINTER(ctypes.c_float), _P], _I),
    "moe_permute_noalloc": ([_DP, _P, _P, _P, _P, _P, _P, _P], _I),
}
_native = None


def native() -> ctypes.CDLL:
    """The loaded libbeam_moe.so.  Raises ImportError if it has not been built:
    there is no other implementation to fall back to."""
    global _native
    if _native is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing; build it with "
                              "`python -m group_limited_routing_bias_b300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, ret) in _sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ret
        _native = lib
    return _native


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def status_string(status: int) -> str:
    return native().moe_status_string(status).decode()


def version() -> int:
    return native().moe_version()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def make_dims(T, H, E, n_group, topk_group, top_k, I, routed_scale) -> MoeDims:
    return MoeDims(T, H, E, n_group, topk_group, top_k, I, routed_scale)


def dims_of(cfg, T: Optional[int] = None) -> MoeDims:
    """Dims from any object with the fields T, H, E, n_group, topk_group, top_k, I, routed_scale."""
    return MoeDims(cfg.T if T is None else T, cfg.H, cfg.E, cfg.n_group, cfg.topk_group, cfg.top_k,
                   cfg.I, cfg.routed_scale)


def check_dims(d: MoeDims) -> int:
    return native().moe_check_dims(ctypes.byref(d))


def workspace_size(d: MoeDims, op: int, wdtype: int = MOE_W_BF16) -> int:
    return native().moe_workspace_size(ctypes.byref(d), wdtype, op)


def alloc_workspace(d: MoeDims, op: int, wdtype: int = MOE_W_BF16, device="cuda") -> torch.Tensor:
    """A zeroed workspace of the right size (device memory from torch's allocator)."""
    n = workspace_size(d, op, wdtype)
    if n == 0:
        raise MoeError("moe_workspace_size", 2)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor], dtype=None, shape=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the workspace's device status bits."""
    bits = ctypes.c_uint32(0)
    st = native().moe_workspace_status(_ptr(ws, torch.uint8, name="ws"), _stream(stream), ctypes.byref(bits))
    if st not in (MOE_OK, 5):
        raise MoeError("moe_workspace_status", st)
    return bits.value


def workspace_init(ws: torch.Tensor, stream=None):
    _check("moe_workspace_init", native().moe_workspace_init(_ptr(ws, torch.uint8, name="ws"), _stream(stream)))


@dataclass
class Experts:
    """Expert weights of one layer.

    bf16: w_gate, w_up [E, I, H], w_down [E, H, I].
    NVFP4: w_* packed e2m1 uint8 [E, N, K/2], s_* e4m3 uint8 [E, N, K/16], g_* fp32 [E].
    FP8: w_* e4m3 uint8 [E, N, K], s_* None, g_* fp32 [E, N] row scales.
    a4 = (x_global, h_global) with NVFP4 weights selects W4A4: x and h are
    quantised to NVFP4 with those static global scales.
    tiled = True: weights in the tiled layouts of moe_pack_bf16 (bf16, same
    shapes), moe_pack_nvfp4 (NVFP4: w_* uint8 [E, N, 9K/16] holding codes and
    block scales, s_* None, wdtype = MOE_W_NVFP4) or moe_pack_fp8 (FP8, same
    shapes); to_tiled() makes such a copy.  wdtype overrides the format that
    the tensors' dtypes imply (needed only for tiled NVFP4).
    """
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    s_gate: Optional[torch.Tensor] = None
    s_up: Optional[torch.Tensor] = None
    s_down: Optional[torch.Tensor] = None
    g_gate: Optional[torch.Tensor] = None
    g_up: Optional[torch.Tensor] = None
    g_down: Optional[torch.Tensor] = None
    a4: Optional[tuple] = None
    tiled: bool = False
    wdtype: Optional[int] = None

    @property
    def dtype(self) -> int:
        if self.wdtype is not None:
            return self.wdtype
        if self.w_gate.dtype != torch.uint8:
            return MOE_W_BF16
        if self.s_gate is None:
            return MOE_W_FP8
        return MOE_W_NVFP4 if self.a4 is None else MOE_W_NVFP4_A4

    def to_tiled(self, stream=None) -> "Experts":
        """A copy with the weights packed into the tiled layout (bf16, NVFP4
        W4A16 or FP8; W4A4 takes row-major weights only)."""
        if self.tiled:
            return self
        if self.dtype == MOE_W_BF16:
            return Experts(*(moe_pack_bf16(w, stream) for w in (self.w_gate, self.w_up, self.w_down)),
                           tiled=True)
        if self.dtype == MOE_W_FP8:
            return Experts(*(moe_pack_fp8(w, stream) for w in (self.w_gate, self.w_up, self.w_down)),
                           None, None, None, self.g_gate, self.g_up, self.g_down, tiled=True)
        if self.dtype == MOE_W_NVFP4:
            return Experts(moe_pack_nvfp4(self.w_gate, self.s_gate, stream),
                           moe_pack_nvfp4(self.w_up, self.s_up, stream),
                           moe_pack_nvfp4(self.w_down, self.s_down, stream), None, None, None,
                           self.g_gate, self.g_up, self.g_down, tiled=True, wdtype=MOE_W_NVFP4)
        raise ValueError("W4A4 experts take row-major weights only")

    def struct(self, d: MoeDims) -> MoeExperts:
        E, H, I = d.E, d.H, d.I
        layout = MOE_LAYOUT_TILED if self.tiled else MOE_LAYOUT_ROWMAJOR
        if self.dtype == MOE_W_BF16:
            bf = torch.bfloat16
            return MoeExperts(MOE_W_BF16, _ptr(self.w_gate, bf, (E, I, H), "w_gate"),
                              _ptr(self.w_up, bf, (E, I, H), "w_up"),
                              _ptr(self.w_down, bf, (E, H, I), "w_down"), None, None, None, None,
                              None, None, 0.0, 0.0,
                              MOE_LAYOUT_TILED if self.tiled else MOE_LAYOUT_ROWMAJOR)
        u8, f32 = torch.uint8, torch.float32
        if self.dtype == MOE_W_FP8:
            return MoeExperts(MOE_W_FP8, _ptr(self.w_gate, u8, (E, I, H), "w_gate"),
                              _ptr(self.w_up, u8, (E, I, H), "w_up"),
                              _ptr(self.w_down, u8, (E, H, I), "w_down"), None, None, None,
                              _ptr(self.g_gate, f32, (E, I), "g_gate"),
                              _ptr(self.g_up, f32, (E, I), "g_up"),
                              _ptr(self.g_down, f32, (E, H), "g_down"), 0.0, 0.0, layout)
        if self.dtype == MOE_W_NVFP4 and self.tiled:
            return MoeExperts(MOE_W_NVFP4,
                              _ptr(self.w_gate, u8, (E, I, H * 9 // 16), "w_gate"),
                              _ptr(self.w_up, u8, (E, I, H * 9 // 16), "w_up"),
                              _ptr(self.w_down, u8, (E, H, I * 9 // 16), "w_down"), None, None, None,
                              _ptr(self.g_gate, f32, (E,), "g_gate"), _ptr(self.g_up, f32, (E,), "g_up"),
                              _ptr(self.g_down, f32, (E,), "g_down"), 0.0, 0.0, layout)
        gx, gh = self.a4 if self.a4 is not None else (0.0, 0.0)
        return MoeExperts(self.dtype,
                          _ptr(self.w_gate, u8, (E, I, H // 2), "w_gate"),
                          _ptr(self.w_up, u8, (E, I, H // 2), "w_up"),
                          _ptr(self.w_down, u8, (E, H, I // 2), "w_down"),
                          _ptr(self.s_gate, u8, (E, I, H // 16), "s_gate"),
                          _ptr(self.s_up, u8, (E, I, H // 16), "s_up"),
                          _ptr(self.s_down, u8, (E, H, I // 16), "s_down"),
                          _ptr(self.g_gate, f32, (E,), "g_gate"), _ptr(self.g_up, f32, (E,), "g_up"),
                          _ptr(self.g_down, f32, (E,), "g_down"), float(gx), float(gh), layout)


def moe_route(d: MoeDims, x, w_router, bias, topk_idx, topk_w, ws, stream=None):
    """Router; fills topk_idx int32 [T,k] and topk_w fp32 [T,k]."""
    T, H, E, k = d.T, d.H, d.E, d.top_k
    _check("moe_route", native().moe_route(
        ctypes.byref(d), _ptr(x, torch.bfloat16, (T, H), "x"),
        _ptr(w_router, torch.float32, (E, H), "w_router"), _ptr(bias, torch.float32, (E,), "bias"),
        _ptr(topk_idx, torch.int32, (T, k), "topk_idx"), _ptr(topk_w, torch.float32, (T, k), "topk_w"),
        _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)))


def moe_route_logits(d: MoeDims, x, w_router, bias, topk_idx, topk_w, logits, ws, stream=None):
    """Router as moe_route, plus the fp32 logits [T, E] the selection was made from."""
    T, H, E, k = d.T, d.H, d.E, d.top_k
    _check("moe_route_logits", native().moe_route_logits(
        ctypes.byref(d), _ptr(x, torch.bfloat16, (T, H), "x"),
        _ptr(w_router, torch.float32, (E, H), "w_router"), _ptr(bias, torch.float32, (E,), "bias"),
        _ptr(topk_idx, torch.int32, (T, k), "topk_idx"), _ptr(topk_w, torch.float32, (T, k), "topk_w"),
        _ptr(logits, torch.float32, (T, E), "logits"),
        _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)))


def moe_permute(d: MoeDims, topk_idx, x, x_perm, expert_offsets, slot_of, row_src, ws, stream=None):
    """Dispatch; fills expert_offsets [E+1], slot_of [T*k], row_src [T*k], x_perm [T*k, H]."""
    T, H, E, Tk = d.T, d.H, d.E, d.T * d.top_k
    _check("moe_permute", native().moe_permute(
        ctypes.byref(d), _ptr(topk_idx, torch.int32, (T, d.top_k), "topk_idx"),
        _ptr(x, torch.bfloat16, (T, H), "x"), _ptr(x_perm, torch.bfloat16, (Tk, H), "x_perm"),
        _ptr(expert_offsets, torch.int32, (E + 1,), "expert_offsets"),
        _ptr(slot_of, torch.int32, (Tk,), "slot_of"), _ptr(row_src, torch.int32, (Tk,), "row_src"),
        _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)))


def moe_experts_swiglu(d: MoeDims, experts: Experts, x_perm, expert_offsets, row_src, topk_w,
                       y_partial, ws, stream=None):
    """Expert SwiGLU MLPs over permuted rows; fills y_partial bf16 [T*k, H]."""
    Tk, H, E = d.T * d.top_k, d.H, d.E
    ex = experts.struct(d)
    _check("moe_experts_swiglu", native().moe_experts_swiglu(
        ctypes.byref(d), ctypes.byref(ex), _ptr(x_perm, torch.bfloat16, (Tk, H), "x_perm"),
        _ptr(expert_offsets, torch.int32, (E + 1,), "expert_offsets"),
        _ptr(row_src, torch.int32, (Tk,), "row_src"),
        _ptr(topk_w, torch.float32, (d.T, d.top_k), "topk_w"),
        _ptr(y_partial, torch.bfloat16, (Tk, H), "y_partial"),
        _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)))


def moe_combine(d: MoeDims, y_partial, slot_of, y, stream=None):
    """Deterministic combine; fills y bf16 [T, H]."""
    Tk, H = d.T * d.top_k, d.H
    _check("moe_combine", native().moe_combine(
        ctypes.byref(d), _ptr(y_partial, torch.bfloat16, (Tk, H), "y_partial"),
        _ptr(slot_of, torch.int32, (Tk,), "slot_of"), _ptr(y, torch.bfloat16, (d.T, H), "y"),
        _stream(stream)))


def moe_forward(d: MoeDims, x, w_router, bias, experts: Experts, y, ws, topk_idx=None, topk_w=None,
                stream=None):
    """The whole block; fills y bf16 [T, H] (and the routing, when given buffers)."""
    T, H, E, k = d.T, d.H, d.E, d.top_k
    ex = experts.struct(d)
    _check("moe_forward", native().moe_forward(
        ctypes.byref(d), _ptr(x, torch.bfloat16, (T, H), "x"),
        _ptr(w_router, torch.float32, (E, H), "w_router"), _ptr(bias, torch.float32, (E,), "bias"),
        ctypes.byref(ex), _ptr(y, torch.bfloat16, (T, H), "y"),
        _ptr(topk_idx, torch.int32, (T, k), "topk_idx"), _ptr(topk_w, torch.float32, (T, k), "topk_w"),
        _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)))


def moe_bias_update(d: MoeDims, topk_idx, bias, gamma_max: float, step: int, total_steps: int,
                    stream=None) -> float:
    """Auxiliary-loss-free bias update, in place on bias fp32 [E]; returns gamma_t."""
    g = ctypes.c_float(0.0)
    _check("moe_bias_update", native().moe_bias_update(
        ctypes.byref(d), _ptr(topk_idx, torch.int32, (d.T, d.top_k), "topk_idx"),
        _ptr(bias, torch.float32, (d.E,), "bias"), float(gamma_max), int(step), int(total_steps),
        ctypes.byref(g), _stream(stream)))
    return g.value


def moe_quantize_nvfp4(x, g: float, q, s, stream=None):
    """NVFP4 quantisation of bf16 rows x [rows, cols] with global scale g:
    fills q uint8 [rows, cols/2] (even column in the low nibble) and
    s uint8 [rows, cols/16] (e4m3 scale codes)."""
    rows, cols = x.shape
    _check("moe_quantize_nvfp4", native().moe_quantize_nvfp4(
        rows, cols, _ptr(x, torch.bfloat16, (rows, cols), "x"), float(g),
        _ptr(q, torch.uint8, (rows, cols // 2), "q"), _ptr(s, torch.uint8, (rows, cols // 16), "s"),
        _stream(stream)))


def moe_pack_bf16(w: torch.Tensor, stream=None) -> torch.Tensor:
    """bf16 expert weights [E, N, K] -> the MMA-tiled layout (same shape and
    dtype; opaque order) for Experts(..., tiled=True)."""
    E, N, K = w.shape
    out = torch.empty_like(w)
    _check("moe_pack_bf16", native().moe_pack_bf16(
        E, N, K, _ptr(w, torch.bfloat16, (E, N, K), "w"), _ptr(out, torch.bfloat16, (E, N, K), "out"),
        _stream(stream)))
    return out


def moe_pack_nvfp4(q: torch.Tensor, s: torch.Tensor, stream=None) -> torch.Tensor:
    """NVFP4 expert weights (codes q uint8 [E, N, K/2], scales s uint8
    [E, N, K/16]) -> the tiled layout, uint8 [E, N, 9K/16] (opaque order),
    for Experts(..., tiled=True, wdtype=MOE_W_NVFP4)."""
    E, N, K2 = q.shape
    K = 2 * K2
    out = torch.empty(E, N, K * 9 // 16, dtype=torch.uint8, device=q.device)
    _check("moe_pack_nvfp4", native().moe_pack_nvfp4(
        E, N, K, _ptr(q, torch.uint8, (E, N, K // 2), "q"), _ptr(s, torch.uint8, (E, N, K // 16), "s"),
        _ptr(out, torch.uint8, (E, N, K * 9 // 16), "out"), _stream(stream)))
    return out


def moe_pack_fp8(q: torch.Tensor, stream=None) -> torch.Tensor:
    """FP8 expert weights (e4m3 codes uint8 [E, N, K]) -> the tiled layout
    (same shape; opaque order) for Experts(..., tiled=True)."""
    E, N, K = q.shape
    out = torch.empty_like(q)
    _check("moe_pack_fp8", native().moe_pack_fp8(
        E, N, K, _ptr(q, torch.uint8, (E, N, K), "q"), _ptr(out, torch.uint8, (E, N, K), "out"),
        _stream(stream)))
    return out


def moe_permute_noalloc(d: MoeDims, topk_idx, x, x_perm, expert_offsets, slot_of, row_src,
                        stream=None):
    """moe_permute without a workspace, for callers that cannot allocate device
    memory (the scratch is a fixed 1 MiB array inside the library; concurrent
    calls race, see include/beam_moe.h)."""
    T, H, E, Tk = d.T, d.H, d.E, d.T * d.top_k
    _check("moe_permute_noalloc", native().moe_permute_noalloc(
        ctypes.byref(d), _ptr(topk_idx, torch.int32, (T, d.top_k), "topk_idx"),
        _ptr(x, torch.bfloat16, (T, H), "x"), _ptr(x_perm, torch.bfloat16, (Tk, H), "x_perm"),
        _ptr(expert_offsets, torch.int32, (E + 1,), "expert_offsets"),
        _ptr(slot_of, torch.int32, (Tk,), "slot_of"), _ptr(row_src, torch.int32, (Tk,), "row_src"),
        _stream(stream)))
