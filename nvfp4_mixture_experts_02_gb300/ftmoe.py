"""Thin ctypes binding of libftmoe.so (include/ft_moe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels. torch supplies device
memory and streams; there is no CPU fallback, and importing this module without the
built library raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libftmoe.so")

FT_OK = 0
STATUS_NAMES = {0: "FT_OK", 1: "FT_ERR_INVALID_ARG", 2: "FT_ERR_UNSUPPORTED_SHAPE",
                3: "FT_ERR_MISALIGNED", 4: "FT_ERR_WORKSPACE_TOO_SMALL", 5: "FT_ERR_CUDA",
                6: "FT_ERR_DEVICE_FLAG", 7: "FT_ERR_TIMEOUT"}

EXPORTED = ["ft_moe_abi_version", "ft_status_string", "ft_moe_route", "ft_moe_workspace_bytes",
            "ft_moe_workspace_init", "ft_moe_nvfp4_decode", "ft_moe_nvfp4_prefill",
            "ft_moe_get_error", "ft_moe_last_cuda_error", "ft_moe_nvfp4_decode_noalloc",
            "ft_moe_nvfp4_decode_routed", "ft_moe_decode_smem_bytes"]


class FtError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        msg = f"{what}: {STATUS_NAMES.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))
        self.status = status


class _Experts(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w13_gscale", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("w2_gscale", ctypes.c_void_p)]


class _Shared(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w13_gscale", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("w2_gscale", ctypes.c_void_p),
                ("gate", ctypes.c_void_p)]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with __graft_entry__.build() "
                          "(nvcc, sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.ft_moe_abi_version.restype = i32
    lib.ft_status_string.restype = ctypes.c_char_p
    lib.ft_status_string.argtypes = [ctypes.c_int]
    lib.ft_moe_route.restype = ctypes.c_int
    lib.ft_moe_route.argtypes = [vp, i32, i32, i32, vp, vp, vp]
    lib.ft_moe_workspace_bytes.restype = sz
    lib.ft_moe_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.ft_moe_decode_smem_bytes.restype = sz
    lib.ft_moe_decode_smem_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.ft_moe_workspace_init.restype = ctypes.c_int
    lib.ft_moe_workspace_init.argtypes = [vp, sz, vp]
    layer = [vp, i32, vp, vp, i32, ctypes.POINTER(_Experts), ctypes.POINTER(_Shared), f32,
             vp, vp, sz, vp]
    for name in ("ft_moe_nvfp4_decode", "ft_moe_nvfp4_prefill"):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = layer
    lib.ft_moe_nvfp4_decode_noalloc.restype = ctypes.c_int
    lib.ft_moe_nvfp4_decode_noalloc.argtypes = layer[:9] + [vp]
    lib.ft_moe_nvfp4_decode_routed.restype = ctypes.c_int
    lib.ft_moe_nvfp4_decode_routed.argtypes = [vp, i32, vp, i32, ctypes.POINTER(_Experts),
                                               ctypes.POINTER(_Shared), f32, vp, vp, vp, vp, sz,
                                               vp]
    lib.ft_moe_last_cuda_error.restype = ctypes.c_char_p
    lib.ft_moe_get_error.restype = ctypes.c_int
    lib.ft_moe_get_error.argtypes = [vp, vp]
    return lib


_LIB = load_library()


def lib() -> ctypes.CDLL:
    return _LIB


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(st: int, what: str):
    if st != FT_OK:
        detail = _LIB.ft_moe_last_cuda_error().decode() if st == 5 else ""
        raise FtError(st, what, detail)


@dataclass
class NvFP4Experts:
    """Routed experts on the device: w13 u8 [E,2I,H/2], s13 u8 [E,2I,H/16], g13 f32 [E],
    w2 u8 [E,H,I/2], s2 u8 [E,H,I/16], g2 f32 [E]."""
    w13: torch.Tensor
    s13: torch.Tensor
    g13: torch.Tensor
    w2: torch.Tensor
    s2: torch.Tensor
    g2: torch.Tensor

    @property
    def E(self):
        return self.w13.shape[0]

    @property
    def H(self):
        return self.w2.shape[1]

    @property
    def I(self):
        return self.w13.shape[1] // 2

    def cstruct(self) -> _Experts:
        return _Experts(self.E, self.H, self.I, _ptr(self.w13), _ptr(self.s13), _ptr(self.g13),
                        _ptr(self.w2), _ptr(self.s2), _ptr(self.g2))


@dataclass
class NvFP4Shared:
    """Shared expert on the device (no E dimension); g13/g2 are 1-element f32 tensors and
    gate is bf16 [H] (any 16-bit dtype holding the bf16 bits)."""
    w13: torch.Tensor
    s13: torch.Tensor
    g13: torch.Tensor
    w2: torch.Tensor
    s2: torch.Tensor
    g2: torch.Tensor
    gate: torch.Tensor

    def cstruct(self) -> _Shared:
        return _Shared(_ptr(self.w13), _ptr(self.s13), _ptr(self.g13), _ptr(self.w2),
                       _ptr(self.s2), _ptr(self.g2), _ptr(self.gate))


def abi_version() -> int:
    return _LIB.ft_moe_abi_version()


def status_string(st: int) -> str:
    return _LIB.ft_status_string(st).decode()


def route(logits: torch.Tensor, k: int, topk_idx=None, topk_w=None, stream=None):
    """ft_moe_route on fp32 logits [T, E] (device). Returns (idx int32 [T,k], w f32 [T,k])."""
    T, E = logits.shape
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    st = _LIB.ft_moe_route(_ptr(logits), T, E, k, _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    _check(st, "ft_moe_route")
    return topk_idx, topk_w


def workspace_bytes(T, k, E, H, I, has_shared, prefill=False) -> int:
    return _LIB.ft_moe_workspace_bytes(T, k, E, H, I, int(bool(has_shared)), int(bool(prefill)))


def new_workspace(T, k, experts: NvFP4Experts, has_shared, prefill=False, device=None,
                  stream=None) -> torch.Tensor:
    n = workspace_bytes(T, k, experts.E, experts.H, experts.I, has_shared, prefill)
    if n == 0 and T == 0:   # an empty batch needs no workspace
        return torch.empty(0, dtype=torch.uint8, device=device or experts.w13.device)
    if n == 0:
        raise FtError(2, "ft_moe_workspace_bytes")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device or experts.w13.device)
    off = (-ws.data_ptr()) % 256                      # 256-byte aligned view
    ws = ws[off:off + n]
    _check(_LIB.ft_moe_workspace_init(_ptr(ws), n, _stream(stream)), "ft_moe_workspace_init")
    return ws


def _layer(fn, name, x, topk_idx, topk_w, experts, shared, limit, out, workspace, stream):
    T = x.shape[0]
    k = topk_idx.shape[1]
    if out is None:
        out = torch.empty((T, experts.H), dtype=torch.bfloat16, device=x.device)
    ex = experts.cstruct()
    sh = shared.cstruct() if shared is not None else None
    st = fn(_ptr(x), T, _ptr(topk_idx), _ptr(topk_w), k, ctypes.byref(ex),
            ctypes.byref(sh) if sh is not None else None, float(limit), _ptr(out),
            _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, name)
    return out


def decode(x, topk_idx, topk_w, experts, shared=None, limit=7.0, out=None, workspace=None,
           stream=None):
    """ft_moe_nvfp4_decode: x bf16 [T,H] (T <= 64) -> out bf16 [T,H]."""
    if workspace is None:
        workspace = new_workspace(x.shape[0], topk_idx.shape[1], experts, shared is not None,
                                  stream=stream)
    return _layer(_LIB.ft_moe_nvfp4_decode, "ft_moe_nvfp4_decode", x, topk_idx, topk_w,
                  experts, shared, limit, out, workspace, stream)


def decode_noalloc(x, topk_idx, topk_w, experts, shared=None, limit=7.0, out=None,
                   stream=None):
    """ft_moe_nvfp4_decode_noalloc: decode with the library's fixed scratch array (no
    workspace, no device allocation by the library)."""
    T, k = x.shape[0], topk_idx.shape[1]
    if out is None:
        out = torch.empty((T, experts.H), dtype=torch.bfloat16, device=x.device)
    ex = experts.cstruct()
    sh = shared.cstruct() if shared is not None else None
    st = _LIB.ft_moe_nvfp4_decode_noalloc(_ptr(x), T, _ptr(topk_idx), _ptr(topk_w), k,
                                          ctypes.byref(ex),
                                          ctypes.byref(sh) if sh is not None else None,
                                          float(limit), _ptr(out), _stream(stream))
    _check(st, "ft_moe_nvfp4_decode_noalloc")
    return out


def decode_routed(x, logits, k, experts, shared=None, limit=7.0, out=None, topk_idx=None,
                  topk_w=None, workspace=None, stream=None):
    """ft_moe_nvfp4_decode_routed: the layer from the router logits f32 [T,E] (T <= 64); one
    launch for T = 1. topk_idx / topk_w (int32 / f32 [T,k]), when given, receive the slots."""
    T = x.shape[0]
    if workspace is None:
        workspace = new_workspace(T, k, experts, shared is not None, stream=stream)
    if out is None:
        out = torch.empty((T, experts.H), dtype=torch.bfloat16, device=x.device)
    ex = experts.cstruct()
    sh = shared.cstruct() if shared is not None else None
    st = _LIB.ft_moe_nvfp4_decode_routed(_ptr(x), T, _ptr(logits), k, ctypes.byref(ex),
                                         ctypes.byref(sh) if sh is not None else None,
                                         float(limit), _ptr(out), _ptr(topk_idx), _ptr(topk_w),
                                         _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "ft_moe_nvfp4_decode_routed")
    return out


def prefill(x, topk_idx, topk_w, experts, shared=None, limit=7.0, out=None, workspace=None,
            stream=None):
    """ft_moe_nvfp4_prefill: x bf16 [T,H] (any T) -> out bf16 [T,H]."""
    if workspace is None:
        workspace = new_workspace(x.shape[0], topk_idx.shape[1], experts, shared is not None,
                                  prefill=True, stream=stream)
    return _layer(_LIB.ft_moe_nvfp4_prefill, "ft_moe_nvfp4_prefill", x, topk_idx, topk_w,
                  experts, shared, limit, out, workspace, stream)


def get_error(workspace, stream=None) -> int:
    return _LIB.ft_moe_get_error(_ptr(workspace), _stream(stream))
