"""Thin ctypes binding of libftmoe.so (include/ft_moe.h): argument checks and marshalling.

Every step of the layer runs in the library's CUDA kernels. torch supplies device
memory and streams; there is no CPU fallback, and importing this module without the
built library raises. Tensors are checked before their pointers are handed over (device,
element type, contiguity, shape): the expert objects once when built, the per-call tensors
on every call.
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
            "ft_moe_nvfp4_decode_routed", "ft_moe_decode_smem_bytes",
            "ft_moe_debug_set_wait_limit", "ft_moe_layer_from_host",
            "ft_moe_fp8block_workspace_bytes", "ft_moe_fp8block_decode",
            "ft_moe_router_logits", "ft_moe_router_route"]

# Leading bytes of a workspace that must be zero before a call (FT_MOE_WORKSPACE_HEAD_BYTES);
# the rest is scratch whose contents never reach an output.
WORKSPACE_HEAD_BYTES = 1024


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


class _F8Experts(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p)]


class _F8Shared(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
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
    lib.ft_moe_layer_from_host.restype = ctypes.c_int
    lib.ft_moe_layer_from_host.argtypes = [vp, vp, i32, i32, ctypes.POINTER(_Experts),
                                           ctypes.POINTER(_Shared), f32, vp, vp, vp, vp, vp, vp,
                                           vp, sz, vp]
    lib.ft_moe_router_logits.restype = ctypes.c_int
    lib.ft_moe_router_logits.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp]
    lib.ft_moe_router_route.restype = ctypes.c_int
    lib.ft_moe_router_route.argtypes = [vp, i32, i32, vp, i32, vp, i32, vp, vp, vp, vp, vp]
    lib.ft_moe_fp8block_workspace_bytes.restype = sz
    lib.ft_moe_fp8block_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.ft_moe_fp8block_decode.restype = ctypes.c_int
    lib.ft_moe_fp8block_decode.argtypes = [vp, i32, vp, vp, i32, ctypes.POINTER(_F8Experts),
                                           ctypes.POINTER(_F8Shared), f32, vp, vp, sz, vp]
    lib.ft_moe_debug_set_wait_limit.restype = ctypes.c_int
    lib.ft_moe_debug_set_wait_limit.argtypes = [ctypes.c_int64]
    return lib


_LIB = load_library()


def lib() -> ctypes.CDLL:
    return _LIB


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream, dev=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    if dev is not None and stream.device_index != dev:
        raise ValueError(f"the tensors are on cuda:{dev}, the stream on cuda:{stream.device_index} "
                         "(torch.cuda.set_device selects the current device)")
    return stream.cuda_stream


def _check(st: int, what: str):
    if st != FT_OK:
        detail = _LIB.ft_moe_last_cuda_error().decode() if st == 5 else ""
        raise FtError(st, what, detail)


# The kernels reach every tensor through its raw pointer, so a host tensor, a narrower
# element type, a strided view or a wrong shape would be read or written out of bounds on
# the GPU. _need refuses those before the call (a few hundred ns per tensor); the expert
# tensors are checked once, when their objects are built.
BF16_BITS = (torch.bfloat16, torch.int16, torch.uint16)   # bf16 values or their bit patterns
_F32 = (torch.float32,)
_I32 = (torch.int32,)


def _need(t, name, dev, dtypes, shape):
    """t on cuda:dev, of one of `dtypes` (None: any 1-byte type), contiguous, of `shape`
    (None: any)."""
    if t.get_device() != dev:
        raise ValueError(f"{name}: expected a tensor on cuda:{dev}, got one on {t.device}")
    if (t.element_size() != 1) if dtypes is None else (t.dtype not in dtypes):
        raise TypeError(f"{name}: element type {t.dtype} is not accepted here")
    if not t.is_contiguous():
        raise ValueError(f"{name}: the tensor must be contiguous")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _need_scalar(t, name, dev):
    _need(t, name, dev, _F32, None)
    if t.numel() != 1:
        raise ValueError(f"{name}: one float32 value expected, got {t.numel()}")


def _device_of(t, what) -> int:
    dev = t.get_device()
    if dev < 0:
        raise ValueError(f"{what}: CUDA tensors are required, got one on {t.device}")
    return dev


@dataclass(frozen=True)
class NvFP4Experts:
    """Routed experts on the device: w13 u8 [E,2I,H/2], s13 u8 [E,2I,H/16], g13 f32 [E],
    w2 u8 [E,H,I/2], s2 u8 [E,H,I/16], g2 f32 [E] (codes and scales: any 1-byte type).
    Checked when built: one device, contiguous, consistent shapes."""
    w13: torch.Tensor
    s13: torch.Tensor
    g13: torch.Tensor
    w2: torch.Tensor
    s2: torch.Tensor
    g2: torch.Tensor

    def __post_init__(self):
        dev = _device_of(self.w13, "NvFP4Experts")
        if self.w13.dim() != 3 or self.w2.dim() != 3:
            raise ValueError("NvFP4Experts: w13 [E,2I,H/2] and w2 [E,H,I/2] are 3-D")
        E, H, I = self.E, self.H, self.I
        _need(self.w13, "w13", dev, None, (E, 2 * I, H // 2))
        _need(self.s13, "s13", dev, None, (E, 2 * I, H // 16))
        _need(self.g13, "g13", dev, _F32, (E,))
        _need(self.w2, "w2", dev, None, (E, H, I // 2))
        _need(self.s2, "s2", dev, None, (E, H, I // 16))
        _need(self.g2, "g2", dev, _F32, (E,))
        object.__setattr__(self, "device_index", dev)
        object.__setattr__(self, "_cs", _Experts(E, H, I, _ptr(self.w13), _ptr(self.s13),
                                                 _ptr(self.g13), _ptr(self.w2), _ptr(self.s2),
                                                 _ptr(self.g2)))

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
        return self._cs


@dataclass(frozen=True)
class NvFP4Shared:
    """Shared expert on the device (no E dimension): w13 [2I,H/2], s13 [2I,H/16], w2 [H,I/2],
    s2 [H,I/16] (any 1-byte type), g13/g2 1-element f32 tensors and gate bf16 [H] (or a
    16-bit integer tensor holding the bf16 bits). Checked when built."""
    w13: torch.Tensor
    s13: torch.Tensor
    g13: torch.Tensor
    w2: torch.Tensor
    s2: torch.Tensor
    g2: torch.Tensor
    gate: torch.Tensor

    def __post_init__(self):
        dev = _device_of(self.w13, "NvFP4Shared")
        if self.w13.dim() != 2 or self.w2.dim() != 2:
            raise ValueError("NvFP4Shared: w13 [2I,H/2] and w2 [H,I/2] are 2-D")
        H, I = self.w2.shape[0], self.w13.shape[0] // 2
        _need(self.w13, "shared w13", dev, None, (2 * I, H // 2))
        _need(self.s13, "shared s13", dev, None, (2 * I, H // 16))
        _need(self.w2, "shared w2", dev, None, (H, I // 2))
        _need(self.s2, "shared s2", dev, None, (H, I // 16))
        _need_scalar(self.g13, "shared g13", dev)
        _need_scalar(self.g2, "shared g2", dev)
        _need(self.gate, "shared gate", dev, BF16_BITS, (H,))
        object.__setattr__(self, "device_index", dev)
        object.__setattr__(self, "H", H)
        object.__setattr__(self, "I", I)
        object.__setattr__(self, "_cs", _Shared(_ptr(self.w13), _ptr(self.s13), _ptr(self.g13),
                                                _ptr(self.w2), _ptr(self.s2), _ptr(self.g2),
                                                _ptr(self.gate)))

    def check_for(self, experts: NvFP4Experts):
        if (self.device_index, self.H, self.I) != (experts.device_index, experts.H, experts.I):
            raise ValueError("shared expert: H, I and the device must match the routed experts")

    def cstruct(self) -> _Shared:
        return self._cs


@dataclass(frozen=True)
class Fp8BlockExperts:
    """Block-FP8 routed experts on the device: w13 u8 [E,2I,H] (E4M3 codes), s13 f32
    [E,2I/128,H/128], w2 u8 [E,H,I], s2 f32 [E,H/128,I/128]. Checked when built."""
    w13: torch.Tensor
    s13: torch.Tensor
    w2: torch.Tensor
    s2: torch.Tensor

    def __post_init__(self):
        dev = _device_of(self.w13, "Fp8BlockExperts")
        if self.w13.dim() != 3 or self.w2.dim() != 3:
            raise ValueError("Fp8BlockExperts: w13 [E,2I,H] and w2 [E,H,I] are 3-D")
        E, H, I = self.w13.shape[0], self.w2.shape[1], self.w13.shape[1] // 2
        t = lambda n: -(-n // 128)
        _need(self.w13, "w13", dev, None, (E, 2 * I, H))
        _need(self.s13, "s13", dev, _F32, (E, t(2 * I), t(H)))
        _need(self.w2, "w2", dev, None, (E, H, I))
        _need(self.s2, "s2", dev, _F32, (E, t(H), t(I)))
        object.__setattr__(self, "device_index", dev)
        object.__setattr__(self, "E", E)
        object.__setattr__(self, "H", H)
        object.__setattr__(self, "I", I)
        object.__setattr__(self, "_cs", _F8Experts(E, H, I, _ptr(self.w13), _ptr(self.s13),
                                                   _ptr(self.w2), _ptr(self.s2)))

    def cstruct(self) -> _F8Experts:
        return self._cs


@dataclass(frozen=True)
class Fp8BlockShared:
    """Block-FP8 shared expert (no E dimension) and its gate vector bf16 [H]."""
    w13: torch.Tensor
    s13: torch.Tensor
    w2: torch.Tensor
    s2: torch.Tensor
    gate: torch.Tensor

    def __post_init__(self):
        dev = _device_of(self.w13, "Fp8BlockShared")
        H, I = self.w2.shape[0], self.w13.shape[0] // 2
        t = lambda n: -(-n // 128)
        _need(self.w13, "shared w13", dev, None, (2 * I, H))
        _need(self.s13, "shared s13", dev, _F32, (t(2 * I), t(H)))
        _need(self.w2, "shared w2", dev, None, (H, I))
        _need(self.s2, "shared s2", dev, _F32, (t(H), t(I)))
        _need(self.gate, "shared gate", dev, BF16_BITS, (H,))
        object.__setattr__(self, "device_index", dev)
        object.__setattr__(self, "H", H)
        object.__setattr__(self, "I", I)
        object.__setattr__(self, "_cs", _F8Shared(_ptr(self.w13), _ptr(self.s13), _ptr(self.w2),
                                                  _ptr(self.s2), _ptr(self.gate)))

    def check_for(self, experts):
        if (self.device_index, self.H, self.I) != (experts.device_index, experts.H, experts.I):
            raise ValueError("shared expert: H, I and the device must match the routed experts")

    def cstruct(self) -> _F8Shared:
        return self._cs


def abi_version() -> int:
    return _LIB.ft_moe_abi_version()


def status_string(st: int) -> str:
    return _LIB.ft_status_string(st).decode()


def route(logits: torch.Tensor, k: int, topk_idx=None, topk_w=None, stream=None):
    """ft_moe_route on fp32 logits [T, E] (device). Returns (idx int32 [T,k], w f32 [T,k])."""
    dev = _device_of(logits, "ft_moe_route")
    if logits.dim() != 2:
        raise ValueError("logits: [T, E] expected")
    _need(logits, "logits", dev, _F32, None)
    T, E = logits.shape
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    else:
        _need(topk_idx, "topk_idx", dev, _I32, (T, k))
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    else:
        _need(topk_w, "topk_w", dev, _F32, (T, k))
    st = _LIB.ft_moe_route(_ptr(logits), T, E, k, _ptr(topk_idx), _ptr(topk_w),
                           _stream(stream, dev))
    _check(st, "ft_moe_route")
    return topk_idx, topk_w


def router_logits(x, w_router, gate=None, logits=None, gate_dot=None, stream=None):
    """ft_moe_router_logits: bf16 x [T,H] and router weights [E,H] (and a bf16 gate [H]) ->
    (logits f32 [T,E], gate dots f32 [T] or None)."""
    dev = _device_of(x, "ft_moe_router_logits")
    if x.dim() != 2 or w_router.dim() != 2:
        raise ValueError("x [T, H] and w_router [E, H] expected")
    T, H = x.shape
    E = w_router.shape[0]
    _need(x, "x", dev, BF16_BITS, (T, H))
    _need(w_router, "w_router", dev, BF16_BITS, (E, H))
    if gate is not None:
        _need(gate, "gate", dev, BF16_BITS, (H,))
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    _need(logits, "logits", dev, _F32, (T, E))
    if gate is not None and gate_dot is None:
        gate_dot = torch.empty((T,), dtype=torch.float32, device=x.device)
    if gate_dot is not None:
        _need(gate_dot, "gate_dot", dev, _F32, (T,))
    st = _LIB.ft_moe_router_logits(_ptr(x), T, H, _ptr(w_router), E, _ptr(gate), _ptr(logits),
                                   _ptr(gate_dot), _stream(stream, dev))
    _check(st, "ft_moe_router_logits")
    return logits, gate_dot


def router_route(x, w_router, k, gate=None, stream=None):
    """ft_moe_router_route: the routing slots (idx int32 [T,k], w f32 [T,k]) from x and the
    router matrix; returns (idx, w, logits, gate dots or None)."""
    dev = _device_of(x, "ft_moe_router_route")
    T, H = x.shape
    E = w_router.shape[0]
    _need(x, "x", dev, BF16_BITS, (T, H))
    _need(w_router, "w_router", dev, BF16_BITS, (E, H))
    if gate is not None:
        _need(gate, "gate", dev, BF16_BITS, (H,))
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    gate_dot = torch.empty((T,), dtype=torch.float32, device=x.device) if gate is not None else None
    idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    st = _LIB.ft_moe_router_route(_ptr(x), T, H, _ptr(w_router), E, _ptr(gate), k, _ptr(logits),
                                  _ptr(gate_dot), _ptr(idx), _ptr(w), _stream(stream, dev))
    _check(st, "ft_moe_router_route")
    return idx, w, logits, gate_dot


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


# Calls made without a workspace share one per (device, stream): launches on one stream run
# in order, so a call never finds its workspace in use by an earlier call that is still
# running. It grows (a new, larger one) when a call needs more; nothing is allocated on
# calls that fit.
_DEFAULT_WS = {}


def default_workspace(T, k, experts: NvFP4Experts, has_shared, prefill=False, stream=None):
    """The workspace a call without one uses: kept per (device, stream) and reused."""
    n = workspace_bytes(T, k, experts.E, experts.H, experts.I, has_shared, prefill)
    if n == 0:
        return new_workspace(T, k, experts, has_shared, prefill, stream=stream)
    if stream is None:
        stream = torch.cuda.current_stream(experts.device_index)
    key = (experts.device_index, stream.cuda_stream)
    ws = _DEFAULT_WS.get(key)
    if ws is None or ws.numel() < n:
        ws = new_workspace(T, k, experts, has_shared, prefill, stream=stream)
        _DEFAULT_WS[key] = ws
    return ws


def _call_tensors(experts, shared, x, out, workspace, T_name="x"):
    """Checks shared by the layer calls: x [T,H] and out [T,H] (bf16 bits), the shared expert
    against the routed ones, the workspace (1-byte elements: numel() is its size in bytes).
    Returns (device, T, out)."""
    dev = experts.device_index
    if x.dim() != 2:
        raise ValueError(f"{T_name}: [T, H] expected")
    T = x.shape[0]
    _need(x, T_name, dev, BF16_BITS, (T, experts.H))
    if shared is not None:
        shared.check_for(experts)
    if out is None:
        out = torch.empty((T, experts.H), dtype=torch.bfloat16, device=x.device)
    else:
        _need(out, "out", dev, BF16_BITS, (T, experts.H))
    if workspace is not None:
        _need(workspace, "workspace", dev, None, None)
    return dev, T, out


def _slots(topk_idx, topk_w, T, dev):
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx: [T, k] expected")
    k = topk_idx.shape[1]
    _need(topk_idx, "topk_idx", dev, _I32, (T, k))
    _need(topk_w, "topk_w", dev, _F32, (T, k))
    return k


def _layer(fn, name, x, topk_idx, topk_w, experts, shared, limit, out, workspace, stream):
    dev, T, out = _call_tensors(experts, shared, x, out, workspace)
    k = _slots(topk_idx, topk_w, T, dev)
    ex = experts.cstruct()
    sh = shared.cstruct() if shared is not None else None
    st = fn(_ptr(x), T, _ptr(topk_idx), _ptr(topk_w), k, ctypes.byref(ex),
            ctypes.byref(sh) if sh is not None else None, float(limit), _ptr(out),
            _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st, name)
    return out


def decode(x, topk_idx, topk_w, experts, shared=None, limit=7.0, out=None, workspace=None,
           stream=None):
    """ft_moe_nvfp4_decode: x bf16 [T,H] (T <= 64) -> out bf16 [T,H]."""
    if workspace is None:
        workspace = default_workspace(x.shape[0], topk_idx.shape[1], experts, shared is not None,
                                      stream=stream)
    return _layer(_LIB.ft_moe_nvfp4_decode, "ft_moe_nvfp4_decode", x, topk_idx, topk_w,
                  experts, shared, limit, out, workspace, stream)


def decode_noalloc(x, topk_idx, topk_w, experts, shared=None, limit=7.0, out=None,
                   stream=None):
    """ft_moe_nvfp4_decode_noalloc: decode with the library's fixed scratch array (no
    workspace, no device allocation by the library)."""
    dev, T, out = _call_tensors(experts, shared, x, out, None)
    k = _slots(topk_idx, topk_w, T, dev)
    ex = experts.cstruct()
    sh = shared.cstruct() if shared is not None else None
    st = _LIB.ft_moe_nvfp4_decode_noalloc(_ptr(x), T, _ptr(topk_idx), _ptr(topk_w), k,
                                          ctypes.byref(ex),
                                          ctypes.byref(sh) if sh is not None else None,
                                          float(limit), _ptr(out), _stream(stream, dev))
    _check(st, "ft_moe_nvfp4_decode_noalloc")
    return out


def decode_routed(x, logits, k, experts, shared=None, limit=7.0, out=None, topk_idx=None,
                  topk_w=None, workspace=None, stream=None):
    """ft_moe_nvfp4_decode_routed: the layer from the router logits f32 [T,E] (T <= 64); one
    launch for T = 1. topk_idx / topk_w (int32 / f32 [T,k]), when given, receive the slots."""
    if workspace is None:
        workspace = default_workspace(x.shape[0], k, experts, shared is not None, stream=stream)
    dev, T, out = _call_tensors(experts, shared, x, out, workspace)
    _need(logits, "logits", dev, _F32, (T, experts.E))
    if topk_idx is not None:
        _need(topk_idx, "topk_idx", dev, _I32, (T, k))
    if topk_w is not None:
        _need(topk_w, "topk_w", dev, _F32, (T, k))
    ex = experts.cstruct()
    sh = shared.cstruct() if shared is not None else None
    st = _LIB.ft_moe_nvfp4_decode_routed(_ptr(x), T, _ptr(logits), k, ctypes.byref(ex),
                                         ctypes.byref(sh) if sh is not None else None,
                                         float(limit), _ptr(out), _ptr(topk_idx), _ptr(topk_w),
                                         _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st, "ft_moe_nvfp4_decode_routed")
    return out


def prefill(x, topk_idx, topk_w, experts, shared=None, limit=7.0, out=None, workspace=None,
            stream=None):
    """ft_moe_nvfp4_prefill: x bf16 [T,H] (any T) -> out bf16 [T,H]."""
    if workspace is None:
        workspace = default_workspace(x.shape[0], topk_idx.shape[1], experts, shared is not None,
                                      prefill=True, stream=stream)
    return _layer(_LIB.ft_moe_nvfp4_prefill, "ft_moe_nvfp4_prefill", x, topk_idx, topk_w,
                  experts, shared, limit, out, workspace, stream)


def _need_host(t, name, dtypes, shape):
    if t.device.type != "cpu":
        raise ValueError(f"{name}: expected a host tensor, got one on {t.device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: element type {t.dtype} is not accepted here")
    if not t.is_contiguous():
        raise ValueError(f"{name}: the tensor must be contiguous")
    if t.shape != shape:
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def layer_from_host(x_host, logits_host, k, experts, shared=None, limit=7.0, out_host=None,
                    x_dev=None, logits_dev=None, out_dev=None, topk_idx_dev=None,
                    topk_w_dev=None, workspace=None, stream=None):
    """ft_moe_layer_from_host: x bf16 [T,H] and logits f32 [T,E] in host memory (pinned for
    asynchronous copies) -> out_host bf16 [T,H], with the device buffers given (or made
    here). Everything is enqueued on the stream; the host output is ready once it is
    synchronised. Returns out_host."""
    dev = experts.device_index
    if x_host.dim() != 2:
        raise ValueError("x_host: [T, H] expected")
    T, H, E = x_host.shape[0], experts.H, experts.E
    _need_host(x_host, "x_host", BF16_BITS, (T, H))
    _need_host(logits_host, "logits_host", _F32, (T, E))
    if out_host is None:
        out_host = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    else:
        _need_host(out_host, "out_host", BF16_BITS, (T, H))
    if shared is not None:
        shared.check_for(experts)
    cuda = torch.device("cuda", dev)
    x_dev = torch.empty((T, H), dtype=torch.bfloat16, device=cuda) if x_dev is None else x_dev
    logits_dev = (torch.empty((T, E), dtype=torch.float32, device=cuda) if logits_dev is None
                  else logits_dev)
    out_dev = torch.empty((T, H), dtype=torch.bfloat16, device=cuda) if out_dev is None else out_dev
    _need(x_dev, "x_dev", dev, BF16_BITS, (T, H))
    _need(logits_dev, "logits_dev", dev, _F32, (T, E))
    _need(out_dev, "out_dev", dev, BF16_BITS, (T, H))
    prefill = T > 64
    if prefill and topk_idx_dev is None:
        topk_idx_dev = torch.empty((T, k), dtype=torch.int32, device=cuda)
    if prefill and topk_w_dev is None:
        topk_w_dev = torch.empty((T, k), dtype=torch.float32, device=cuda)
    if topk_idx_dev is not None:
        _need(topk_idx_dev, "topk_idx_dev", dev, _I32, (T, k))
    if topk_w_dev is not None:
        _need(topk_w_dev, "topk_w_dev", dev, _F32, (T, k))
    if workspace is None:
        workspace = default_workspace(T, k, experts, shared is not None, prefill=prefill,
                                      stream=stream)
    _need(workspace, "workspace", dev, None, None)
    ex = experts.cstruct()
    sh = shared.cstruct() if shared is not None else None
    st = _LIB.ft_moe_layer_from_host(_ptr(x_host), _ptr(logits_host), T, k, ctypes.byref(ex),
                                     ctypes.byref(sh) if sh is not None else None, float(limit),
                                     _ptr(out_host), _ptr(x_dev), _ptr(logits_dev),
                                     _ptr(topk_idx_dev), _ptr(topk_w_dev), _ptr(out_dev),
                                     _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st, "ft_moe_layer_from_host")
    return out_host


def fp8block_workspace_bytes(T, k, E, H, I, has_shared) -> int:
    return _LIB.ft_moe_fp8block_workspace_bytes(T, k, E, H, I, int(bool(has_shared)))


def new_fp8block_workspace(T, k, experts: Fp8BlockExperts, has_shared, stream=None):
    n = fp8block_workspace_bytes(T, k, experts.E, experts.H, experts.I, has_shared)
    if n == 0:
        raise FtError(2, "ft_moe_fp8block_workspace_bytes")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=experts.w13.device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    _check(_LIB.ft_moe_workspace_init(_ptr(ws), n, _stream(stream)), "ft_moe_workspace_init")
    return ws


def fp8block_decode(x, topk_idx, topk_w, experts: Fp8BlockExperts, shared=None, limit=7.0,
                    out=None, workspace=None, stream=None):
    """ft_moe_fp8block_decode: x bf16 [T,H] (T <= 64) with block-FP8 experts -> out bf16
    [T,H]."""
    if workspace is None:
        workspace = new_fp8block_workspace(x.shape[0], topk_idx.shape[1], experts,
                                           shared is not None, stream=stream)
    dev, T, out = _call_tensors(experts, shared, x, out, workspace)
    k = _slots(topk_idx, topk_w, T, dev)
    ex = experts.cstruct()
    sh = shared.cstruct() if shared is not None else None
    st = _LIB.ft_moe_fp8block_decode(_ptr(x), T, _ptr(topk_idx), _ptr(topk_w), k,
                                     ctypes.byref(ex), ctypes.byref(sh) if sh is not None else None,
                                     float(limit), _ptr(out), _ptr(workspace), workspace.numel(),
                                     _stream(stream, dev))
    _check(st, "ft_moe_fp8block_decode")
    return out


def get_error(workspace, stream=None) -> int:
    dev = _device_of(workspace, "ft_moe_get_error")
    return _LIB.ft_moe_get_error(_ptr(workspace), _stream(stream, dev))


def debug_set_wait_limit(iterations: int | None):
    """Test hook: how often a decode kernel polls for the other CTAs' results before it
    flags FT_ERR_TIMEOUT and goes on (None: the default bound)."""
    _check(_LIB.ft_moe_debug_set_wait_limit(-1 if iterations is None else int(iterations)),
           "ft_moe_debug_set_wait_limit")
