"""ctypes binding of the C ABI in include/attn.h — argument marshalling only.

Every computation happens in the library's CUDA kernels; this module turns
torch tensors into pointers and strides, fills the parameter structs, calls
the entry points and raises on a non-OK status. There is no fallback: if the
shared library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libattn_gb300.so")

ATTN_OK = 0
ATTN_ERR_INVALID = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_ALIGN = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_TIMEOUT = -5
ATTN_ERR_WORKSPACE = -6
ATTN_BF16 = 0
ATTN_F32 = 1
ATTN_F16 = 2
ATTN_E4M3 = 3

STATUS_NAMES = {
    ATTN_OK: "ATTN_OK", ATTN_ERR_INVALID: "ATTN_ERR_INVALID", ATTN_ERR_UNSUPPORTED: "ATTN_ERR_UNSUPPORTED",
    ATTN_ERR_ALIGN: "ATTN_ERR_ALIGN", ATTN_ERR_CUDA: "ATTN_ERR_CUDA", ATTN_ERR_TIMEOUT: "ATTN_ERR_TIMEOUT",
    ATTN_ERR_WORKSPACE: "ATTN_ERR_WORKSPACE",
}

# every symbol include/attn.h declares
EXPORTED = ("attn_fwd", "attn_fwd_fp8", "attn_bwd", "attn_bwd_noalloc", "attn_bwd_deterministic", "attn_bwd_workspace_size",
            "attn_decode",
            "attn_decode_workspace_size", "attn_status", "attn_last_error",
            "attn_set_wait_timeout_ns", "attn_debug_set_producer_stall", "attn_debug_set_bwd_events",
            "attn_debug_launch_count", "attn_debug_launch_name", "attn_version")

_i64x3 = ctypes.c_int64 * 3


class FwdParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32), ("d", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("causal", ctypes.c_int32), ("scale", ctypes.c_float),
        ("reserved0", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("q_stride", _i64x3), ("k_stride", _i64x3), ("v_stride", _i64x3), ("o_stride", _i64x3),
        ("mask", ctypes.c_void_p), ("mask_stride", _i64x3),
    ]


class BwdParams(ctypes.Structure):
    _fields_ = [
        ("fwd", FwdParams),
        ("dout", ctypes.c_void_p), ("do_stride", _i64x3),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dq_stride", _i64x3), ("dk_stride", _i64x3), ("dv_stride", _i64x3),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


class Fp8Params(ctypes.Structure):
    _fields_ = [
        ("f", FwdParams),
        ("q_descale", ctypes.c_float), ("k_descale", ctypes.c_float), ("v_descale", ctypes.c_float),
        ("reserved1", ctypes.c_int32),
    ]


class DecodeParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("nq", ctypes.c_int32), ("nk", ctypes.c_int32),
        ("d", ctypes.c_int32), ("dtype", ctypes.c_int32), ("causal", ctypes.c_int32), ("scale", ctypes.c_float),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("q_stride", _i64x3), ("k_stride", _i64x3), ("v_stride", _i64x3), ("o_stride", _i64x3),
        ("num_splits", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"attention library not built ({LIB_PATH}); run `python -m attn_fwd_03_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    lib.attn_fwd.argtypes = [ctypes.POINTER(FwdParams), ctypes.c_void_p]
    lib.attn_fwd.restype = ctypes.c_int
    lib.attn_fwd_fp8.argtypes = [ctypes.POINTER(Fp8Params), ctypes.c_void_p]
    lib.attn_fwd_fp8.restype = ctypes.c_int
    lib.attn_bwd.argtypes = [ctypes.POINTER(BwdParams), ctypes.c_void_p]
    lib.attn_bwd.restype = ctypes.c_int
    lib.attn_bwd_noalloc.argtypes = [ctypes.POINTER(BwdParams), ctypes.c_void_p]
    lib.attn_bwd_noalloc.restype = ctypes.c_int
    lib.attn_bwd_deterministic.argtypes = [ctypes.POINTER(BwdParams), ctypes.c_void_p]
    lib.attn_bwd_deterministic.restype = ctypes.c_int
    lib.attn_bwd_workspace_size.argtypes = [ctypes.POINTER(FwdParams)]
    lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.attn_decode.argtypes = [ctypes.POINTER(DecodeParams), ctypes.c_void_p]
    lib.attn_decode.restype = ctypes.c_int
    lib.attn_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeParams)]
    lib.attn_decode_workspace_size.restype = ctypes.c_size_t
    lib.attn_status.argtypes = [ctypes.c_void_p]
    lib.attn_status.restype = ctypes.c_int
    lib.attn_last_error.argtypes = []
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.attn_set_wait_timeout_ns.restype = None
    lib.attn_debug_set_producer_stall.argtypes = [ctypes.c_int32]
    lib.attn_debug_set_producer_stall.restype = None
    lib.attn_debug_set_bwd_events.argtypes = [ctypes.c_void_p]
    lib.attn_debug_set_bwd_events.restype = None
    lib.attn_debug_launch_count.argtypes = []
    lib.attn_debug_launch_count.restype = ctypes.c_uint64
    lib.attn_debug_launch_name.argtypes = [ctypes.c_uint32]
    lib.attn_debug_launch_name.restype = ctypes.c_char_p
    lib.attn_version.argtypes = []
    lib.attn_version.restype = ctypes.c_int32
    return lib


lib = _load()


def _check(status: int) -> None:
    if status != ATTN_OK:
        raise AttnError(status, lib.attn_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _strides3(t: torch.Tensor):
    s = t.stride()
    return _i64x3(s[0], s[1], s[2])


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return ATTN_BF16
    if t == torch.float32:
        return ATTN_F32
    if t == torch.float16:
        return ATTN_F16
    if t in (torch.float8_e4m3fn, torch.uint8):
        return ATTN_E4M3
    raise TypeError(f"unsupported dtype {t}")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def fwd_params(q, k, v, o, lse, scale: float, causal: bool, mask: Optional[torch.Tensor]) -> FwdParams:
    """Fill the forward struct from [B, H, N, d] tensors (last dim contiguous)."""
    B, H, N, d = q.shape
    p = FwdParams()
    p.B, p.H, p.N, p.d = B, H, N, d
    p.dtype = _dtype_code(q.dtype)
    p.causal = int(bool(causal))
    p.scale = float(scale)
    p.reserved0 = 0
    p.q, p.k, p.v, p.o, p.lse = _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse)
    p.q_stride, p.k_stride = _strides3(q), _strides3(k)
    p.v_stride, p.o_stride = _strides3(v), _strides3(o)
    if mask is not None:
        m = mask.expand(B, H, N, N)
        p.mask = m.data_ptr()
        p.mask_stride = _strides3(m)
    else:
        p.mask = None
        p.mask_stride = _i64x3(0, 0, 0)
    return p


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: Optional[float] = None,
             causal: bool = False, mask: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O and LSE of exact attention; inputs [B, H, N, d] on the GPU."""
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    p = fwd_params(q, k, v, out, lse, scale, causal, mask)
    _check(lib.attn_fwd(ctypes.byref(p), ctypes.c_void_p(_stream_handle(stream))))
    return out, lse


def attn_fwd_fp8(q, k, v, q_descale: float, k_descale: float, v_descale: float, *,
                 scale: Optional[float] = None, causal: bool = False, mask: Optional[torch.Tensor] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """FP8 forward: q, k, v are [B, H, N, d] (d = 128 or 256) E4M3 tensors (torch.float8_e4m3fn, or
    uint8 holding the codes) standing for code x descale; O is bf16, LSE fp32."""
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    p = Fp8Params()
    p.f = fwd_params(q, k, v, out, lse, scale, causal, mask)
    p.q_descale, p.k_descale, p.v_descale = float(q_descale), float(k_descale), float(v_descale)
    p.reserved1 = 0
    _check(lib.attn_fwd_fp8(ctypes.byref(p), ctypes.c_void_p(_stream_handle(stream))))
    return out, lse


def bwd_workspace_size(q: torch.Tensor) -> int:
    B, H, N, d = q.shape
    p = FwdParams()
    p.B, p.H, p.N, p.d = B, H, N, d
    return int(lib.attn_bwd_workspace_size(ctypes.byref(p)))


def _bwd_call(entry, q, k, v, o, lse, dout, scale, causal, mask, dq, dk, dv, workspace, stream):
    """Fill attn_bwd_params and call `entry` (one of the C backward entry points).
    workspace: a device tensor, None to allocate one here, or False for none (attn_bwd_noalloc)."""
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q, memory_format=torch.contiguous_format) if dq is None else dq
    dk = torch.empty_like(k, memory_format=torch.contiguous_format) if dk is None else dk
    dv = torch.empty_like(v, memory_format=torch.contiguous_format) if dv is None else dv
    bp = BwdParams()
    bp.fwd = fwd_params(q, k, v, o, lse, scale, causal, mask)
    bp.dout, bp.do_stride = _ptr(dout), _strides3(dout)
    bp.dq, bp.dk, bp.dv = _ptr(dq), _ptr(dk), _ptr(dv)
    bp.dq_stride, bp.dk_stride, bp.dv_stride = _strides3(dq), _strides3(dk), _strides3(dv)
    if workspace is False:
        bp.workspace, bp.workspace_bytes = None, 0
    else:
        if workspace is None:
            workspace = torch.empty(max(bwd_workspace_size(q), 1), dtype=torch.uint8, device=q.device)
        bp.workspace = workspace.data_ptr()
        bp.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(entry(ctypes.byref(bp), ctypes.c_void_p(_stream_handle(stream))))
    return dq, dk, dv


def attn_bwd(q, k, v, o, lse, dout, *, scale: Optional[float] = None, causal: bool = False,
             mask: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of sum(dout * O) by recomputation from O and LSE."""
    return _bwd_call(lib.attn_bwd, q, k, v, o, lse, dout, scale, causal, mask, dq, dk, dv, workspace, stream)


def attn_bwd_deterministic(q, k, v, o, lse, dout, *, scale: Optional[float] = None, causal: bool = False,
                           mask: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None, workspace=None,
                           stream=None):
    """attn_bwd with dQ summed over key tiles in a fixed order, so all three
    gradients are the same bits on every call."""
    return _bwd_call(lib.attn_bwd_deterministic, q, k, v, o, lse, dout, scale, causal, mask, dq, dk, dv, workspace,
                     stream)


def attn_bwd_noalloc(q, k, v, o, lse, dout, *, scale: Optional[float] = None, causal: bool = False,
                     mask: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None, stream=None):
    """attn_bwd using the library's built-in 40 MiB scratch instead of a
    workspace, for callers that must not allocate device memory at this point.
    Only the gradient outputs are allocated here (when not given)."""
    return _bwd_call(lib.attn_bwd_noalloc, q, k, v, o, lse, dout, scale, causal, mask, dq, dk, dv, False, stream)


def decode_params(q, k, v, o, lse, scale: float, causal: bool, num_splits: int = 0) -> DecodeParams:
    B, H, nq, d = q.shape
    p = DecodeParams()
    p.B, p.H, p.nq, p.nk, p.d = B, H, nq, k.shape[2], d
    p.dtype = _dtype_code(q.dtype)
    p.causal = 1 if causal else 0
    p.scale = float(scale)
    p.q, p.k, p.v, p.o, p.lse = _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse)
    p.q_stride, p.k_stride, p.v_stride, p.o_stride = _strides3(q), _strides3(k), _strides3(v), _strides3(o)
    p.num_splits = int(num_splits)
    return p


def decode_workspace_size(q, k, v, *, causal: bool = False, num_splits: int = 0) -> int:
    """Bytes of workspace attn_decode needs for these shapes."""
    o = q  # only shapes and strides are read
    lse = q
    return int(lib.attn_decode_workspace_size(ctypes.byref(decode_params(q, k, v, o, lse, 1.0, causal,
                                                                          num_splits))))


def attn_decode(q, k, v, *, scale: Optional[float] = None, causal: bool = False, out=None, lse=None,
                workspace=None, num_splits: int = 0, stream=None):
    """Split-KV decode: q [B, H, nq <= 128, d] against k, v [B, H, nk, d]. With causal the
    queries are the last nq positions. Returns (O, LSE)."""
    B, H, nq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty((B, H, nq, d), dtype=q.dtype, device=q.device) if out is None else out
    lse = torch.empty((B, H, nq), dtype=torch.float32, device=q.device) if lse is None else lse
    p = decode_params(q, k, v, out, lse, scale, causal, num_splits)
    if workspace is None:
        need = int(lib.attn_decode_workspace_size(ctypes.byref(p)))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(lib.attn_decode(ctypes.byref(p), ctypes.c_void_p(_stream_handle(stream))))
    return out, lse


def attn_status(stream=None) -> int:
    """Synchronize and return the status code (does not raise)."""
    return int(lib.attn_status(ctypes.c_void_p(_stream_handle(stream))))


def last_error() -> str:
    return lib.attn_last_error().decode(errors="replace")


def set_wait_timeout_ns(ns: int) -> None:
    lib.attn_set_wait_timeout_ns(int(ns))


def debug_set_producer_stall(kv_tiles: int) -> None:
    lib.attn_debug_set_producer_stall(int(kv_tiles))


def debug_set_bwd_events(events=None) -> None:
    """Time the three backward launches: `events` is four torch.cuda.Event
    objects (already recorded once, so their handles exist) or None."""
    if events is None:
        lib.attn_debug_set_bwd_events(None)
        return
    handles = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
    lib.attn_debug_set_bwd_events(ctypes.cast(handles, ctypes.c_void_p))


def launch_count() -> int:
    """Kernels the library has launched from this host thread so far."""
    return int(lib.attn_debug_launch_count())


def launch_names(count: int):
    """Symbol names of the last `count` (<= 16) kernels launched from this host thread,
    oldest first."""
    names = [lib.attn_debug_launch_name(i) for i in range(count)]
    return [n.decode(errors="replace") if n is not None else None for n in reversed(names)]


def version() -> int:
    return int(lib.attn_version())
