"""liboss: online-softmax row softmax, fused attention forward, split-KV
decode and the (m, l, O) merge on one GB300 (sm_103a).

This module is the thin Python binding over the C ABI in ``include/oss.h``:
it checks tensor dtypes and devices, allocates outputs with PyTorch, passes
raw device pointers and the current CUDA stream to ``liboss.so`` and turns a
non-OK status into an exception. Every step of the computation runs in the
library's CUDA kernels; there is no CPU fallback, and a missing library is an
error.
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

__all__ = [
    "OssError",
    "library_path",
    "load",
    "softmax_rows",
    "softmax_rows_from_host",
    "softmax_rows_multipass",
    "softmax_rows_16bit",
    "softmax_rows_workspace_bytes",
    "attention_fwd",
    "attention_fwd_from_host",
    "attention_fwd_partial",
    "attention_fwd_workspace_bytes",
    "attention_decode_splitkv",
    "merge_partials",
    "decode_from_host",
    "check_device_error",
    "debug_inject_fault",
    "set_rescale_policy",
    "rescale_policy",
    "RESCALE_POLICIES",
    "abi_version",
    "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboss.so")

OS_OK = 0
STATUS_NAMES = {
    0: "OS_OK",
    1: "OS_ERR_INVALID_ARGUMENT",
    2: "OS_ERR_MISALIGNED",
    3: "OS_ERR_UNSUPPORTED",
    4: "OS_ERR_CUDA",
    5: "OS_ERR_TIMEOUT",
}

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float

# name -> (restype, argtypes), the signatures of include/oss.h
_SIGNATURES = {
    "os_softmax_rows": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _vp]),
    "os_softmax_rows_16bit": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _i32, _vp]),
    "os_softmax_rows_ws": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _vp, _i64, _vp]),
    "os_softmax_rows_16bit_ws": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _i32, _vp,
                                        _i64, _vp]),
    "os_softmax_rows_workspace_bytes": (_i64, [_i64, _i64, _i32]),
    "os_softmax_rows_from_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i64,
                                         _vp]),
    "os_softmax_rows_multipass": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _i32,
                                         _vp]),
    "os_attention_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32,
                                ctypes.c_int, _vp]),
    "os_attention_fwd_ws": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32,
                                   ctypes.c_int, _vp, _i64, _vp]),
    "os_attention_fwd_workspace_bytes": (_i64, [_i32, _i32, _i32, _i32, _i32, ctypes.c_int]),
    "os_attention_fwd_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                        _f32, ctypes.c_int, _vp]),
    "os_attention_fwd_partial": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32,
                                        ctypes.c_int, _vp, _vp, _vp, _i32, _i32, _vp]),
    "os_attention_decode_splitkv": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                           _f32, _vp, _vp, _vp, _vp]),
    "os_merge_partials": (_i32, [_vp, _vp, _vp, _i64, _i32, _i32, ctypes.c_int, _vp, _vp, _vp,
                                 _vp, _vp]),
    "os_check_device_error": (_i32, [_vp, ctypes.POINTER(_i32)]),
    "os_attention_set_rescale_policy": (_i32, [_i32]),
    "os_attention_rescale_policy": (_i32, []),
    "os_debug_inject_fault": (_i32, [_i32, _i32, _i64]),
    "os_status_string": (ctypes.c_char_p, [_i32]),
    "os_abi_version": (_i32, []),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib: Optional[ctypes.CDLL] = None


class OssError(RuntimeError):
    """A liboss call returned a non-OK status."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)}")


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load liboss.so (built by ``pass_attention_gb300.build_lib``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"liboss is not built ({_LIB_PATH} is missing); build it with "
                "`python -m pass_attention_gb300.build_lib`")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def abi_version() -> int:
    return int(load().os_abi_version())


def _check(status: int, where: str) -> None:
    if status != OS_OK:
        raise OssError(status, where)


def _stream_ptr(stream, device: torch.device) -> int:
    """The CUDA stream to enqueue on: ``stream``, else the current stream of
    the inputs' device. A stream of another device is refused."""
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return stream.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (liboss has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")


def _dense(t: torch.Tensor, name: str) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _same_device(device: torch.device, **tensors) -> None:
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, the inputs on {device}")


def _out(t, name: str, dtype: torch.dtype, shape, device: torch.device) -> torch.Tensor:
    """A caller-supplied output: a dense CUDA tensor of exactly this dtype and
    shape on the inputs' device (the kernels write every element of it and
    nothing around it, so a short, strided, host or foreign-device buffer is
    refused before the library is called)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (liboss has no CPU path)")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the inputs on {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# Workspaces of the *_ws entry points, one per (device, stream, kind): calls
# on one stream run one after another and may share one; calls on other
# streams get their own. Each is zero-filled when made, and the calls leave
# what must start at zero at zero again.
_WORKSPACES: dict = {}


def _workspace(device: torch.device, stream_ptr: int, nbytes: int, kind: str = "attn") -> torch.Tensor:
    key = (device.index, stream_ptr, kind)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws


# ---------------------------------------------------------------------------
# os_softmax_rows
# ---------------------------------------------------------------------------

def softmax_rows_workspace_bytes(rows: int, cols: int, dtype=torch.float32) -> int:
    """Workspace bytes os_softmax_rows_ws uses for such rows (0: none)."""
    code = 0 if dtype == torch.float32 else _DTYPE_CODES[dtype]
    n = int(load().os_softmax_rows_workspace_bytes(int(rows), int(cols), code))
    if n < 0:
        raise OssError(4, "os_softmax_rows_workspace_bytes")
    return n

def softmax_rows(x: torch.Tensor, scale: float = 1.0, y: Optional[torch.Tensor] = None,
                 m: Optional[torch.Tensor] = None, l: Optional[torch.Tensor] = None,
                 stream=None):
    """Row softmax of ``scale * x`` (fp32 [rows, cols], unit column stride).

    Returns ``(y, m, l)``; see ``os_softmax_rows`` in include/oss.h.
    """
    _need(x, "x", torch.float32, 2)
    if x.stride(1) != 1:
        raise ValueError("x must have unit column stride")
    rows, cols = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, 2)
    _same_device(dev, y=y)
    if y.stride(1) != 1 or tuple(y.shape) != (rows, cols):
        raise ValueError("y must be [rows, cols] with unit column stride")
    m = _out(torch.empty(rows, dtype=torch.float32, device=dev) if m is None else m,
             "m", torch.float32, (rows,), dev)
    l = _out(torch.empty(rows, dtype=torch.float32, device=dev) if l is None else l,
             "l", torch.float32, (rows,), dev)
    with torch.cuda.device(dev):
        sp = _stream_ptr(stream, dev)
        need = softmax_rows_workspace_bytes(rows, cols)
        ws = _workspace(dev, sp, need, "rows") if need > 0 else None
        st = load().os_softmax_rows_ws(x.data_ptr(), y.data_ptr(), m.data_ptr(), l.data_ptr(), rows,
                                       cols, x.stride(0), y.stride(0), float(scale), _ptr(ws),
                                       need if ws is not None else 0, sp)
    _check(st, "os_softmax_rows_ws")
    return y, m, l


_DTYPE_CODES = {torch.bfloat16: 1, torch.float16: 2}


def softmax_rows_16bit(x: torch.Tensor, scale: float = 1.0, y: Optional[torch.Tensor] = None,
                       m: Optional[torch.Tensor] = None, l: Optional[torch.Tensor] = None,
                       stream=None):
    """Row softmax of ``scale * x`` for bf16 or fp16 rows ([rows, cols], unit
    column stride); y has x's type, m and l are fp32. See
    ``os_softmax_rows_16bit``."""
    if not isinstance(x, torch.Tensor) or x.dtype not in _DTYPE_CODES:
        raise TypeError("x must be a bfloat16 or float16 torch.Tensor")
    _need(x, "x", x.dtype, 2)
    if x.stride(1) != 1:
        raise ValueError("x must have unit column stride")
    rows, cols = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((rows, cols), dtype=x.dtype, device=dev)
    _need(y, "y", x.dtype, 2)
    _same_device(dev, y=y)
    if y.stride(1) != 1 or tuple(y.shape) != (rows, cols):
        raise ValueError("y must be [rows, cols] with unit column stride")
    m = _out(torch.empty(rows, dtype=torch.float32, device=dev) if m is None else m,
             "m", torch.float32, (rows,), dev)
    l = _out(torch.empty(rows, dtype=torch.float32, device=dev) if l is None else l,
             "l", torch.float32, (rows,), dev)
    with torch.cuda.device(dev):
        sp = _stream_ptr(stream, dev)
        need = softmax_rows_workspace_bytes(rows, cols, x.dtype)
        ws = _workspace(dev, sp, need, "rows") if need > 0 else None
        st = load().os_softmax_rows_16bit_ws(x.data_ptr(), y.data_ptr(), m.data_ptr(), l.data_ptr(),
                                             rows, cols, x.stride(0), y.stride(0), float(scale),
                                             _DTYPE_CODES[x.dtype], _ptr(ws),
                                             need if ws is not None else 0, sp)
    _check(st, "os_softmax_rows_16bit_ws")
    return y, m, l


def softmax_rows_multipass(x: torch.Tensor, passes: int, scale: float = 1.0,
                           y: Optional[torch.Tensor] = None, m: Optional[torch.Tensor] = None,
                           l: Optional[torch.Tensor] = None, stream=None):
    """The 2- or 3-pass comparator of softmax_rows (same outputs; x is read
    from HBM ``passes`` times). See ``os_softmax_rows_multipass``."""
    _need(x, "x", torch.float32, 2)
    if x.stride(1) != 1:
        raise ValueError("x must have unit column stride")
    rows, cols = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, 2)
    _same_device(dev, y=y)
    if y.stride(1) != 1 or tuple(y.shape) != (rows, cols):
        raise ValueError("y must be [rows, cols] with unit column stride")
    m = _out(torch.empty(rows, dtype=torch.float32, device=dev) if m is None else m,
             "m", torch.float32, (rows,), dev)
    l = _out(torch.empty(rows, dtype=torch.float32, device=dev) if l is None else l,
             "l", torch.float32, (rows,), dev)
    with torch.cuda.device(dev):
        st = load().os_softmax_rows_multipass(x.data_ptr(), y.data_ptr(), m.data_ptr(),
                                              l.data_ptr(), rows, cols, x.stride(0), y.stride(0),
                                              float(scale), int(passes), _stream_ptr(stream, dev))
    _check(st, "os_softmax_rows_multipass")
    return y, m, l


def softmax_rows_from_host(x_host: torch.Tensor, scale: float = 1.0, out=None, device="cuda",
                           chunk_rows: Optional[int] = None, x_dev: Optional[torch.Tensor] = None,
                           y_dev: Optional[torch.Tensor] = None):
    """End-to-end call on host memory through os_softmax_rows_from_host: the
    library copies x to the GPU, runs the row softmax and copies y, m and l
    back into (pinned) host tensors, in blocks of ``chunk_rows`` rows (default:
    about 64 MiB of x a block) whose upload, kernel and download overlap.
    Returns host (y, m, l) once the stream has finished them. ``x_dev`` /
    ``y_dev`` are optional device buffers of x's shape to reuse across calls."""
    if not isinstance(x_host, torch.Tensor) or x_host.dim() != 2 or x_host.dtype != torch.float32 \
            or x_host.is_cuda:
        raise ValueError("x_host must be a 2-D float32 host tensor")
    _dense(x_host, "x_host")
    rows, cols = x_host.shape
    dev = torch.device(device)
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = (torch.empty((rows, cols), dtype=torch.float32, pin_memory=True),
               torch.empty(rows, dtype=torch.float32, pin_memory=True),
               torch.empty(rows, dtype=torch.float32, pin_memory=True))
    y_host, m_host, l_host = out
    for name, t, shape in (("y_host", y_host, (rows, cols)), ("m_host", m_host, (rows,)),
                           ("l_host", l_host, (rows,))):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.float32 \
                or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a dense float32 host tensor of shape {shape}")
    x_dev = torch.empty((rows, cols), dtype=torch.float32, device=dev) if x_dev is None \
        else _out(x_dev, "x_dev", torch.float32, (rows, cols), dev)
    y_dev = torch.empty((rows, cols), dtype=torch.float32, device=dev) if y_dev is None \
        else _out(y_dev, "y_dev", torch.float32, (rows, cols), dev)
    m_dev = torch.empty(rows, dtype=torch.float32, device=dev)
    l_dev = torch.empty(rows, dtype=torch.float32, device=dev)
    if chunk_rows is not None and chunk_rows < 1:
        raise ValueError("chunk_rows must be at least 1")
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        st = load().os_softmax_rows_from_host(
            x_host.data_ptr(), y_host.data_ptr(), m_host.data_ptr(), l_host.data_ptr(),
            x_dev.data_ptr(), y_dev.data_ptr(), m_dev.data_ptr(), l_dev.data_ptr(), rows, cols,
            ctypes.c_float(scale), 0 if chunk_rows is None else int(chunk_rows), stream.cuda_stream)
        _check(st, "os_softmax_rows_from_host")
        stream.synchronize()
    return out


# ---------------------------------------------------------------------------
# os_attention_fwd
# ---------------------------------------------------------------------------

def attention_fwd_workspace_bytes(B: int, H: int, Sq: int, Sk: int, D: int = 128,
                                  causal: bool = False) -> int:
    """Workspace bytes os_attention_fwd_ws uses for this shape on the current
    device (0: none)."""
    n = int(load().os_attention_fwd_workspace_bytes(B, H, Sq, Sk, D, int(bool(causal))))
    if n < 0:
        raise OssError(4, "os_attention_fwd_workspace_bytes")
    return n


def attention_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  scale: Optional[float] = None, causal: bool = False,
                  o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  stream=None):
    """Fused attention forward on bf16 [B, H, S, D] tensors.

    Returns ``(o, lse)``; see ``os_attention_fwd`` in include/oss.h.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
        _dense(t, n)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if tuple(k.shape) != (B, H, Sk, D) or tuple(v.shape) != (B, H, Sk, D):
        raise ValueError("k and v must be [B, H, Sk, D] matching q")
    dev = q.device
    _same_device(dev, k=k, v=v)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = _out(torch.empty_like(q) if o is None else o, "o", torch.bfloat16, q.shape, dev)
    lse = _out(torch.empty((B, H, Sq), dtype=torch.float32, device=dev) if lse is None else lse,
               "lse", torch.float32, (B, H, Sq), dev)
    with torch.cuda.device(dev):
        sp = _stream_ptr(stream, dev)
        need = attention_fwd_workspace_bytes(B, H, Sq, Sk, D, causal)
        ws = _workspace(dev, sp, need, "attn") if need > 0 else None
        st = load().os_attention_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), B, H, Sq, Sk, D, float(scale),
                                        int(bool(causal)), _ptr(ws), need if ws is not None else 0,
                                        sp)
    _check(st, "os_attention_fwd_ws")
    return o, lse


def attention_fwd_partial(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                          part_m: torch.Tensor, part_l: torch.Tensor, part_o: torch.Tensor,
                          index: int, scale: Optional[float] = None, causal: bool = False,
                          stream=None):
    """Partial softmax states of q against one shard k, v (bf16 [B, H, S, D]).

    part_m, part_l: fp32 [B, H, Sq, S_shards]; part_o: fp32 [B, H, Sq,
    S_shards, D]; writes slot ``index``. See ``os_attention_fwd_partial``.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
        _dense(t, n)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if tuple(k.shape) != (B, H, Sk, D) or tuple(v.shape) != (B, H, Sk, D):
        raise ValueError("k and v must be [B, H, Sk, D] matching q")
    dev = q.device
    _same_device(dev, k=k, v=v)
    _need(part_m, "part_m", torch.float32, 4)
    stride = part_m.shape[-1]
    _out(part_m, "part_m", torch.float32, (B, H, Sq, stride), dev)
    _out(part_l, "part_l", torch.float32, (B, H, Sq, stride), dev)
    _out(part_o, "part_o", torch.float32, (B, H, Sq, stride, D), dev)
    if not 0 <= int(index) < stride:
        raise ValueError(f"index {index} outside the {stride} partial slots")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(dev):
        st = load().os_attention_fwd_partial(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, H, Sq,
                                             Sk, D, float(scale), int(bool(causal)),
                                             part_m.data_ptr(), part_l.data_ptr(),
                                             part_o.data_ptr(), stride, int(index),
                                             _stream_ptr(stream, dev))
    _check(st, "os_attention_fwd_partial")


def attention_fwd_from_host(q_host, k_host, v_host, scale=None, causal=False, out=None,
                            device="cuda"):
    """End-to-end call on host memory: copy q, k, v to the GPU, run
    os_attention_fwd, copy o and lse back. Returns host (o, lse)."""
    q, k, v = (t.to(device, non_blocking=True) for t in (q_host, k_host, v_host))
    o, lse = attention_fwd(q, k, v, scale, causal)
    if out is None:
        out = (torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
               torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True))
    out[0].copy_(o, non_blocking=True)
    out[1].copy_(lse, non_blocking=True)
    torch.cuda.current_stream().synchronize()
    return out


# ---------------------------------------------------------------------------
# os_attention_decode_splitkv / os_merge_partials
# ---------------------------------------------------------------------------

def attention_decode_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                             kv_len: torch.Tensor, num_splits: int,
                             scale: Optional[float] = None, part_m=None, part_l=None,
                             part_o=None, stream=None):
    """Split-KV decode partials. q [B, H, D], k/v [B, H, Lmax, D] bf16,
    kv_len [B] int32 (device). Returns ``(part_m, part_l, part_o)``."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    _need(kv_len, "kv_len", torch.int32, 1)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (kv_len, "kv_len")):
        _dense(t, n)
    B, H, D = q.shape
    Lmax = k.shape[2]
    if tuple(k.shape) != (B, H, Lmax, D) or tuple(v.shape) != (B, H, Lmax, D):
        raise ValueError("k and v must be [B, H, Lmax, D] matching q")
    if kv_len.numel() != B:
        raise ValueError("kv_len must have B entries")
    dev = q.device
    _same_device(dev, k=k, v=v, kv_len=kv_len)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    S = int(num_splits)
    if S < 1:
        raise ValueError("num_splits must be >= 1")
    part_m = _out(torch.empty((B, H, S), dtype=torch.float32, device=dev) if part_m is None
                  else part_m, "part_m", torch.float32, (B, H, S), dev)
    part_l = _out(torch.empty((B, H, S), dtype=torch.float32, device=dev) if part_l is None
                  else part_l, "part_l", torch.float32, (B, H, S), dev)
    part_o = _out(torch.empty((B, H, S, D), dtype=torch.float32, device=dev) if part_o is None
                  else part_o, "part_o", torch.float32, (B, H, S, D), dev)
    with torch.cuda.device(dev):
        st = load().os_attention_decode_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                kv_len.data_ptr(), B, H, Lmax, D, S, float(scale),
                                                part_m.data_ptr(), part_l.data_ptr(),
                                                part_o.data_ptr(), _stream_ptr(stream, dev))
    _check(st, "os_attention_decode_splitkv")
    return part_m, part_l, part_o


def merge_partials(part_m: torch.Tensor, part_l: torch.Tensor, part_o: torch.Tensor,
                   finalize: bool = True, o_out=None, m_out=None, l_out=None, lse_out=None,
                   stream=None):
    """Merge partials over their split axis. part_m/part_l [..., S],
    part_o [..., S, D] fp32. Returns ``(o, m, l, lse)`` with o bf16 [..., D]
    (finalize) or fp32 [..., D] (unnormalised, finalize=False)."""
    for t, n in ((part_m, "part_m"), (part_l, "part_l"), (part_o, "part_o")):
        if not t.is_cuda or t.dtype != torch.float32:
            raise TypeError(f"{n} must be a CUDA float32 tensor")
        _dense(t, n)
    lead = tuple(part_m.shape[:-1])
    S = part_m.shape[-1]
    D = part_o.shape[-1]
    if tuple(part_l.shape) != tuple(part_m.shape) or tuple(part_o.shape) != lead + (S, D):
        raise ValueError("partials must be [..., S] and [..., S, D]")
    groups = 1
    for n in lead:
        groups *= n
    dev = part_m.device
    _same_device(dev, part_l=part_l, part_o=part_o)
    o_dtype = torch.bfloat16 if finalize else torch.float32
    o_out = _out(torch.empty(lead + (D,), dtype=o_dtype, device=dev) if o_out is None else o_out,
                 "o_out", o_dtype, lead + (D,), dev)
    m_out = _out(torch.empty(lead, dtype=torch.float32, device=dev) if m_out is None else m_out,
                 "m_out", torch.float32, lead, dev)
    l_out = _out(torch.empty(lead, dtype=torch.float32, device=dev) if l_out is None else l_out,
                 "l_out", torch.float32, lead, dev)
    lse_out = _out(torch.empty(lead, dtype=torch.float32, device=dev) if lse_out is None
                   else lse_out, "lse_out", torch.float32, lead, dev)
    with torch.cuda.device(dev):
        st = load().os_merge_partials(part_m.data_ptr(), part_l.data_ptr(), part_o.data_ptr(),
                                      groups, S, D, int(bool(finalize)), o_out.data_ptr(),
                                      _ptr(m_out), _ptr(l_out), _ptr(lse_out),
                                      _stream_ptr(stream, dev))
    _check(st, "os_merge_partials")
    return o_out, m_out, l_out, lse_out


def decode_from_host(q_host, k_host, v_host, kv_len_host, num_splits, scale=None, out=None,
                     device="cuda"):
    """End-to-end split-KV decode on host memory: copy inputs to the GPU, run
    the decode partials and the merge, copy o and lse back."""
    q, k, v, kv = (t.to(device, non_blocking=True) for t in (q_host, k_host, v_host, kv_len_host))
    pm, pl, po = attention_decode_splitkv(q, k, v, kv, num_splits, scale)
    o, _, _, lse = merge_partials(pm, pl, po, finalize=True)
    if out is None:
        out = (torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
               torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True))
    out[0].copy_(o, non_blocking=True)
    out[1].copy_(lse, non_blocking=True)
    torch.cuda.current_stream().synchronize()
    return out


RESCALE_POLICIES = {"threshold": 0, "on_rise": 1, "always": 2}


def set_rescale_policy(policy) -> None:
    """Rescale policy of this thread's later attention calls: "threshold"
    (default), "on_rise" or "always" (or the os_rescale_policy value). See
    ``os_attention_set_rescale_policy``."""
    code = RESCALE_POLICIES.get(policy, policy)
    _check(load().os_attention_set_rescale_policy(int(code)), "os_attention_set_rescale_policy")


def rescale_policy() -> str:
    code = int(load().os_attention_rescale_policy())
    return {v: k for k, v in RESCALE_POLICIES.items()}[code]


def debug_inject_fault(kind: int, step: int = 0, timeout_ns: int = 0) -> None:
    """Test hook: arm a fault for the next attention_fwd call (kind 1) or
    row softmax call (kind 2) on this thread; kind 0 disarms (see
    ``os_debug_inject_fault`` in include/oss.h)."""
    _check(load().os_debug_inject_fault(int(kind), int(step), int(timeout_ns)),
           "os_debug_inject_fault")


def check_device_error(stream=None) -> int:
    """Synchronise ``stream`` and read/clear the device error word; raises
    OssError(OS_ERR_TIMEOUT) when a kernel gave up on a bounded wait."""
    code = _i32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if stream is None else stream.device
    with torch.cuda.device(dev):
        st = load().os_check_device_error(_stream_ptr(stream, dev), ctypes.byref(code))
    if st != OS_OK:
        # a launch that gave up may have left counters in its workspace:
        # later calls get fresh zero-filled ones
        _WORKSPACES.clear()
    _check(st, f"os_check_device_error (code {code.value:#x})")
    return int(code.value)
