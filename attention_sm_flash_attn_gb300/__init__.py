"""Fused scaled-dot-product attention for GB300 (sm_103a): thin Python binding.

Every function here only marshals arguments for libsdpa_gb300.so (C ABI in
include/sdpa_gb300.h); all arithmetic runs in the library's CUDA kernels.
PyTorch provides device memory and streams.  If the library is missing the
calls raise: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

__all__ = [
    "sdpa_prefill", "sdpa_decode", "prefill_workspace_bytes", "prefill_launches",
    "decode_workspace_bytes",
    "device_status", "status_string", "library_path", "load_library", "SdpaError",
    "EXPORTED_SYMBOLS",
]

SDPA_F16, SDPA_BF16 = 0, 1
EXPORTED_SYMBOLS = ("sdpa_prefill", "sdpa_prefill_workspace_bytes", "sdpa_prefill_launches",
                    "sdpa_prefill_ex", "sdpa_decode_ex", "sdpa_decode",
                    "sdpa_decode_workspace_bytes", "sdpa_device_status", "sdpa_status_string",
                    "sdpa_version", "sdpa_decode_noalloc", "sdpa_selftest_timeout")
# Size of the library-resident scratch used by sdpa_decode_noalloc (see the header).
NOALLOC_SCRATCH_BYTES = 24 << 20

_lock = threading.Lock()
_lib = None


class SdpaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None):
    """Load (without building) the shared library and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        path = path or _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run attention_sm_flash_attn_gb300.build")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        attn = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i, vp, sz, vp]
        lib.sdpa_prefill.argtypes = attn
        lib.sdpa_prefill.restype = i
        lib.sdpa_decode.argtypes = attn
        lib.sdpa_decode.restype = i
        # ..., Lk, Dqk, Dv, scale, causal, window, dtype, kv_capacity, kv_ring,
        # bias, bias strides (b, h, q), ws, bytes, stream
        ll = ctypes.c_longlong
        attn_ex = attn[:10] + [i] + attn[10:14] + [i, i, vp, ll, ll, ll] + attn[14:]
        lib.sdpa_prefill_ex.argtypes = attn_ex
        lib.sdpa_prefill_ex.restype = i
        lib.sdpa_decode_ex.argtypes = attn_ex
        lib.sdpa_decode_ex.restype = i
        lib.sdpa_prefill_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.sdpa_prefill_workspace_bytes.restype = sz
        lib.sdpa_prefill_launches.argtypes = [i, i, i, i, i, i, i, i, sz]
        lib.sdpa_prefill_launches.restype = i
        lib.sdpa_decode_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.sdpa_decode_workspace_bytes.restype = sz
        lib.sdpa_device_status.argtypes = [vp, ctypes.POINTER(i)]
        lib.sdpa_device_status.restype = i
        lib.sdpa_status_string.argtypes = [i]
        lib.sdpa_status_string.restype = ctypes.c_char_p
        lib.sdpa_version.argtypes = []
        lib.sdpa_version.restype = i
        lib.sdpa_decode_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i, vp]
        lib.sdpa_decode_noalloc.restype = i
        lib.sdpa_selftest_timeout.argtypes = [vp, vp, vp, vp, i, i, vp, sz, vp,
                                              ctypes.POINTER(i)]
        lib.sdpa_selftest_timeout.restype = i
        if path == _build.LIB_PATH:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().sdpa_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return SDPA_F16
    if t.dtype == torch.bfloat16:
        return SDPA_BF16
    raise TypeError(f"only float16 / bfloat16 are supported, got {t.dtype}")


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check(q, k, v, out, lk=None):
    """Shapes: q [B, Hq, Lq, Dqk], k [B, Hkv, L, Dqk], v [B, Hkv, L, Dv], out [B, Hq,
    Lq, Dv]; L is Lk, or the capacity of a K/V cache when ``lk`` is given."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, L, D]")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D [B, H, L, D]")
    if not (q.dtype == k.dtype == v.dtype == out.dtype):
        raise TypeError("q, k, v, out must share one dtype")
    B, Hq, Lq, D = q.shape
    _, Hkv, L, _ = k.shape
    Dv = v.shape[3]
    if tuple(k.shape) != (B, Hkv, L, D) or tuple(v.shape) != (B, Hkv, L, Dv):
        raise ValueError("k must be [B, Hkv, L, Dqk] and v [B, Hkv, L, Dv] with q's B and Dqk")
    if tuple(out.shape) != (B, Hq, Lq, Dv):
        raise ValueError("out must be [B, Hq, Lq, Dv]")
    Lk = L if lk is None else int(lk)
    return B, Hq, Hkv, Lq, Lk, D, Dv


def prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, causal=False, window=0) -> int:
    return int(load_library().sdpa_prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, int(causal),
                                                           int(window)))


def prefill_launches(B, Hq, Hkv, Lq, Lk, D, causal=False, window=0, workspace_bytes=0) -> int:
    """Kernel launches one sdpa_prefill call makes with that much workspace."""
    n = int(load_library().sdpa_prefill_launches(B, Hq, Hkv, Lq, Lk, D, int(causal), int(window),
                                                  int(workspace_bytes)))
    if n < 0:
        raise SdpaError(n, "sdpa_prefill_launches")
    return n


def decode_workspace_bytes(B, Hq, Hkv, Lq, D) -> int:
    return int(load_library().sdpa_decode_workspace_bytes(B, Hq, Hkv, Lq, D))


def _workspace(nbytes: int, device, workspace):
    if nbytes == 0:
        return workspace
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace


def bias_strides(shape, strides, B, Hq, Lq, Lk):
    """Element strides (batch, head, query row) the library reads a bias of this
    shape and these strides with: a size-1 dim broadcasts (stride 0); the shape
    must broadcast to [B, Hq, Lq, Lk] and the key dim must be dense."""
    if len(shape) != 4 or shape[3] != Lk:
        raise ValueError("bias must be 4-D [B or 1, Hq or 1, Lq or 1, Lk]")
    for n, full in zip(shape[:3], (B, Hq, Lq)):
        if n not in (1, full):
            raise ValueError("bias must broadcast to [B, Hq, Lq, Lk]")
    if Lk > 1 and strides[3] != 1:
        raise ValueError("bias rows must be contiguous along keys")
    return tuple(0 if shape[d] == 1 else int(strides[d]) for d in range(3))


def _bias_args(bias, q, B, Hq, Lq, Lk):
    """(pointer, stride_b, stride_h, stride_q) of a bias broadcastable to [B, Hq,
    Lq, Lk] (see bias_strides)."""
    if bias is None:
        return None, 0, 0, 0
    if not bias.is_cuda or bias.device != q.device:
        raise ValueError("bias must be a CUDA tensor on q's device")
    if bias.dtype != q.dtype:
        raise TypeError("bias must have q's dtype")
    sb, sh, sq = bias_strides(tuple(bias.shape), bias.stride(), B, Hq, Lq, Lk)
    return bias.data_ptr(), sb, sh, sq


def _call(entry, ex_entry, q, k, v, out, B, Hq, Hkv, Lq, Lk, D, Dv, scale, causal, window, lk,
          ring, workspace, stream, bias=None):
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lib = load_library()
    head = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq, Hkv, Lq, Lk, D)
    tail = (float(scale), int(bool(causal)), int(window), _dtype_code(q))
    bias_ptr, sb, sh, sq = _bias_args(bias, q, B, Hq, Lq, Lk)
    if lk is None and not ring and Dv == D and bias is None:
        rc = getattr(lib, entry)(*head, *tail, ws_ptr, ws_len, _stream_ptr(stream))
        name = entry
    else:
        rc = getattr(lib, ex_entry)(*head, Dv, *tail, int(k.shape[2]), int(bool(ring)), bias_ptr,
                                    sb, sh, sq, ws_ptr, ws_len, _stream_ptr(stream))
        name = ex_entry
    if rc != 0:
        raise SdpaError(rc, name)
    return out


def _out(q, v, out):
    if out is None:
        out = torch.empty(q.shape[:3] + (v.shape[3],), dtype=q.dtype, device=q.device)
    return out


def _checked(out, stream, check, name):
    """With check=True: synchronise the stream and raise if a kernel reported a
    device-side failure (its output is then unspecified)."""
    if check:
        status, detail = device_status(stream)
        if status != 0:
            raise SdpaError(status, f"{name} (device code {detail:#x})")
    return out


def sdpa_prefill(q, k, v, out=None, *, scale=None, causal=False, window=0, workspace=None,
                 stream=None, lk=None, ring=False, bias=None, check=False):
    """Fused attention over [B, H, L, D] fp16/bf16 CUDA tensors (see sdpa_prefill and
    sdpa_prefill_ex in include/sdpa_gb300.h).  Returns ``out``.  ``workspace`` may
    be a uint8 CUDA tensor; when None one is allocated with torch if the schedule
    wants it.  v may have its own head dim (Q/K 192 with V 256).  With ``lk``
    given (or ``ring``), k and v are a K/V cache of k.shape[2] rows holding
    Lk = lk keys.  ``bias`` (q's dtype, [B or 1, Hq or 1, Lq or 1, Lk], dense along
    keys) is added to the scaled scores; -inf hides a key.  ``check=True``
    synchronises and raises SdpaError if a kernel reported a device-side failure
    (see sdpa_device_status); otherwise call device_status() yourself."""
    out = _out(q, v, out)
    B, Hq, Hkv, Lq, Lk, D, Dv = _check(q, k, v, out, lk)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, causal, window)
    workspace = _workspace(need, q.device, workspace)
    _call("sdpa_prefill", "sdpa_prefill_ex", q, k, v, out, B, Hq, Hkv, Lq, Lk, D, Dv,
          scale, causal, window, lk, ring, workspace, stream, bias)
    return _checked(out, stream, check, "sdpa_prefill")


def sdpa_decode(q, k, v, out=None, *, scale=None, causal=True, window=0, workspace=None,
                stream=None, lk=None, ring=False, bias=None, check=False):
    """Split-KV decode / verify for 1 <= Lq <= 8 (see sdpa_decode and sdpa_decode_ex
    in include/sdpa_gb300.h).  Returns ``out``.  Head dims, ``lk``, ``ring``,
    ``bias`` and ``check`` as for sdpa_prefill."""
    out = _out(q, v, out)
    B, Hq, Hkv, Lq, Lk, D, Dv = _check(q, k, v, out, lk)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = decode_workspace_bytes(B, Hq, Hkv, Lq, Dv)
    workspace = _workspace(need, q.device, workspace)
    _call("sdpa_decode", "sdpa_decode_ex", q, k, v, out, B, Hq, Hkv, Lq, Lk, D, Dv,
          scale, causal, window, lk, ring, workspace, stream, bias)
    return _checked(out, stream, check, "sdpa_decode")


def device_status(stream=None):
    """(status, detail): synchronises the stream and reads/clears the device status word."""
    detail = ctypes.c_int(0)
    rc = load_library().sdpa_device_status(_stream_ptr(stream), ctypes.byref(detail))
    return int(rc), int(detail.value)
