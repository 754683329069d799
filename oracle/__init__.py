"""fp64 CPU oracle for scaled-dot-product attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The library (``attention_sm_flash_attn_gb300``) never
does, and this package imports nothing from it: the two share no code.

The arithmetic lives in ``sdpa_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it with gcc on first use and marshals arguments.

Definition (restated from the pages, cited in ``sdpa_oracle.c``): for query
row i of head h, with G = Hq/Hkv, KV head g = h // G and bottom-right position
p_i = Lk - Lq + i, the visible keys are
``{j : (not causal or j <= p_i) and (W == 0 or p_i - j < W)}``; scores are
``scale * q.k`` over the exact fp16/bf16 input values; the softmax runs over
the visible keys only; the output is the softmax-weighted sum of V rows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_sdpa.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle_sdpa.so`` next to its source."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.c_void_p
        c_int, c_double = ctypes.c_int, ctypes.c_double
        lib.oracle_sdpa.argtypes = [u16p, u16p, u16p, c_int, c_int, c_int, c_int, c_int,
                                    c_int, c_int, c_int, c_double, c_int, c_int,
                                    ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, c_int]
        lib.oracle_sdpa.restype = c_int
        i64 = ctypes.c_int64
        lib.oracle_sdpa_bias.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, c_int, c_int,
                                         c_int, c_int, c_int, c_int, c_int, c_int, c_double,
                                         c_int, c_int, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_void_p, c_int]
        lib.oracle_sdpa_bias.restype = c_int
        lib.oracle_row_scores.argtypes = [u16p, u16p, c_int, c_int, c_int, c_int, c_int,
                                          c_int, c_int, c_double, c_int, c_int, c_int,
                                          ctypes.c_void_p]
        lib.oracle_row_scores.restype = c_int
        lib.oracle_row_probs.argtypes = [u16p, u16p, c_int, c_int, c_int, c_int, c_int,
                                         c_int, c_int, c_double, c_int, c_int, c_int,
                                         c_int, c_int, ctypes.c_void_p]
        lib.oracle_row_probs.restype = c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = c_int
        _lib = lib
        return lib


def _as_u16(t: torch.Tensor):
    """A contiguous CPU fp16/bf16 tensor viewed as raw 16-bit words (no copy of values)."""
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError(f"oracle inputs must be fp16 or bf16, got {t.dtype}")
    t = t.detach().to("cpu").contiguous()
    return t, t.view(torch.int16).numpy()


def _dtype_code(t: torch.Tensor) -> int:
    return BF16 if t.dtype == torch.bfloat16 else F16


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def sdpa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: float | None = None,
         causal: bool = False, window: int = 0, rows=None, nthreads: int = 0,
         bias: torch.Tensor | None = None) -> np.ndarray:
    """Exact-input fp64 attention.

    q: [B, Hq, Lq, Dqk], k: [B, Hkv, Lk, Dqk], v: [B, Hkv, Lk, Dv], all fp16 or all
    bf16 (CPU or GPU tensors; they are copied to host).  ``rows`` is None (every
    row; result shaped [B, Hq, Lq, Dv]) or an iterable of flat row ids
    ``(b * Hq + h) * Lq + i`` (result shaped [len(rows), Dv]).  ``bias`` (same
    dtype, shape [B or 1, Hq or 1, Lq or 1, Lk]) is added to the scaled scores;
    -inf removes a key, and a row left without keys outputs zeros.
    """
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    B, Hq, Lq, Dqk = q.shape
    Bk, Hkv, Lk, Dk = k.shape
    if Bk != B or Dk != Dqk or tuple(v.shape[:3]) != (B, Hkv, Lk):
        raise ValueError("shape mismatch between q, k, v")
    Dv = v.shape[3]
    if scale is None:
        scale = 1.0 / float(Dqk) ** 0.5
    qt, qn = _as_u16(q)
    kt, kn = _as_u16(k)
    vt, vn = _as_u16(v)
    if rows is None:
        ids = None
        n = B * Hq * Lq
    else:
        ids = np.ascontiguousarray(np.asarray(list(rows), dtype=np.int64))
        n = ids.shape[0]
    out = np.zeros((n, Dv), dtype=np.float64)
    if bias is None:
        rc = _load().oracle_sdpa(
            qn.ctypes.data, kn.ctypes.data, vn.ctypes.data, _dtype_code(q), B, Hq, Hkv, Lq, Lk,
            Dqk, Dv, float(scale), int(bool(causal)), int(window),
            None if ids is None else ids.ctypes.data, n, out.ctypes.data, int(nthreads))
    else:
        if bias.dtype != q.dtype or bias.dim() != 4 or bias.shape[3] != Lk:
            raise ValueError("bias must be [B or 1, Hq or 1, Lq or 1, Lk] in q's dtype")
        b0, h0, q0 = bias.shape[:3]
        if b0 not in (1, B) or h0 not in (1, Hq) or q0 not in (1, Lq):
            raise ValueError("bias must broadcast to [B, Hq, Lq, Lk]")
        bt, bn = _as_u16(bias)
        sb = 0 if b0 == 1 else h0 * q0 * Lk
        sh = 0 if h0 == 1 else q0 * Lk
        sq = 0 if q0 == 1 else Lk
        rc = _load().oracle_sdpa_bias(
            qn.ctypes.data, kn.ctypes.data, vn.ctypes.data, bn.ctypes.data, sb, sh, sq,
            _dtype_code(q), B, Hq, Hkv, Lq, Lk, Dqk, Dv, float(scale), int(bool(causal)),
            int(window), None if ids is None else ids.ctypes.data, n, out.ctypes.data,
            int(nthreads))
        del bt
    if rc != 0:
        raise ValueError(f"oracle_sdpa rejected the call (status {rc})")
    del qt, kt, vt
    if rows is None:
        return out.reshape(B, Hq, Lq, Dv)
    return out


def row_scores(q: torch.Tensor, k: torch.Tensor, b: int, h: int, i: int, *,
               scale: float | None = None) -> np.ndarray:
    """Step 1 alone: the scaled scores of row (b, h, i) against every key, unmasked."""
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    qt, qn = _as_u16(q)
    kt, kn = _as_u16(k)
    out = np.zeros(Lk, dtype=np.float64)
    rc = _load().oracle_row_scores(qn.ctypes.data, kn.ctypes.data, _dtype_code(q), B, Hq,
                                   Hkv, Lq, Lk, D, float(scale), b, h, i, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_row_scores rejected the call (status {rc})")
    return out


def row_probs(q: torch.Tensor, k: torch.Tensor, b: int, h: int, i: int, *,
              scale: float | None = None, causal: bool = False, window: int = 0) -> np.ndarray:
    """Steps 1-2: the softmax weights of row (b, h, i) over every key (0 where masked)."""
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    qt, qn = _as_u16(q)
    kt, kn = _as_u16(k)
    out = np.zeros(Lk, dtype=np.float64)
    rc = _load().oracle_row_probs(qn.ctypes.data, kn.ctypes.data, _dtype_code(q), B, Hq,
                                  Hkv, Lq, Lk, D, float(scale), int(bool(causal)),
                                  int(window), b, h, i, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_row_probs rejected the call (status {rc})")
    return out
