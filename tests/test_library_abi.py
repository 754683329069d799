"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side argument validation rejects bad calls before any CUDA call.

No test here launches a kernel: they run on a machine without a GPU.
"""
import ctypes
import os
import re

import pytest

import attention_sm_flash_attn_gb300 as gb
from attention_sm_flash_attn_gb300 import build as gbbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "sdpa_gb300.h")


@pytest.fixture(scope="module")
def lib():
    gbbuild.build()
    return gb.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(sdpa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    assert set(gb.EXPORTED_SYMBOLS) == set(names), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert lib.sdpa_version() == 100
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.sdpa_status_string(code).decode() != "unknown status"
    assert lib.sdpa_status_string(-99).decode() == "unknown status"


FAKE = ctypes.c_void_p(0x10000)   # a 16-byte aligned value; validation fails before any use
ODD = ctypes.c_void_p(0x10008)


def call(lib, fn, q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, Hq=2, Hkv=1, Lq=4, Lk=8, D=256,
         scale=0.0625, causal=1, window=0, dtype=0, ws=FAKE, ws_bytes=1 << 20):
    return getattr(lib, fn)(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, dtype,
                            ws, ws_bytes, None)


BAD = [
    (dict(q=None), -1), (dict(B=0), -1), (dict(Hq=3, Hkv=2), -1), (dict(Lk=0), -1),
    (dict(causal=2), -1), (dict(window=-1), -1), (dict(causal=0, window=4), -1),
    (dict(Lq=9, Lk=8), -1), (dict(scale=-1.0), -1), (dict(scale=float("nan")), -1),
    (dict(D=64), -2), (dict(D=96), -2), (dict(D=320), -2), (dict(dtype=2), -2),
    (dict(k=ODD), -6),
]


@pytest.mark.parametrize("fn", ["sdpa_prefill", "sdpa_decode"])
@pytest.mark.parametrize("kw,code", BAD)
def test_invalid_arguments_are_rejected_on_the_host(lib, fn, kw, code):
    assert call(lib, fn, **kw) == code


def test_decode_rejects_more_than_eight_rows(lib):
    assert call(lib, "sdpa_decode", Lq=9, Lk=64) == -1


def test_decode_rejects_a_misaligned_workspace_on_the_host(lib):
    # Whether a decode call needs a workspace at all depends on the device's
    # split plan (the GPU tests cover both); a misaligned one is refused first.
    assert call(lib, "sdpa_decode", ws=ODD, ws_bytes=1 << 20) == -6


def test_workspace_queries_reject_bad_shapes(lib):
    assert lib.sdpa_decode_workspace_bytes(1, 3, 2, 1, 256) == 0
    assert lib.sdpa_decode_workspace_bytes(1, 2, 1, 9, 256) == 0
    assert lib.sdpa_prefill_workspace_bytes(1, 2, 1, 4, 8, 96, 1, 0) == 0


def test_launch_query_rejects_bad_arguments_on_the_host(lib):
    assert lib.sdpa_prefill_launches(1, 2, 1, 4, 8, 96, 1, 0, 0) == -2    # head dim
    assert lib.sdpa_prefill_launches(1, 3, 2, 4, 8, 256, 1, 0, 0) == -1   # Hq % Hkv
    assert lib.sdpa_prefill_launches(1, 2, 1, 4, 8, 256, 0, 16, 0) == -1  # window w/o causal
    assert lib.sdpa_prefill_launches(1, 2, 1, 9, 8, 256, 1, 0, 0) == -1   # causal Lq > Lk


def call_ex(lib, fn, cap, ring, Lq=4, Lk=3000, window=1024, causal=1, Dqk=256, Dv=256,
            bias=None, sb=0, sh=0, sq=0):
    return getattr(lib, fn)(FAKE, FAKE, FAKE, FAKE, 1, 2, 1, Lq, Lk, Dqk, Dv, 0.0625, causal,
                            window, 0, cap, ring, bias, sb, sh, sq, FAKE, 1 << 20, None)


@pytest.mark.parametrize("fn", ["sdpa_prefill_ex", "sdpa_decode_ex"])
def test_cache_layouts_are_checked_on_the_host(lib, fn):
    assert call_ex(lib, fn, 2000, 0) == -1          # packed cache shorter than Lk
    assert call_ex(lib, fn, 1000, 1) == -1          # ring not a multiple of 128
    assert call_ex(lib, fn, 896, 1) == -1           # ring misses keys the window sees
    assert call_ex(lib, fn, 4096, 2) == -1          # ring flag not 0/1
    assert call_ex(lib, fn, 0, 0) == -1
    assert call_ex(lib, fn, 2048, 1, window=0) == -1  # no window: the ring must hold all Lk


@pytest.mark.parametrize("fn", ["sdpa_prefill_ex", "sdpa_decode_ex"])
def test_unequal_head_dims_are_checked_on_the_host(lib, fn):
    for dqk, dv in ((256, 128), (128, 256), (192, 128), (512, 256), (256, 192)):
        assert call_ex(lib, fn, 3000, 0, Dqk=dqk, Dv=dv) == -2, (dqk, dv)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        gb.load_library(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("fn", ["sdpa_prefill_ex", "sdpa_decode_ex"])
def test_bias_arguments_are_checked_on_the_host(lib, fn):
    ok = dict(cap=3000, ring=0)
    assert call_ex(lib, fn, bias=FAKE, sb=-8, **ok) == -1
    assert call_ex(lib, fn, bias=FAKE, sh=-1, **ok) == -1
    assert call_ex(lib, fn, bias=FAKE, sq=1 << 60, **ok) == -1
    assert call_ex(lib, fn, bias=ctypes.c_void_p(0x10001), sq=3000, **ok) == -6   # odd address


def test_bias_strides_broadcast_and_views():
    import torch
    B, Hq, Lq, Lk = 2, 4, 9, 40
    full = torch.zeros(B, Hq, Lq, Lk)
    assert gb.bias_strides(full.shape, full.stride(), B, Hq, Lq, Lk) == (Hq * Lq * Lk, Lq * Lk, Lk)
    shared = torch.zeros(1, 1, Lq, Lk)
    assert gb.bias_strides(shared.shape, shared.stride(), B, Hq, Lq, Lk) == (0, 0, Lk)
    per_head_row = torch.zeros(B, Hq, 1, Lk)
    assert gb.bias_strides(per_head_row.shape, per_head_row.stride(), B, Hq, Lq, Lk) == \
        (Hq * Lk, Lk, 0)
    # a [.., :Lk] view of wider rows keeps the wider row stride
    wide = torch.zeros(1, Hq, Lq, Lk + 3)[..., :Lk]
    assert gb.bias_strides(wide.shape, wide.stride(), B, Hq, Lq, Lk) == (0, Lq * (Lk + 3), Lk + 3)
    # an expanded tensor: stride 0 where it was expanded
    exp = torch.zeros(1, 1, 1, Lk).expand(B, Hq, Lq, Lk)
    assert gb.bias_strides(exp.shape, exp.stride(), B, Hq, Lq, Lk) == (0, 0, 0)


@pytest.mark.parametrize("shape,strides", [((1, 1, 1, 39), (39, 39, 39, 1)),
                                           ((3, 1, 1, 40), (40, 40, 40, 1)),
                                           ((1, 1, 9, 40), (360, 360, 1, 9)),
                                           ((1, 40), (40, 1))])
def test_bias_strides_reject_bad_layouts(shape, strides):
    with pytest.raises(ValueError):
        gb.bias_strides(shape, strides, 2, 4, 9, 40)
