"""Bounds evidence without a sanitizer: guard canaries around every buffer the
library writes.

`out`, the caller's workspace and (for decode) the split partials inside it are
carved out of larger device buffers whose margins before and after hold a fixed
byte pattern.  Ragged calls (query and key counts that are not multiples of the
128/256-row or 64/128-key tiles, Lq 1..8 decode, every head dim, bias, ring
caches) run through every kernel variant; afterwards the margins must be byte
for byte what they were, and every element of `out` must have been written
(none still holds the pattern, which is no value attention can produce here).
The epilogues store partial tiles, so an off-by-one in a row or column guard
would land in a margin.
"""
import math

import numpy as np
import pytest
import torch

import attention_sm_flash_attn_gb300 as gb
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"
MARGIN = 8192          # elements (16-bit) or bytes around each carved buffer
SENT16 = 0x7BCD        # fp16 ~6.3e4, bf16 ~2.1e36: never an output of these calls
SENT8 = 0xA5
TOL = {torch.float16: 4e-3, torch.bfloat16: 1.6e-2}


class Carved16:
    """A [shape] fp16/bf16 tensor in the middle of a sentinel-filled buffer."""

    def __init__(self, shape, dtype):
        self.n = int(np.prod(shape))
        self.big = torch.full((2 * MARGIN + self.n,), SENT16, dtype=torch.int16, device=DEV)
        self.t = self.big[MARGIN:MARGIN + self.n].view(dtype).view(shape)

    def check(self, what):
        lo, hi = self.big[:MARGIN], self.big[MARGIN + self.n:]
        assert bool((lo == SENT16).all()), f"{what}: write before the buffer"
        assert bool((hi == SENT16).all()), f"{what}: write past the end of the buffer"
        inner = self.big[MARGIN:MARGIN + self.n]
        assert not bool((inner == SENT16).any()), f"{what}: elements left unwritten"


class CarvedBytes:
    """`nbytes` of workspace (256-byte aligned) inside a sentinel-filled buffer."""

    def __init__(self, nbytes):
        self.n = int(nbytes)
        self.big = torch.full((2 * MARGIN + self.n,), SENT8, dtype=torch.uint8, device=DEV)
        self.t = self.big[MARGIN:MARGIN + self.n] if self.n else None

    def check(self, what):
        lo, hi = self.big[:MARGIN], self.big[MARGIN + self.n:]
        assert bool((lo == SENT8).all()), f"{what}: workspace write before its start"
        assert bool((hi == SENT8).all()), f"{what}: workspace write past its end"


def draw(B, Hq, Hkv, Lq, Lk, Dqk, Dv, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lq, Dqk, generator=g).to(dtype)
    k = torch.randn(B, Hkv, Lk, Dqk, generator=g).to(dtype)
    v = torch.randn(B, Hkv, Lk, Dv, generator=g).to(dtype)
    return q, k, v


def oracle_check(out, q, k, v, causal, window, dtype, bias=None):
    ref = oracle.sdpa(q, k, v, causal=causal, window=window, bias=bias)
    err = float(np.max(np.abs(out.cpu().double().numpy() - ref)))
    assert err < TOL[dtype], f"max abs err {err}"


PREFILL = [
    # B, Hq, Hkv, Lq, Lk, Dqk, Dv, causal, window, workspace, bias  (variant it runs)
    (1, 4, 2, 300, 1000, 256, 256, True, 0, True, False),      # 2-SM, Q in TMEM, persistent
    (2, 2, 1, 257, 383, 256, 256, True, 0, False, False),      # 2-SM, Q in TMEM, one pair a tile
    (1, 4, 2, 301, 1300, 256, 256, True, 300, True, False),    # 2-SM (window >= 256)
    (1, 2, 2, 131, 700, 256, 256, True, 100, True, False),     # one CTA (short window)
    (1, 4, 2, 200, 333, 128, 128, True, 0, True, False),       # 2-SM at head_dim 128
    (1, 4, 2, 200, 333, 192, 192, True, 0, True, False),       # one CTA at head_dim 192
    (1, 4, 2, 139, 500, 192, 256, True, 0, True, False),       # Q/K 192 with V 256
    (1, 2, 1, 200, 5000, 512, 512, True, 0, True, False),      # pair, split keys + merge kernel
    (1, 2, 2, 77, 129, 512, 512, False, 0, False, False),      # pair, one launch
    (1, 4, 2, 190, 700, 256, 256, True, 0, True, True),        # 2-SM with a bias
    (1, 3, 1, 1, 129, 256, 256, False, 0, False, False),       # one query row
]


@pytest.mark.parametrize("case", PREFILL)
def test_prefill_writes_stay_inside_out_and_workspace(case):
    B, Hq, Hkv, Lq, Lk, Dqk, Dv, causal, window, use_ws, use_bias = case
    dtype = torch.bfloat16 if use_bias else torch.float16
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, Dqk, Dv, dtype, seed=Lq * 7 + Lk)
    bias = None
    if use_bias:
        g = torch.Generator().manual_seed(3)
        bias = torch.randn(1, 1, Lq, Lk, generator=g)
        bias = bias.masked_fill(torch.rand(1, 1, Lq, Lk, generator=g) < 0.25,
                                float("-inf")).to(dtype)
    out = Carved16((B, Hq, Lq, Dv), dtype)
    need = gb.prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, Dqk, causal, window) if use_ws else 0
    ws = CarvedBytes(need)
    gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), out.t, causal=causal, window=window,
                    workspace=ws.t, bias=None if bias is None else bias.to(DEV))
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    out.check("out")
    ws.check("workspace")
    oracle_check(out.t, q, k, v, causal, window, dtype, bias)


DECODE = [
    # B, Hq, Hkv, Lk, D, window
    (1, 16, 8, 3001, 256, 1024),
    (1, 16, 1, 2999, 512, 0),
    (2, 6, 2, 777, 192, 0),
    (1, 20, 1, 1000, 128, 0),     # 20 query heads per kv head: a partly filled second head block
    (1, 4, 4, 65, 512, 64),
]


@pytest.mark.parametrize("Lq", [1, 3, 8])
@pytest.mark.parametrize("case", DECODE)
def test_decode_writes_stay_inside_out_and_workspace(case, Lq):
    B, Hq, Hkv, Lk, D, window = case
    dtype = torch.float16
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, D, dtype, seed=Lq + Lk)
    out = Carved16((B, Hq, Lq, D), dtype)
    ws = CarvedBytes(gb.decode_workspace_bytes(B, Hq, Hkv, Lq, D))
    gb.sdpa_decode(q.to(DEV), k.to(DEV), v.to(DEV), out.t, causal=True, window=window,
                   workspace=ws.t)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    out.check("out")
    ws.check("workspace")
    oracle_check(out.t, q, k, v, True, window, dtype)


def test_decode_from_a_ring_writes_stay_inside():
    B, Hq, Hkv, Lq, Lk, D, window, cap = 1, 16, 8, 5, 5000, 256, 1024, 1152
    dtype = torch.bfloat16
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, D, dtype, seed=9)
    idx = torch.arange(Lk - cap, Lk)
    kc = torch.zeros(B, Hkv, cap, D, dtype=dtype)
    vc = torch.zeros(B, Hkv, cap, D, dtype=dtype)
    kc[:, :, idx % cap] = k[:, :, idx]
    vc[:, :, idx % cap] = v[:, :, idx]
    out = Carved16((B, Hq, Lq, D), dtype)
    ws = CarvedBytes(gb.decode_workspace_bytes(B, Hq, Hkv, Lq, D))
    gb.sdpa_decode(q.to(DEV), kc.to(DEV), vc.to(DEV), out.t, causal=True, window=window,
                   workspace=ws.t, lk=Lk, ring=True)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    out.check("out")
    ws.check("workspace")
    oracle_check(out.t, q, k, v, True, window, dtype)


def test_sentinels_are_not_attention_outputs():
    """The pattern is far outside what any of these calls can output (|out| is
    bounded by max |v|, at most ~6 for N(0, 1) draws of this size)."""
    s = torch.tensor([SENT16], dtype=torch.int16)
    assert abs(float(s.view(torch.float16))) > 6e4
    assert abs(float(s.view(torch.bfloat16))) > 1e30
    assert math.isfinite(float(s.view(torch.float16)))
