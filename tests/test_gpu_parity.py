"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerance (max abs error on unit-variance inputs): 4e-3 for fp16, 1.6e-2 for
bf16.  Cases span several 128-row query tiles and 128-key tiles with ragged
tails, grouped-query heads, bottom-right causal masks, sliding windows, the
split and persistent prefill paths, every head dim (128, 192, 256, 512) and
both dtypes.  Exact pins: one key (Lk = 1) and window 1 make every softmax
weight exactly 1, so the GPU output must equal the value row bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import attention_sm_flash_attn_gb300 as gb
import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.float16: 4e-3, torch.bfloat16: 1.6e-2}
DEV = "cuda"


def draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed, amp=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, Hq, Lq, D, generator=g) * amp).to(dtype)
    k = (torch.randn(B, Hkv, Lk, D, generator=g) * amp).to(dtype)
    v = (torch.randn(B, Hkv, Lk, D, generator=g) * amp).to(dtype)
    return q, k, v


def max_err(got, ref):
    return float(np.max(np.abs(got.detach().cpu().double().numpy() - ref)))


PREFILL_CASES = [
    # B, Hq, Hkv, Lq, Lk, D, causal, window
    (1, 2, 1, 128, 128, 256, True, 0),      # the tiny causal self-attention workload
    (1, 2, 1, 128, 128, 256, True, 32),     # ... and its window-32 variant
    (1, 4, 2, 200, 333, 256, True, 0),      # ragged q and k tails, bottom-right
    (2, 2, 1, 130, 257, 256, False, 0),     # non-causal, batch 2
    (1, 2, 2, 300, 300, 256, True, 7),      # narrow window crossing tile edges
    (1, 4, 1, 64, 700, 256, True, 100),     # window, Lq << Lk
    (1, 3, 1, 1, 129, 256, True, 0),        # a single query row
    (1, 2, 1, 128, 128, 512, True, 0),
    (1, 4, 2, 150, 300, 512, True, 50),
    (1, 2, 2, 70, 129, 512, False, 0),
    (1, 2, 1, 129, 4100, 256, True, 0),     # long keys: split-KV prefill + combine
    (1, 2, 1, 300, 100, 256, False, 0),     # non-causal, more queries than keys, keys < 1 tile
    (1, 2, 2, 513, 65, 256, False, 0),      # query rows spill into a third 256-row tile
    (3, 4, 4, 257, 1000, 256, True, 0),     # batch 3, one row past a 256-row tile
    (1, 2, 1, 256, 3000, 512, True, 0),     # long keys at head_dim 512
    (1, 4, 2, 600, 1500, 256, True, 300),   # 2-SM window >= 256, head-paired tiles, ragged
    (1, 3, 1, 400, 900, 256, True, 256),    # 2-SM window, odd group size (256-row tiles)
    # head_dim 192 (one-CTA variant) and 128 (2-SM variant, one CTA for short windows)
    (1, 2, 1, 128, 128, 192, True, 0),
    (1, 4, 2, 200, 333, 192, True, 0),
    (1, 2, 2, 300, 300, 192, True, 7),
    (2, 2, 1, 130, 257, 192, False, 0),
    (1, 2, 1, 129, 4100, 192, True, 0),
    (1, 2, 1, 128, 128, 128, True, 0),
    (1, 4, 2, 200, 333, 128, True, 0),
    (2, 2, 1, 130, 257, 128, False, 0),
    (1, 4, 1, 64, 700, 128, True, 100),
    (1, 2, 2, 600, 1500, 128, True, 300),
    (1, 2, 1, 129, 4100, 128, True, 0),
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", PREFILL_CASES)
def test_prefill_matches_oracle(case, dtype):
    B, Hq, Hkv, Lq, Lk, D, causal, window = case
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed=abs(hash(case)) % 10000)
    scale = 1.0 / math.sqrt(D)
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=causal,
                          window=window)
    torch.cuda.synchronize()
    ref = oracle.sdpa(q, k, v, scale=scale, causal=causal, window=window)
    assert gb.device_status()[0] == 0
    err = max_err(out, ref)
    assert err < TOL[dtype], f"max abs err {err}"


@pytest.mark.parametrize("case", [(1, 2, 1, 128, 4100, 256, True, 0), (1, 2, 1, 64, 3000, 512, False, 0)])
def test_prefill_without_workspace_matches_split_path(case):
    """The same call with and without a workspace both match the oracle: with
    one, head_dim 256 runs the persistent schedule and head_dim 512 splits key
    ranges merged by the combine kernel; without one, each query tile is one
    CTA (pair) over its whole key range."""
    B, Hq, Hkv, Lq, Lk, D, causal, window = case
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, torch.float16, seed=5)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    need = gb.prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, causal, window)
    assert need > 0
    a = gb.sdpa_prefill(qd, kd, vd, causal=causal, window=window)
    out = torch.empty_like(qd)
    lib = gb.load_library()
    rc = lib.sdpa_prefill(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), B, Hq, Hkv,
                          Lq, Lk, D, 1.0 / math.sqrt(D), int(causal), window, 0, None, 0,
                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    ref = oracle.sdpa(q, k, v, causal=causal, window=window)
    assert max_err(a, ref) < 4e-3
    assert max_err(out, ref) < 4e-3


@pytest.mark.parametrize("D", [128, 192, 256, 512])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_single_key_is_exact(D, dtype):
    q, k, v = draw(1, 4, 2, 5, 1, D, dtype, seed=11)
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), causal=False)
    want = v.repeat_interleave(2, dim=1).expand(-1, -1, 5, -1)
    assert torch.equal(out.cpu(), want)


@pytest.mark.parametrize("D", [128, 192, 256, 512])
def test_window_one_is_exact(D):
    Lq, Lk = 150, 300
    q, k, v = draw(1, 2, 1, Lq, Lk, D, torch.bfloat16, seed=12)
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, window=1).cpu()
    for h in range(2):
        assert torch.equal(out[0, h], v[0, 0, Lk - Lq:])


def test_zero_scale_gives_mean_of_visible_values():
    Lq, Lk = 40, 300
    q, k, v = draw(1, 2, 1, Lq, Lk, 256, torch.float16, seed=13)
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, window=37, scale=0.0)
    ref = oracle.sdpa(q, k, v, causal=True, window=37, scale=0.0)
    assert max_err(out, ref) < 4e-3


# ---------------------------------------------------------------- decode

DECODE_CASES = [
    # B, Hq, Hkv, Lk, D, window
    (1, 16, 8, 5000, 256, 1024),
    (1, 16, 1, 3000, 512, 0),
    (2, 4, 2, 777, 256, 0),
    (1, 32, 1, 1000, 256, 0),    # 32 query heads per kv head: two head blocks
    (1, 4, 4, 129, 512, 64),
    (1, 16, 8, 5000, 192, 1024),
    (2, 8, 2, 777, 128, 0),
]


@pytest.mark.parametrize("Lq", [1, 2, 4, 8])
@pytest.mark.parametrize("case", DECODE_CASES)
def test_decode_matches_oracle(case, Lq):
    B, Hq, Hkv, Lk, D, window = case
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, torch.float16, seed=Lq * 100 + Lk)
    out = gb.sdpa_decode(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, window=window)
    torch.cuda.synchronize()
    ref = oracle.sdpa(q, k, v, causal=True, window=window)
    assert gb.device_status()[0] == 0
    assert max_err(out, ref) < 4e-3


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", DECODE_CASES)
def test_decode_rows_are_bit_identical_to_single_row_calls(case, dtype):
    """Row i of an Lq = M call equals, bit for bit, the Lq = 1 call over the
    key prefix physically trimmed to Lk - M + 1 + i keys."""
    B, Hq, Hkv, Lk, D, window = case
    for M in (2, 4, 8):
        q, k, v = draw(B, Hq, Hkv, M, Lk, D, dtype, seed=M + 7)
        qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
        block = gb.sdpa_decode(qd, kd, vd, causal=True, window=window)
        for i in range(M):
            n = Lk - M + 1 + i
            row = gb.sdpa_decode(qd[:, :, i:i + 1].contiguous(), kd[:, :, :n].contiguous(),
                                 vd[:, :, :n].contiguous(), causal=True, window=window)
            assert torch.equal(block[:, :, i], row[:, :, 0]), (M, i)


def test_decode_agrees_with_prefill_within_tolerance():
    q, k, v = draw(1, 16, 8, 4, 2000, 256, torch.float16, seed=21)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    a = gb.sdpa_decode(qd, kd, vd, causal=True, window=1024)
    b = gb.sdpa_prefill(qd, kd, vd, causal=True, window=1024)
    assert float((a.float() - b.float()).abs().max()) < 4e-3


@pytest.mark.parametrize("D", [128, 256, 512])
def test_large_scale_exercises_the_rescale(D):
    """scale = 1 on unit-variance inputs: row maxima jump by far more than the
    lazy-rescale threshold from tile to tile, so O is rescaled in tensor
    memory many times; the result still matches the oracle."""
    Lq, Lk = 300, 2000
    q, k, v = draw(1, 4, 2, Lq, Lk, D, torch.float16, seed=14 + D)
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=1.0)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    ref = oracle.sdpa(q, k, v, causal=True, scale=1.0)
    assert max_err(out, ref) < 4e-3


def test_decode_workspace_rules():
    """Head dims up to 256 with one cluster of splits per head group need no
    workspace (NULL is accepted and the result matches the oracle); head dim
    512 merges split partials in a second kernel and refuses a NULL workspace."""
    lib = gb.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for D, need_ws in ((256, False), (512, True)):
        Hq, Hkv, Lq, Lk = 16, 8 if D == 256 else 1, 4, 5000
        q, k, v = draw(1, Hq, Hkv, Lq, Lk, D, torch.float16, seed=D)
        assert (gb.decode_workspace_bytes(1, Hq, Hkv, Lq, D) > 0) == need_ws
        qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
        out = torch.zeros_like(qd)
        rc = lib.sdpa_decode(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), 1, Hq,
                             Hkv, Lq, Lk, D, 1.0 / math.sqrt(D), 1, 1024, 0, None, 0, stream)
        if need_ws:
            assert rc == -3
            continue
        assert rc == 0
        torch.cuda.synchronize()
        assert gb.device_status()[0] == 0
        ref = oracle.sdpa(q, k, v, causal=True, window=1024)
        assert max_err(out, ref) < 4e-3
