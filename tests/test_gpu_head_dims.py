"""GPU parity with a V head dim different from Q/K's: Q/K 192 with V 256.

"Fused SDPA full-attention for head_dim=192/256" (MLX PR #3660, thread under
"Additional head dimension discovered") names Q=192/K=192/V=256 heads as the
ones its Q != V check keeps off the fused path.  Here they run the one-CTA
kernel: scores over 192 columns, output over 256.  Compared with the fp64
oracle (which takes Dqk and Dv separately), at the tolerance of the other
parity tests; decode rows must stay bit-identical to single-row calls.
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
DQK, DV = 192, 256


def draw(B, Hq, Hkv, Lq, Lk, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lq, DQK, generator=g).to(dtype)
    k = torch.randn(B, Hkv, Lk, DQK, generator=g).to(dtype)
    v = torch.randn(B, Hkv, Lk, DV, generator=g).to(dtype)
    return q, k, v


def err(out, ref):
    return float(np.max(np.abs(out.detach().cpu().double().numpy() - ref)))


PREFILL = [
    # B, Hq, Hkv, Lq, Lk, causal, window
    (1, 2, 1, 128, 128, True, 0),
    (1, 4, 2, 200, 333, True, 0),
    (2, 2, 1, 130, 257, False, 0),
    (1, 2, 2, 300, 300, True, 7),
    (1, 4, 2, 300, 2000, True, 512),
    (1, 2, 1, 129, 4100, True, 0),      # long keys: persistent schedule
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", PREFILL)
def test_prefill_qk192_v256_matches_oracle(case, dtype):
    B, Hq, Hkv, Lq, Lk, causal, window = case
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, dtype, seed=sum(case))
    scale = 1.0 / math.sqrt(DQK)
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=causal,
                          window=window)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    assert out.shape == (B, Hq, Lq, DV)
    ref = oracle.sdpa(q, k, v, scale=scale, causal=causal, window=window)
    assert err(out, ref) < TOL[dtype]


@pytest.mark.parametrize("Lq", [1, 4, 8])
@pytest.mark.parametrize("window", [0, 1024])
def test_decode_qk192_v256_matches_oracle(Lq, window):
    q, k, v = draw(1, 16, 8, Lq, 5000, torch.float16, seed=Lq + window)
    out = gb.sdpa_decode(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, window=window)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    ref = oracle.sdpa(q, k, v, causal=True, window=window)
    assert err(out, ref) < TOL[torch.float16]


def test_decode_qk192_v256_rows_match_single_row_calls():
    M, Lk, window = 4, 5000, 1024
    q, k, v = (x.to(DEV) for x in draw(1, 16, 8, M, Lk, torch.bfloat16, seed=9))
    block = gb.sdpa_decode(q, k, v, causal=True, window=window)
    for i in range(M):
        n = Lk - M + 1 + i
        row = gb.sdpa_decode(q[:, :, i:i + 1].contiguous(), k[:, :, :n].contiguous(),
                             v[:, :, :n].contiguous(), causal=True, window=window)
        assert torch.equal(block[:, :, i], row[:, :, 0]), i


def test_qk192_v256_from_a_ring_equals_packed():
    Lk, cap, window = 9000, 1152, 1024
    q, k, v = (x.to(DEV) for x in draw(1, 16, 8, 4, Lk, torch.float16, seed=10))
    want = gb.sdpa_decode(q, k, v, causal=True, window=window)
    idx = torch.arange(Lk - cap, Lk, device=DEV)
    kc = torch.zeros(1, 8, cap, DQK, dtype=k.dtype, device=DEV)
    vc = torch.zeros(1, 8, cap, DV, dtype=v.dtype, device=DEV)
    kc[:, :, idx % cap] = k[:, :, idx]
    vc[:, :, idx % cap] = v[:, :, idx]
    got = gb.sdpa_decode(q, kc, vc, causal=True, window=window, lk=Lk, ring=True)
    assert torch.equal(got, want)
