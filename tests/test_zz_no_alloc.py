"""sdpa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers run inside a host runtime that owns the device heap and forbids
allocation on its execution path, or in latency-critical loops where a
cudaMalloc is not acceptable; they cannot pass sdpa_decode a workspace.  The
no-alloc entry point keeps its split partials in a scratch array that is part
of the library itself.  These tests call it through the C ABI and check it
against the regular sdpa_decode entry point (same tolerance as the other GPU
parity tests; the two share the kernels, so they also agree bit for bit), on
two calls in a row, compare the second call with the fp64 oracle, and check
that an oversized call is refused cleanly.

The file is named so that pytest collects it last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import attention_sm_flash_attn_gb300 as gb
import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.float16: 4e-3, torch.bfloat16: 1.6e-2}


def draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return tuple((torch.randn(*shape, generator=g)).to(dtype).cuda()
                 for shape in ((B, Hq, Lq, D), (B, Hkv, Lk, D), (B, Hkv, Lk, D)))


def noalloc(q, k, v, out, causal, window):
    lib = gb.load_library()
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    code = gb.SDPA_BF16 if q.dtype == torch.bfloat16 else gb.SDPA_F16
    return lib.sdpa_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq,
                                   Hkv, Lq, Lk, D, 1.0 / math.sqrt(D), int(causal), window, code,
                                   torch.cuda.current_stream().cuda_stream)


CASES = [
    # B, Hq, Hkv, Lq, Lk, D, window, dtype
    (1, 16, 8, 4, 5000, 256, 1024, torch.float16),
    (1, 16, 1, 8, 3000, 512, 0, torch.bfloat16),
]


@pytest.mark.parametrize("case", CASES)
def test_noalloc_matches_decode_on_two_calls_in_a_row(case):
    B, Hq, Hkv, Lq, Lk, D, window, dtype = case
    for call in range(2):
        q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed=100 * call + Lk)
        want = gb.sdpa_decode(q, k, v, causal=True, window=window)
        got = torch.full_like(q, float("nan"))
        rc = noalloc(q, k, v, got, True, window)
        assert rc == 0, gb.status_string(rc)
        torch.cuda.synchronize()
        assert gb.device_status()[0] == 0
        err = float((got.float() - want.float()).abs().max())
        assert err < TOL[dtype], (call, err)
        assert torch.equal(got, want), call
    # the last call against the fp64 oracle as well
    ref = oracle.sdpa(q.cpu(), k.cpu(), v.cpu(), causal=True, window=window)
    err = float(np.max(np.abs(got.cpu().double().numpy() - ref)))
    assert err < TOL[dtype], err


def test_noalloc_rejects_calls_beyond_its_scratch():
    # 2048 query heads x 8 rows x (512 + 2) fp32 partials (one split) is about
    # 34 MB, beyond the built-in scratch; the call must be refused before anything
    # is queued.
    B, Hq, Hkv, Lq, Lk, D = 1, 2048, 256, 8, 256, 512
    assert gb.decode_workspace_bytes(B, Hq, Hkv, Lq, D) > gb.NOALLOC_SCRATCH_BYTES
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, torch.float16, seed=3)
    out = torch.zeros_like(q)
    rc = noalloc(q, k, v, out, True, 0)
    assert rc == -7
    assert "scratch" in gb.status_string(rc)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
