"""Device-side failure detection, tested without a GPU fault.

sdpa_selftest_timeout runs a small call whose "query tile ready" signal is
withheld: the MMA issuer's bounded wait gives up after about 2 s, every CTA
drains its in-flight copies and MMAs and exits, and the host reads
SDPA_ERR_DEVICE_TIMEOUT with the code of the wait that gave up.  Each kernel
variant is covered (2-SM prefill and head-dim-split pair at head_dim 256/512,
single-CTA and pair decode).  Afterwards a normal call must still match the
oracle: the CUDA context stays usable.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import attention_sm_flash_attn_gb300 as gb
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [256, 512])
@pytest.mark.parametrize("decode", [0, 1])
def test_withheld_signal_times_out_cleanly(D, decode):
    Lq = 1 if decode else 128
    g = torch.Generator().manual_seed(D + decode)
    q = torch.randn(1, 2, Lq, D, generator=g).half().cuda()
    k = torch.randn(1, 1, 128, D, generator=g).half().cuda()
    v = torch.randn(1, 1, 128, D, generator=g).half().cuda()
    out = torch.zeros_like(q)
    nws = gb.decode_workspace_bytes(1, 2, 1, 1, D) if decode else 0
    ws = torch.zeros(max(nws, 16), dtype=torch.uint8, device="cuda")
    detail = ctypes.c_int(0)
    lib = gb.load_library()
    rc = lib.sdpa_selftest_timeout(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), D,
                                   decode, ws.data_ptr(), nws,
                                   torch.cuda.current_stream().cuda_stream, ctypes.byref(detail))
    assert rc == -5, gb.status_string(rc)
    # the code of the first wait that gave up: the query-tile wait (0x100) or a
    # wait that depends on it (the producer's slot-free wait, the softmax's
    # scores-ready wait, ...), all in the device-timeout range
    assert 0x100 <= detail.value <= 0x10a, hex(detail.value)
    assert gb.device_status() == (0, 0)  # the status word was cleared
    # The context is still usable: a normal call of the same kernel variant is correct.
    ref = oracle.sdpa(q.cpu(), k.cpu(), v.cpu(), causal=True)
    got = (gb.sdpa_decode if decode else gb.sdpa_prefill)(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert float(np.max(np.abs(got.cpu().double().numpy() - ref))) < 4e-3


def test_persistent_prefix_wait_timeout_stores_nan_rows():
    """Persistent prefill whose tail pieces never publish their partials: each
    unit that owns such a tile gives up its bounded wait (code 0x10a), merges
    nothing and stores NaN rows, so skipping the status check cannot turn the
    timeout into plausible numbers.  A normal call afterwards is correct."""
    D, Lq, Lk = 256, 256, 4096
    g = torch.Generator().manual_seed(77)
    q = torch.randn(1, 2, Lq, D, generator=g).half().cuda()
    k = torch.randn(1, 1, Lk, D, generator=g).half().cuda()
    v = torch.randn(1, 1, Lk, D, generator=g).half().cuda()
    out = torch.zeros_like(q)
    nws = gb.prefill_workspace_bytes(1, 2, 1, Lq, Lk, D, True, 0)
    assert nws > 0
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    detail = ctypes.c_int(0)
    lib = gb.load_library()
    rc = lib.sdpa_selftest_timeout(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), D,
                                   2, ws.data_ptr(), nws,
                                   torch.cuda.current_stream().cuda_stream, ctypes.byref(detail))
    if rc == -2:
        pytest.skip("this device's persistent schedule has no tail pieces for the shape")
    assert rc == -5, gb.status_string(rc)
    assert detail.value == 0x10a, hex(detail.value)
    # every query tile of this shape is a leftover tile with a tail on other units
    assert bool(torch.isnan(out.float()).all())
    assert gb.device_status() == (0, 0)
    ref = oracle.sdpa(q.cpu(), k.cpu(), v.cpu(), causal=True, rows=range(0, 2 * Lq, 37))
    got = gb.sdpa_prefill(q, k, v, causal=True, workspace=ws, check=True)
    sel = got.reshape(-1, D)[torch.arange(0, 2 * Lq, 37, device="cuda")]
    assert float(np.max(np.abs(sel.cpu().double().numpy() - ref))) < 4e-3
