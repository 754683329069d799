"""K/V read from a caller's cache: strided rows and ring buffers.

The pages' decode reads keys from caches: strided, sliced rows for classic
decode and per-row verify, and a ring addressed by a cursor for sliding-window
layers, wrapped or not ("fix: Gemma 4 MTP never engages on CUDA (GB10)",
sections "Current Behavior", "Proposed Solution", "Implementation Notes").

Every case is checked two ways:
  * against the fp64 oracle, element by element (4e-3 fp16, 1.6e-2 bf16), on
    the LOGICAL keys: key j is built on the host by plain indexing, row j of a
    strided cache or row j mod capacity of a ring, independently of the
    library's addressing;
  * bit for bit against the same call on packed K/V (the layout changes only
    which row holds a key, never the arithmetic).
Cache rows no query row can see hold random (finite) values that must not leak
in.
"""
import numpy as np
import pytest
import torch

import attention_sm_flash_attn_gb300 as gb
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = {torch.float16: 4e-3, torch.bfloat16: 1.6e-2}


def draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lq, D, generator=g).to(dtype).to(DEV)
    k = torch.randn(B, Hkv, Lk, D, generator=g).to(dtype).to(DEV)
    v = torch.randn(B, Hkv, Lk, D, generator=g).to(dtype).to(DEV)
    return q, k, v


def strided_cache(x, cap, seed):
    """[B, H, cap, D] cache: the Lk keys in rows 0..Lk-1, random rows after."""
    g = torch.Generator().manual_seed(seed)
    c = torch.randn(x.shape[0], x.shape[1], cap, x.shape[3], generator=g).to(x.dtype).to(DEV)
    c[:, :, :x.shape[2]] = x
    return c


def ring_cache(x, cap, seed):
    """[B, H, cap, D] ring: key p in row p mod cap for the last cap keys."""
    g = torch.Generator().manual_seed(seed)
    c = torch.randn(x.shape[0], x.shape[1], cap, x.shape[3], generator=g).to(x.dtype).to(DEV)
    Lk = x.shape[2]
    idx = torch.arange(max(0, Lk - cap), Lk, device=DEV)
    c[:, :, idx % cap] = x[:, :, idx]
    return c


def logical_keys(cache, Lk, ring, lo):
    """[B, H, Lk, D] host tensor of the keys a call over `cache` reads: key j is
    cache row j (strided) or row j mod capacity (ring).  Keys below `lo` are
    outside every row's window and may have been overwritten in a ring; they
    are filled with zeros (they get weight 0 in the oracle too)."""
    c = cache.cpu()
    cap = c.shape[2]
    out = torch.zeros(c.shape[0], c.shape[1], Lk, c.shape[3], dtype=c.dtype)
    j = torch.arange(lo, Lk)
    out[:, :, lo:] = c[:, :, (j % cap) if ring else j]
    return out


def first_visible_key(Lq, Lk, window):
    return max(0, Lk - Lq - window + 1) if window else 0


def check_oracle(got, q, kc, vc, Lk, ring, window, dtype):
    Lq = q.shape[2]
    lo = first_visible_key(Lq, Lk, window)
    kl, vl = logical_keys(kc, Lk, ring, lo), logical_keys(vc, Lk, ring, lo)
    ref = oracle.sdpa(q.cpu(), kl, vl, causal=True, window=window)
    g = got.cpu().double().numpy()
    assert np.isfinite(g).all()
    err = float(np.max(np.abs(g - ref)))
    assert err < TOL[dtype], f"max abs err {err}"


PREFILL = [
    # B, Hq, Hkv, Lq, Lk, D, window, cap, ring
    (1, 8, 4, 300, 3000, 256, 0, 4096, False),     # 2-SM variant, persistent, strided
    (1, 4, 2, 300, 3000, 192, 0, 3200, False),     # one-CTA variant, strided
    (1, 8, 4, 300, 10000, 256, 1024, 1408, True),  # 2-SM variant, wrapped ring
    (1, 4, 4, 200, 5000, 256, 100, 384, True),     # one CTA (short window), wrapped ring
    (1, 4, 2, 150, 4000, 512, 512, 768, True),     # head-dim-split pair, wrapped ring
    (1, 8, 4, 300, 700, 256, 1024, 1024, True),    # ring not yet wrapped
    (1, 4, 2, 200, 3000, 512, 0, 3100, False),     # head-dim-split pair, strided, no window
]


@pytest.mark.parametrize("case", PREFILL)
def test_prefill_from_cache(case):
    B, Hq, Hkv, Lq, Lk, D, window, cap, ring = case
    dtype = torch.float16
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed=Lk + D)
    want = gb.sdpa_prefill(q, k, v, causal=True, window=window)
    make = ring_cache if ring else strided_cache
    kc, vc = make(k, cap, 1), make(v, cap, 2)
    got = gb.sdpa_prefill(q, kc, vc, causal=True, window=window, lk=Lk, ring=ring)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    check_oracle(got, q, kc, vc, Lk, ring, window, dtype)
    assert torch.equal(got, want)


DECODE = [
    # B, Hq, Hkv, Lk, D, window, cap, ring
    (1, 16, 8, 20000, 256, 1024, 1152, True),   # wrapped ring (sliding layer)
    (1, 16, 1, 20000, 512, 0, 24576, False),    # strided full-attention cache
    (2, 8, 2, 3000, 192, 0, 3072, False),
    (1, 16, 8, 900, 256, 1024, 1152, True),     # ring not yet wrapped
    (1, 16, 1, 5000, 512, 1024, 1152, True),    # head-dim-split pair over a wrapped ring
]


@pytest.mark.parametrize("Lq", [1, 4, 8])
@pytest.mark.parametrize("case", DECODE)
def test_decode_from_cache(case, Lq):
    B, Hq, Hkv, Lk, D, window, cap, ring = case
    dtype = torch.bfloat16
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed=Lk + Lq)
    want = gb.sdpa_decode(q, k, v, causal=True, window=window)
    make = ring_cache if ring else strided_cache
    kc, vc = make(k, cap, 3), make(v, cap, 4)
    got = gb.sdpa_decode(q, kc, vc, causal=True, window=window, lk=Lk, ring=ring)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    check_oracle(got, q, kc, vc, Lk, ring, window, dtype)
    assert torch.equal(got, want)


def test_verify_rows_over_a_ring_match_single_row_calls():
    """Row i of an Lq = M verify call over a wrapped ring equals the Lq = 1 call
    over the trimmed prefix (Lk - M + 1 + i keys) of the same ring, and every row
    matches the oracle on the logical keys."""
    B, Hq, Hkv, Lk, D, window, cap = 1, 16, 8, 20000, 256, 1024, 1152
    M = 4
    q, k, v = draw(B, Hq, Hkv, M, Lk, D, torch.float16, seed=5)
    kc, vc = ring_cache(k, cap, 6), ring_cache(v, cap, 7)
    block = gb.sdpa_decode(q, kc, vc, causal=True, window=window, lk=Lk, ring=True)
    torch.cuda.synchronize()
    check_oracle(block, q, kc, vc, Lk, True, window, torch.float16)
    for i in range(M):
        row = gb.sdpa_decode(q[:, :, i:i + 1].contiguous(), kc, vc, causal=True, window=window,
                             lk=Lk - M + 1 + i, ring=True)
        assert torch.equal(block[:, :, i], row[:, :, 0]), i


def test_logical_key_builder_reads_ring_rows():
    """The test's own key builder: a ring of capacity 256 holding keys 0..599
    puts key j in row j mod 256; the builder reads it back from there."""
    x = torch.arange(600, dtype=torch.float32).view(1, 1, 600, 1).expand(1, 1, 600, 8)
    x = x.contiguous().to(torch.float16).to(DEV)
    ring = ring_cache(x, 256, 0)
    back = logical_keys(ring, 600, True, 600 - 256)
    assert torch.equal(back[:, :, 600 - 256:], x.cpu()[:, :, 600 - 256:])


@pytest.mark.parametrize("kw", [dict(cap=1000, ring=True),     # not a multiple of 128
                                dict(cap=896, ring=True),      # misses keys the window sees
                                dict(cap=2000, ring=False)])   # shorter than Lk
def test_bad_cache_layouts_are_rejected(kw):
    q, k, v = draw(1, 4, 2, 4, 3000, 256, torch.float16, seed=8)
    kc = torch.zeros(1, 2, kw["cap"], 256, dtype=torch.float16, device=DEV)
    with pytest.raises(gb.SdpaError):
        gb.sdpa_decode(q, kc, kc.clone(), causal=True, window=1024, lk=3000, ring=kw["ring"])
