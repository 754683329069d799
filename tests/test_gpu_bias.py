"""GPU parity of the additive bias (mask array) against the fp64 oracle.

"fix: gemma-4 long-prompt prefill OOMs on CUDA" (mlxcel issue #672, sections
"Root cause" and "Suggested fix direction") has models hand attention a dense
additive mask, and cuDNN's flash path take such a mask as a bias.  The kernels
add bias[b, h, i, j] to the scaled score on top of the causal / window flags;
-inf hides a key and a row with every key hidden outputs zeros.  Every variant
is covered (2-SM, one CTA, head-dim-split pair, persistent and per-tile
prefill, split decode), with broadcast shapes, vector and element-wise bias
reads, a ring cache, and decode row invariance.
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


def draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed, Dv=None):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lq, D, generator=g).to(dtype)
    k = torch.randn(B, Hkv, Lk, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, Lk, Dv or D, generator=g).to(dtype)
    return q, k, v


def make_bias(shape, Lk, dtype, seed, hide=0.25, pad=0):
    """N(0, 2) entries with about ``hide`` of them -inf, as a [.., Lk] view of a
    buffer whose rows are Lk + pad long (pad > 0 gives strides that are not
    16-byte multiples, so the kernel reads element by element)."""
    g = torch.Generator().manual_seed(seed)
    full = torch.randn(*shape, Lk + pad, generator=g) * 2.0
    full[torch.rand(*shape, Lk + pad, generator=g) < hide] = -math.inf
    full = full.to(dtype)
    return full[..., :Lk]


def sample_rows(B, Hq, Lq, seed, per_head=48):
    rng = np.random.default_rng(seed)
    ids = []
    for b in range(B):
        for h in range(Hq):
            base = (b * Hq + h) * Lq
            ids.extend(base + int(i) for i in rng.integers(0, Lq, per_head))
            ids.append(base + Lq - 1)
            ids.append(base)
    return np.unique(np.asarray(ids, dtype=np.int64))


def check(out, q, k, v, bias, scale, causal, window, ids, dtype, Dv):
    ref = oracle.sdpa(q, k, v, scale=scale, causal=causal, window=window, rows=ids,
                      bias=bias.cpu())
    got = out.reshape(-1, Dv)[torch.as_tensor(ids, device=DEV)].double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - ref)))
    assert err < TOL[dtype], f"max abs err {err}"


PREFILL = [
    # B, Hq, Hkv, Lq, Lk, D, Dv, causal, window, bias shape, pad
    (1, 8, 4, 600, 2100, 256, 256, True, 0, (1, 1, 600), 0),       # 2-SM, one mask for all heads
    (2, 4, 2, 300, 777, 256, 256, False, 0, (2, 4, 1), 0),         # per-head row bias, ragged Lk
    (1, 4, 2, 400, 1500, 256, 256, True, 100, (1, 4, 400), 3),     # one CTA, element-wise reads
    (1, 4, 2, 200, 900, 512, 512, True, 0, (1, 1, 200), 0),        # head-dim-split pair
    (1, 4, 4, 257, 1025, 192, 256, True, 0, (1, 1, 257), 5),       # Q/K 192, V 256
    (1, 8, 2, 512, 3000, 128, 128, True, 0, (1, 8, 512), 0),       # 2-SM, head dim 128
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", PREFILL)
def test_prefill_with_bias_matches_oracle(case, dtype):
    B, Hq, Hkv, Lq, Lk, D, Dv, causal, window, shape, pad = case
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed=Lq + Lk, Dv=Dv)
    bias = make_bias(shape, Lk, dtype, seed=Lk, pad=pad)
    scale = 1.0 / math.sqrt(D)
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=causal,
                          window=window, bias=_device_view(bias, pad))
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    check(out, q, k, v, bias.contiguous(), scale, causal, window,
          sample_rows(B, Hq, Lq, seed=Lq), dtype, Dv)


def _device_view(bias, pad):
    """The same [.., Lk] view on the device, rows still Lk + pad apart."""
    if pad == 0:
        return bias.contiguous().to(DEV)
    Lk = bias.shape[-1]
    full = torch.empty(*bias.shape[:-1], Lk + pad, dtype=bias.dtype)
    full[..., :Lk] = bias
    full[..., Lk:] = 0
    return full.to(DEV)[..., :Lk]


def test_persistent_prefill_with_bias_and_fully_hidden_rows():
    """Persistent schedule (suffix pieces merged by the prefix unit), with some
    rows whose every visible key the bias hides: those output zeros."""
    B, Hq, Hkv, Lq, Lk, D = 1, 20, 4, 1024, 8192, 256
    dtype = torch.float16
    assert gb.prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, True, 0) > 0
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed=71)
    bias = make_bias((1, Hq, 1), Lk, dtype, seed=72, hide=0.5)
    bias = bias.expand(1, Hq, Lq, Lk).clone()
    bias[0, 3, 17] = -math.inf
    bias[0, 11, 1000] = -math.inf
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, bias=bias.to(DEV))
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    ids = sample_rows(B, Hq, Lq, seed=73, per_head=16)
    ids = np.unique(np.concatenate([ids, [3 * Lq + 17, 11 * Lq + 1000]]))
    check(out, q, k, v, bias, 1.0 / math.sqrt(D), True, 0, ids, dtype, D)
    assert torch.all(out[0, 3, 17] == 0) and torch.all(out[0, 11, 1000] == 0)


def test_per_tile_prefill_with_bias_matches_persistent():
    B, Hq, Hkv, Lq, Lk, D = 1, 4, 2, 512, 16384, 256
    q, k, v = (x.to(DEV) for x in draw(B, Hq, Hkv, Lq, Lk, D, torch.bfloat16, seed=74))
    bias = make_bias((1, 1, Lq), Lk, torch.bfloat16, seed=75).to(DEV)
    a = gb.sdpa_prefill(q, k, v, causal=True, bias=bias)
    b = gb.sdpa_prefill(q, k, v, causal=True, bias=bias,
                        workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    assert float((a.double() - b.double()).abs().max()) < TOL[torch.bfloat16]


def test_zero_bias_and_flag_pattern_bias_match_the_plain_call():
    """A zero bias, and a 0/-inf bias holding the causal pattern on a call without
    flags, both give the plain causal result (to rounding: the bias path moves
    scores to the log2 domain one step earlier)."""
    B, Hq, Hkv, Lq, Lk, D = 1, 4, 2, 300, 700, 256
    q, k, v = (x.to(DEV) for x in draw(B, Hq, Hkv, Lq, Lk, D, torch.float16, seed=76))
    want = gb.sdpa_prefill(q, k, v, causal=True)
    zero = torch.zeros(1, 1, 1, Lk, dtype=torch.float16, device=DEV)
    i = torch.arange(Lq, device=DEV).view(-1, 1)
    j = torch.arange(Lk, device=DEV).view(1, -1)
    pattern = torch.zeros(Lq, Lk, device=DEV).masked_fill(j > Lk - Lq + i, -math.inf)
    pattern = pattern.to(torch.float16).view(1, 1, Lq, Lk)
    for got in (gb.sdpa_prefill(q, k, v, causal=True, bias=zero),
                gb.sdpa_prefill(q, k, v, causal=False, bias=pattern)):
        assert float((got.double() - want.double()).abs().max()) < 2e-3


DECODE = [
    # B, Hq, Hkv, Lk, D, window, cap, ring, bias shape (Lq filled in), pad
    (1, 16, 8, 9000, 256, 1024, 1152, True, "per_row", 0),
    (2, 16, 1, 5000, 512, 0, 5000, False, "shared", 0),
    (1, 8, 2, 3001, 192, 0, 3001, False, "per_row", 3),
]


@pytest.mark.parametrize("Lq", [1, 4, 8])
@pytest.mark.parametrize("case", DECODE)
def test_decode_with_bias_matches_oracle(case, Lq):
    B, Hq, Hkv, Lk, D, window, cap, ring, kind, pad = case
    dtype = torch.bfloat16
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed=Lk + Lq)
    shape = (B, Hq, Lq) if kind == "per_row" else (1, 1, Lq)
    bias = make_bias(shape, Lk, dtype, seed=Lq, pad=pad)
    kd, vd = k.to(DEV), v.to(DEV)
    if ring:
        kc = torch.zeros(B, Hkv, cap, D, dtype=dtype, device=DEV)
        vc = torch.zeros_like(kc)
        idx = torch.arange(max(0, Lk - cap), Lk, device=DEV)
        kc[:, :, idx % cap] = kd[:, :, idx]
        vc[:, :, idx % cap] = vd[:, :, idx]
        out = gb.sdpa_decode(q.to(DEV), kc, vc, causal=True, window=window, lk=Lk, ring=True,
                             bias=_device_view(bias, pad))
    else:
        out = gb.sdpa_decode(q.to(DEV), kd, vd, causal=True, window=window,
                             bias=_device_view(bias, pad))
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    ids = np.arange(B * Hq * Lq, dtype=np.int64)
    check(out, q, k, v, bias.contiguous(), 1.0 / math.sqrt(D), True, window, ids, dtype, D)


@pytest.mark.parametrize("D,window", [(256, 1024), (512, 0)])
def test_decode_rows_with_bias_match_single_row_calls(D, window):
    """Row i of an Lq = M call with a per-row bias equals, bit for bit, the Lq = 1
    call over the trimmed prefix (Lk - M + 1 + i keys) with that row's bias."""
    B, Hq, Hkv, Lk, M = 1, 16, 8 if D == 256 else 1, 6000, 8
    q, k, v = (x.to(DEV) for x in draw(B, Hq, Hkv, M, Lk, D, torch.float16, seed=D))
    bias = make_bias((B, Hq, M), Lk, torch.float16, seed=D + 1).to(DEV)
    block = gb.sdpa_decode(q, k, v, causal=True, window=window, bias=bias)
    for i in range(M):
        n = Lk - M + 1 + i
        row = gb.sdpa_decode(q[:, :, i:i + 1].contiguous(), k[:, :, :n].contiguous(),
                             v[:, :, :n].contiguous(), causal=True, window=window,
                             bias=bias[:, :, i:i + 1, :n])
        assert torch.equal(block[:, :, i], row[:, :, 0]), i
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0


@pytest.mark.parametrize("bad", [dict(shape=(1, 1, 1, 99)), dict(shape=(1, 3, 1, 100)),
                                 dict(shape=(1, 1, 1, 100), dtype=torch.bfloat16),
                                 dict(shape=(1, 1, 1, 100), on_cpu=True),
                                 dict(shape=(1, 1, 100, 1), transpose=True)])
def test_bad_bias_is_rejected(bad):
    q, k, v = (x.to(DEV) for x in draw(1, 4, 2, 4, 100, 256, torch.float16, seed=77))
    b = torch.zeros(*bad["shape"], dtype=bad.get("dtype", torch.float16),
                    device="cpu" if bad.get("on_cpu") else DEV)
    if bad.get("transpose"):
        b = torch.zeros(1, 1, 100, 4, dtype=torch.float16, device=DEV).transpose(2, 3)
    with pytest.raises((ValueError, TypeError)):
        gb.sdpa_decode(q, k, v, causal=True, bias=b)
