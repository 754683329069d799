"""GPU parity of the persistent prefill schedule (head_dim 128/192/256 with a workspace).

Resident units take the query tiles in waves, then share the leftover partial
wave by key tiles: a leftover tile's prefix stays on one unit, its suffix is cut
into pieces on the other units, and the prefix unit merges their fp32 partials
in key order.  The shapes below make the leftover wave split over many suffix
pieces (full waves plus a tail, fewer query tiles than units, a sliding window);
rows are sampled across every query tile, with all rows of the last (leftover)
tiles, and compared with the fp64 oracle.  The merge order is fixed, so a
repeated call is bit-identical, and a workspace that still holds the flags of
the previous call must not leak that call's partials.
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

CASES = [
    # B, Hq, Hkv, Lq, Lk, causal, window
    (1, 20, 4, 1024, 8192, True, 0),     # one full wave of 256-row tiles plus a split tail
    (1, 4, 2, 512, 16384, True, 0),      # 8 query tiles, far fewer than units
    (2, 3, 3, 700, 5000, False, 0),      # non-causal, ragged last query tile
    (1, 8, 2, 2048, 6000, True, 1024),   # sliding window on the 2-SM variant
]


def draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lq, D, generator=g).to(dtype)
    k = torch.randn(B, Hkv, Lk, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, Lk, D, generator=g).to(dtype)
    return q, k, v


def rows_to_check(B, Hq, Lq, seed):
    """Every row of the first 256 queries of each head (the last query tiles in
    the schedule's order), plus 64 random rows per head."""
    rng = np.random.default_rng(seed)
    ids = []
    for b in range(B):
        for h in range(Hq):
            base = (b * Hq + h) * Lq
            ids.extend(base + i for i in range(min(Lq, 256)))
            ids.extend(base + int(i) for i in rng.integers(0, Lq, 64))
    return np.unique(np.asarray(ids, dtype=np.int64))


def check_against_oracle(case, dtype, D):
    B, Hq, Hkv, Lq, Lk, causal, window = case
    assert gb.prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, causal, window) > 0
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, dtype, seed=sum(case))
    scale = 1.0 / math.sqrt(D)
    out = gb.sdpa_prefill(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=causal,
                          window=window)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    ids = rows_to_check(B, Hq, Lq, seed=len(case))
    ref = oracle.sdpa(q, k, v, scale=scale, causal=causal, window=window, rows=ids)
    got = out.reshape(-1, D)[torch.as_tensor(ids, device=DEV)].double().cpu().numpy()
    err = float(np.max(np.abs(got - ref)))
    assert err < TOL[dtype], f"max abs err {err}"


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", CASES)
def test_persistent_prefill_matches_oracle(case, dtype):
    check_against_oracle(case, dtype, 256)


@pytest.mark.parametrize("D", [128, 192])
@pytest.mark.parametrize("case", [CASES[0], CASES[3]])
def test_persistent_prefill_other_head_dims(case, D):
    """head_dim 128 runs the 2-SM variant, 192 the one-CTA variant."""
    check_against_oracle(case, torch.float16, D)


def test_persistent_prefill_is_deterministic_and_ignores_stale_flags():
    B, Hq, Hkv, Lq, Lk, causal, window = CASES[0]
    D = 256
    need = gb.prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, causal, window)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    q, k, v = (x.to(DEV) for x in draw(B, Hq, Hkv, Lq, Lk, D, torch.float16, seed=11))
    a = gb.sdpa_prefill(q, k, v, causal=causal, window=window, workspace=ws)
    b = gb.sdpa_prefill(q, k, v, causal=causal, window=window, workspace=ws)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    assert torch.equal(a, b)
    # Same workspace, new inputs: partials and flags of the previous call are
    # still there and must be ignored (each launch waits for its own epoch).
    q2, k2, v2 = draw(B, Hq, Hkv, Lq, Lk, D, torch.float16, seed=12)
    c = gb.sdpa_prefill(q2.to(DEV), k2.to(DEV), v2.to(DEV), causal=causal, window=window,
                        workspace=ws)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    ids = rows_to_check(B, Hq, Lq, seed=3)
    ref = oracle.sdpa(q2, k2, v2, causal=causal, window=window, rows=ids)
    got = c.reshape(-1, D)[torch.as_tensor(ids, device=DEV)].double().cpu().numpy()
    assert float(np.max(np.abs(got - ref))) < TOL[torch.float16]


def test_persistent_and_per_tile_launch_agree():
    """With a workspace too small for the persistent schedule the call falls back
    to one CTA pair per query tile; both results match the oracle."""
    B, Hq, Hkv, Lq, Lk, causal, window = CASES[1]
    D = 256
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, torch.bfloat16, seed=21)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    a = gb.sdpa_prefill(qd, kd, vd, causal=causal, window=window)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    b = gb.sdpa_prefill(qd, kd, vd, causal=causal, window=window, workspace=small)
    torch.cuda.synchronize()
    assert gb.device_status()[0] == 0
    ids = rows_to_check(B, Hq, Lq, seed=4)
    ref = oracle.sdpa(q, k, v, causal=causal, window=window, rows=ids)
    sel = torch.as_tensor(ids, device=DEV)
    for out in (a, b):
        got = out.reshape(-1, D)[sel].double().cpu().numpy()
        assert float(np.max(np.abs(got - ref))) < TOL[torch.bfloat16]


@pytest.mark.parametrize("rep", range(3))
def test_persistent_prefill_under_contention(rep):
    """The persistent grid is sized to the occupancy limit and its units wait
    (bounded) on one another.  Here cuBLAS GEMMs on another stream hold the SMs
    while the prefill is queued, so its units become resident piecemeal.  The
    call must either match the oracle or report the timeout through the device
    status, never return wrong numbers with a clean status."""
    B, Hq, Hkv, Lq, Lk, causal, window = CASES[0]
    D = 256
    q, k, v = draw(B, Hq, Hkv, Lq, Lk, D, torch.float16, seed=31 + rep)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    need = gb.prefill_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, causal, window)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    out = torch.empty_like(qd)
    n = 4096 + 2048 * rep
    a = torch.randn(n, n, device=DEV, dtype=torch.bfloat16)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        for _ in range(6):
            a = (a @ a) * (1.0 / n)
    gb.sdpa_prefill(qd, kd, vd, out, causal=causal, window=window, workspace=ws)
    with torch.cuda.stream(side):
        for _ in range(3):
            a = (a @ a) * (1.0 / n)
    torch.cuda.synchronize()
    status, detail = gb.device_status()
    ids = rows_to_check(B, Hq, Lq, seed=5 + rep)
    got = out.reshape(-1, D)[torch.as_tensor(ids, device=DEV)].double().cpu().numpy()
    if status != 0:
        assert detail == 0x10a, hex(detail)
        assert np.isnan(got).any()
        return
    ref = oracle.sdpa(q, k, v, causal=causal, window=window, rows=ids)
    assert float(np.max(np.abs(got - ref))) < TOL[torch.float16]
