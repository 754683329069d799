"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test is chosen so that a plausible mistake in the oracle (a wrong mask
edge, a wrong GQA head map, a dropped term of the contraction, a bad fp16/bf16
widening, a wrong bottom-right offset) fails at least one of them:

* a library routine: torch's scaled_dot_product_attention in float64 with an
  explicit boolean mask;
* brute force with numpy on tiny inputs;
* closed forms (one key, window 1, constant values, zero query, huge scale);
* invariants named by the method (rows of P sum to 1, window >= Lk equals
  causal, GQA equals MHA over repeated KV heads, D=256 scores are the sum of
  the two D=128 halves, causal rows equal prefix attention);
* the pages' own printed numbers (input byte counts) and a hand-derived
  two-key example, under tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from attention_sm_flash_attn_gb300.inputs import LONGKV, PREFILL128K, Workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_qkv(B, Hq, Hkv, Lq, Lk, D, dtype=torch.float16, seed=0, Dv=None, amp=1.0):
    g = torch.Generator().manual_seed(seed)
    Dv = D if Dv is None else Dv
    q = (torch.randn(B, Hq, Lq, D, generator=g) * amp).to(dtype)
    k = (torch.randn(B, Hkv, Lk, D, generator=g) * amp).to(dtype)
    v = (torch.randn(B, Hkv, Lk, Dv, generator=g) * amp).to(dtype)
    return q, k, v


def mask_matrix(Lq, Lk, causal, window):
    """Boolean [Lq, Lk] visibility built from index grids (bottom-right aligned)."""
    i = torch.arange(Lq).view(-1, 1)
    j = torch.arange(Lk).view(1, -1)
    p = Lk - Lq + i
    m = torch.ones(Lq, Lk, dtype=torch.bool)
    if causal:
        m &= j <= p
    if window:
        m &= (p - j) < window
    return m


def torch_reference(q, k, v, scale, causal, window):
    """torch's SDPA in float64 with an explicit mask; KV heads repeated for GQA."""
    G = q.shape[1] // k.shape[1]
    kk = k.double().repeat_interleave(G, dim=1)
    vv = v.double().repeat_interleave(G, dim=1)
    m = mask_matrix(q.shape[2], k.shape[2], causal, window)
    return F.scaled_dot_product_attention(q.double(), kk, vv, attn_mask=m, scale=scale)


CASES = [
    # B, Hq, Hkv, Lq, Lk, D, causal, window
    (1, 2, 1, 128, 128, 256, True, 0),
    (1, 2, 1, 128, 128, 256, True, 32),
    (2, 4, 2, 33, 97, 256, True, 7),
    (1, 4, 1, 5, 160, 512, True, 1),
    (1, 4, 4, 64, 64, 256, False, 0),
    (2, 2, 2, 17, 150, 512, False, 0),
    (1, 4, 2, 40, 40, 256, True, 200),
    (1, 3, 1, 1, 129, 256, True, 0),
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", CASES)
def test_matches_torch_sdpa_float64(case, dtype):
    B, Hq, Hkv, Lq, Lk, D, causal, window = case
    q, k, v = rand_qkv(B, Hq, Hkv, Lq, Lk, D, dtype, seed=hash(case) % 1000)
    scale = 1.0 / math.sqrt(D)
    got = oracle.sdpa(q, k, v, scale=scale, causal=causal, window=window)
    ref = torch_reference(q, k, v, scale, causal, window).numpy()
    assert np.max(np.abs(got - ref)) < 1e-12


def numpy_dense(q, k, v, scale, causal, window):
    """Brute force: dense scores, explicit per-element mask loop, direct softmax."""
    q = q.double().numpy()
    k = k.double().numpy()
    v = v.double().numpy()
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, Lq, v.shape[3]))
    for b in range(B):
        for h in range(Hq):
            s = scale * q[b, h] @ k[b, h // G].T
            for i in range(Lq):
                for j in range(Lk):
                    p = Lk - Lq + i
                    if (causal and j > p) or (window and p - j >= window):
                        s[i, j] = -np.inf
            e = np.exp(s - s.max(axis=1, keepdims=True))
            out[b, h] = (e / e.sum(axis=1, keepdims=True)) @ v[b, h // G]
    return out


@pytest.mark.parametrize("case", [(1, 2, 1, 12, 20, 256, True, 3), (1, 4, 2, 9, 9, 512, True, 0),
                                  (2, 2, 1, 6, 11, 256, False, 0)])
def test_matches_numpy_brute_force(case):
    B, Hq, Hkv, Lq, Lk, D, causal, window = case
    q, k, v = rand_qkv(B, Hq, Hkv, Lq, Lk, D, torch.bfloat16, seed=7)
    scale = 1.0 / math.sqrt(D)
    got = oracle.sdpa(q, k, v, scale=scale, causal=causal, window=window)
    ref = numpy_dense(q, k, v, scale, causal, window)
    assert np.max(np.abs(got - ref)) < 1e-12


@pytest.mark.parametrize("dims", [(128, 128), (192, 192), (192, 256)])
def test_other_head_dims_match_torch_and_brute_force(dims):
    """Head dims 128 and 192, and Q/K 192 with V 256: scores over Dqk columns,
    output over Dv, against both independent references."""
    D, Dv = dims
    q, k, v = rand_qkv(1, 4, 2, 13, 29, D, torch.float16, seed=D + Dv, Dv=Dv)
    scale = 1.0 / math.sqrt(D)
    for causal, window in ((True, 0), (True, 7), (False, 0)):
        got = oracle.sdpa(q, k, v, scale=scale, causal=causal, window=window)
        assert got.shape == (1, 4, 13, Dv)
        ref = torch_reference(q, k, v, scale, causal, window).numpy()
        assert np.max(np.abs(got - ref)) < 1e-12
        assert np.max(np.abs(got - numpy_dense(q, k, v, scale, causal, window))) < 1e-12


def test_two_key_worked_example():
    gold = json.load(open(os.path.join(GOLDEN, "two_key_softmax.json")))
    D = 256
    q = torch.zeros(1, 1, 1, D, dtype=torch.float16)
    k = torch.zeros(1, 1, 2, D, dtype=torch.float16)
    v = torch.zeros(1, 1, 2, D, dtype=torch.float16)
    q[0, 0, 0, 0] = 1
    k[0, 0, 0, 0] = 1
    k[0, 0, 1, 1] = 1
    v[0, 0, 0, 0] = 1
    v[0, 0, 1, 1] = 1
    o = oracle.sdpa(q, k, v, scale=1.0)[0, 0, 0]
    np.testing.assert_allclose(o[:2], gold["expected_out_first_two"], rtol=0, atol=1e-15)
    assert np.all(o[2:] == 0)


# ---------------------------------------------------------------- closed forms

def test_single_key_returns_that_value_exactly():
    q, k, v = rand_qkv(1, 4, 2, 3, 1, 256, torch.float16, seed=3)
    o = oracle.sdpa(q, k, v, causal=False)
    want = v.double().repeat_interleave(2, dim=1)[:, :, 0:1, :].expand(-1, -1, 3, -1).numpy()
    assert np.array_equal(o, want)


@pytest.mark.parametrize("Lq,Lk", [(16, 16), (5, 40)])
def test_window_one_returns_own_value(Lq, Lk):
    q, k, v = rand_qkv(1, 2, 1, Lq, Lk, 256, torch.bfloat16, seed=4)
    o = oracle.sdpa(q, k, v, causal=True, window=1)
    vv = v.double().numpy()[0, 0]
    for h in range(2):
        for i in range(Lq):
            assert np.array_equal(o[0, h, i], vv[Lk - Lq + i])


def test_constant_values_give_that_constant():
    q, k, _ = rand_qkv(1, 2, 1, 20, 50, 256, torch.float16, seed=5)
    c = torch.linspace(-3, 3, 256).to(torch.float16)
    v = c.view(1, 1, 1, -1).expand(1, 1, 50, 256).contiguous()
    o = oracle.sdpa(q, k, v, causal=True, window=9)
    np.testing.assert_allclose(o, np.broadcast_to(c.double().numpy(), o.shape), rtol=1e-14,
                               atol=1e-15)


@pytest.mark.parametrize("window", [0, 1, 6])
def test_zero_query_gives_mean_of_visible_values(window):
    Lq, Lk = 12, 30
    _, k, v = rand_qkv(1, 1, 1, Lq, Lk, 256, torch.float16, seed=6)
    q = torch.zeros(1, 1, Lq, 256, dtype=torch.float16)
    o = oracle.sdpa(q, k, v, causal=True, window=window)
    vv = torch.cat([torch.zeros(1, 256, dtype=torch.float64), v[0, 0].double().cumsum(0)])
    for i in range(Lq):
        p = Lk - Lq + i
        lo = 0 if window == 0 else max(0, p - window + 1)
        mean = (vv[p + 1] - vv[lo]) / (p + 1 - lo)
        np.testing.assert_allclose(o[0, 0, i], mean.numpy(), rtol=1e-12, atol=1e-13)


def test_huge_scale_selects_argmax_key():
    q, k, v = rand_qkv(1, 2, 2, 6, 24, 256, torch.float16, seed=8)
    scale = 1e7
    o = oracle.sdpa(q, k, v, scale=scale, causal=True)
    s = torch.einsum("bhid,bhjd->bhij", q.double(), k.double())
    m = mask_matrix(6, 24, True, 0)
    s = s.masked_fill(~m, -float("inf"))
    idx = s.argmax(-1)
    for h in range(2):
        for i in range(6):
            assert np.array_equal(o[0, h, i], v[0, h, idx[0, h, i]].double().numpy())


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5)])
def test_probability_rows_sum_to_one(causal, window):
    q, k, _ = rand_qkv(1, 4, 2, 10, 37, 256, torch.bfloat16, seed=9)
    for h in range(4):
        for i in (0, 4, 9):
            P = oracle.row_probs(q, k, 0, h, i, causal=causal, window=window)
            assert abs(P.sum() - 1.0) < 1e-13
            assert np.all(P >= 0)
            m = mask_matrix(10, 37, causal, window)[i].numpy()
            assert np.all(P[~m] == 0) and np.all(P[m] > 0)


@pytest.mark.parametrize("W", [64, 65, 1000])
def test_window_at_least_lk_equals_causal(W):
    q, k, v = rand_qkv(1, 2, 1, 40, 64, 256, torch.float16, seed=10)
    a = oracle.sdpa(q, k, v, causal=True, window=W)
    b = oracle.sdpa(q, k, v, causal=True, window=0)
    assert np.array_equal(a, b)


def test_window_below_lk_differs_from_causal():
    q, k, v = rand_qkv(1, 2, 1, 40, 64, 256, torch.float16, seed=10)
    a = oracle.sdpa(q, k, v, causal=True, window=63)
    b = oracle.sdpa(q, k, v, causal=True, window=0)
    assert not np.array_equal(a, b)


def test_gqa_equals_mha_with_repeated_kv_heads():
    q, k, v = rand_qkv(2, 8, 2, 9, 21, 256, torch.bfloat16, seed=11)
    a = oracle.sdpa(q, k, v, causal=True, window=4)
    b = oracle.sdpa(q, k.repeat_interleave(4, dim=1).contiguous(),
                    v.repeat_interleave(4, dim=1).contiguous(), causal=True, window=4)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("D", [256, 512])
def test_scores_are_sum_of_two_half_dim_contractions(D):
    q, k, _ = rand_qkv(1, 2, 1, 4, 33, D, torch.float16, seed=12)
    h = D // 2
    q1, q2 = q[..., :h].contiguous(), q[..., h:].contiguous()
    k1, k2 = k[..., :h].contiguous(), k[..., h:].contiguous()
    for head in range(2):
        for i in range(4):
            full = oracle.row_scores(q, k, 0, head, i, scale=1.0)
            halves = (oracle.row_scores(q1, k1, 0, head, i, scale=1.0)
                      + oracle.row_scores(q2, k2, 0, head, i, scale=1.0))
            np.testing.assert_allclose(full, halves, rtol=1e-13, atol=1e-12)
            # and neither half alone is the full product
            assert np.max(np.abs(full - oracle.row_scores(q1, k1, 0, head, i, scale=1.0))) > 1e-3


def test_scores_scale_multiplies():
    q, k, _ = rand_qkv(1, 1, 1, 2, 9, 256, torch.float16, seed=13)
    a = oracle.row_scores(q, k, 0, 0, 1, scale=1.0)
    b = oracle.row_scores(q, k, 0, 0, 1, scale=0.0625)
    np.testing.assert_allclose(b, a * 0.0625, rtol=1e-15, atol=0)
    dots = (q[0, 0, 1].double() @ k[0, 0].double().T).numpy()
    np.testing.assert_allclose(a, dots, rtol=1e-13, atol=1e-12)


def test_key_permutation_invariance_noncausal():
    q, k, v = rand_qkv(1, 2, 1, 7, 50, 256, torch.float16, seed=14)
    perm = torch.randperm(50, generator=torch.Generator().manual_seed(1))
    a = oracle.sdpa(q, k, v, causal=False)
    b = oracle.sdpa(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), causal=False)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_causal_row_equals_prefix_attention():
    L = 24
    q, k, v = rand_qkv(1, 2, 1, L, L, 256, torch.bfloat16, seed=15)
    a = oracle.sdpa(q, k, v, causal=True)
    for i in (0, 1, 11, 23):
        b = oracle.sdpa(q[:, :, i:i + 1].contiguous(), k[:, :, :i + 1].contiguous(),
                        v[:, :, :i + 1].contiguous(), causal=False)
        np.testing.assert_allclose(a[:, :, i], b[:, :, 0], rtol=0, atol=1e-14)


@pytest.mark.parametrize("window", [0, 5])
def test_bottom_right_row_equals_trimmed_prefix_call(window):
    """Row i of an Lq-row causal call equals the single-row call over keys [0, Lk-Lq+i]."""
    Lq, Lk = 4, 40
    q, k, v = rand_qkv(1, 4, 2, Lq, Lk, 256, torch.float16, seed=16)
    a = oracle.sdpa(q, k, v, causal=True, window=window)
    for i in range(Lq):
        n = Lk - Lq + i + 1
        b = oracle.sdpa(q[:, :, i:i + 1].contiguous(), k[:, :, :n].contiguous(),
                        v[:, :, :n].contiguous(), causal=True, window=window)
        assert np.array_equal(a[:, :, i], b[:, :, 0])


def test_rows_subset_matches_full_call():
    q, k, v = rand_qkv(2, 4, 2, 10, 30, 256, torch.float16, seed=17)
    full = oracle.sdpa(q, k, v, causal=True, window=7)
    ids = [0, 5, 17, 39, 40, 79]
    part = oracle.sdpa(q, k, v, causal=True, window=7, rows=ids)
    assert np.array_equal(part, full.reshape(-1, 256)[ids])


# ---------------------------------------------------------------- widening of inputs

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_input_widening_is_exact(dtype):
    """Lk = 1 makes the output equal to v[0]; compare with torch's own widening,
    including subnormals, the largest finite values and negative zero."""
    info = torch.finfo(dtype)
    special = torch.tensor([0.0, -0.0, 1.0, -1.5, info.max, -info.max, info.tiny,
                            info.tiny / 4, 3.140625, 65504.0 if dtype == torch.float16 else 1e30],
                           dtype=torch.float64).to(dtype)
    D = 256
    vals = torch.cat([special, torch.randn(D - special.numel(),
                                           generator=torch.Generator().manual_seed(2)).to(dtype)])
    v = vals.view(1, 1, 1, D).contiguous()
    q = torch.ones(1, 1, 1, D, dtype=dtype)
    k = torch.ones(1, 1, 1, D, dtype=dtype)
    o = oracle.sdpa(q, k, v, causal=False, scale=0.0)
    assert np.array_equal(o[0, 0, 0], vals.double().numpy())


# ---------------------------------------------------------------- argument checks

@pytest.mark.parametrize("kw", [dict(causal=False, window=4), dict(causal=True, window=-1)])
def test_rejects_bad_mask_arguments(kw):
    q, k, v = rand_qkv(1, 2, 1, 4, 8, 256)
    with pytest.raises(ValueError):
        oracle.sdpa(q, k, v, **kw)


def test_rejects_causal_with_more_queries_than_keys():
    q, k, v = rand_qkv(1, 2, 1, 9, 8, 256)
    with pytest.raises(ValueError):
        oracle.sdpa(q, k, v, causal=True)


def test_rejects_indivisible_heads():
    q, k, v = rand_qkv(1, 3, 2, 4, 8, 256)
    with pytest.raises(ValueError):
        oracle.sdpa(q, k, v)


# ---------------------------------------------------------------- the pages' numbers

def test_workload_shapes_reproduce_the_pages_input_sizes():
    gold = json.load(open(os.path.join(GOLDEN, "page_input_sizes.json")))
    hd = gold["heads"]
    for row in gold["rows"]:
        nbytes = hd["bytes_per_elem"] * hd["head_dim"] * (
            hd["n_q"] * row["qL"] + 2 * hd["n_kv"] * row["kL"])
        assert nbytes == row["inputs_MiB"] * 2 ** 20
    # the named workloads use the same head geometry
    for w in (LONGKV, PREFILL128K):
        assert (w.Hq, w.Hkv, w.D) == (hd["n_q"], hd["n_kv"], hd["head_dim"])
    assert (LONGKV.Lq, LONGKV.Lk) == (gold["rows"][0]["qL"], gold["rows"][0]["kL"])
    assert (PREFILL128K.Lq, PREFILL128K.Lk) == (gold["rows"][2]["qL"], gold["rows"][2]["kL"])


# --- additive bias (mask array) ------------------------------------------------
# "fix: gemma-4 long-prompt prefill OOMs on CUDA" (mlxcel issue #672, sections
# "Root cause" and "Suggested fix direction") describes the model handing SDPA a
# dense additive mask (0 for a visible key, -inf for a hidden one) and cuDNN's
# flash path taking such a mask as a bias.  The bias is added to the scaled
# scores; a row whose keys are all hidden outputs zeros.

BIAS_SHAPES = [(1, 1, 1), (2, 1, 1), (1, 4, 1), (1, 1, 9), (2, 4, 9)]


def rand_bias(shape, Lk, dtype, seed, hide=0.3):
    """Finite N(0, 2) entries with about ``hide`` of them -inf."""
    g = torch.Generator().manual_seed(seed)
    b = torch.randn(*shape, Lk, generator=g) * 2.0
    b[torch.rand(*shape, Lk, generator=g) < hide] = -math.inf
    return b.to(dtype)


def torch_bias_reference(q, k, v, scale, causal, window, bias):
    """torch's SDPA in float64 with a float mask: the bias plus -inf where the
    causal / window flags hide a key; rows left without keys are zeros."""
    G = q.shape[1] // k.shape[1]
    kk = k.double().repeat_interleave(G, dim=1)
    vv = v.double().repeat_interleave(G, dim=1)
    m = mask_matrix(q.shape[2], k.shape[2], causal, window)
    add = bias.double().expand(q.shape[0], q.shape[1], q.shape[2], k.shape[2]).clone()
    add = add.masked_fill(~m, -math.inf)
    out = F.scaled_dot_product_attention(q.double(), kk, vv, attn_mask=add, scale=scale)
    empty = torch.isinf(add).all(dim=-1, keepdim=True)
    return out.masked_fill(empty, 0.0)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", BIAS_SHAPES)
def test_bias_matches_torch_sdpa_float_mask(shape, dtype):
    B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 9, 40, 256
    q, k, v = rand_qkv(B, Hq, Hkv, Lq, Lk, D, dtype, seed=31)
    bias = rand_bias(shape, Lk, dtype, seed=sum(shape))
    scale = 1.0 / math.sqrt(D)
    for causal, window in ((False, 0), (True, 0), (True, 5)):
        got = oracle.sdpa(q, k, v, scale=scale, causal=causal, window=window, bias=bias)
        ref = torch_bias_reference(q, k, v, scale, causal, window, bias).numpy()
        assert np.max(np.abs(got - ref)) < 1e-12, (causal, window)


def test_bias_matches_numpy_brute_force():
    """Dense scores plus the bias element by element, softmax by hand."""
    B, Hq, Hkv, Lq, Lk, D, Dv = 1, 2, 1, 6, 11, 192, 256
    q, k, v = rand_qkv(B, Hq, Hkv, Lq, Lk, D, torch.bfloat16, seed=33, Dv=Dv)
    bias = rand_bias((B, Hq, Lq), Lk, torch.bfloat16, seed=34, hide=0.2)
    bias[0, 1, 2, :] = -math.inf          # one row with every key hidden
    scale = 0.07
    got = oracle.sdpa(q, k, v, scale=scale, causal=False, bias=bias)
    qn, kn, vn, bn = (x.double().numpy() for x in (q, k, v, bias))
    for h in range(Hq):
        for i in range(Lq):
            s = [scale * float(np.dot(qn[0, h, i], kn[0, 0, j])) + bn[0, h, i, j]
                 for j in range(Lk)]
            if all(x == -math.inf for x in s):
                want = np.zeros(Dv)
            else:
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                want = sum(e[j] * vn[0, 0, j] for j in range(Lk)) / sum(e)
            assert np.max(np.abs(got[0, h, i] - want)) < 1e-12, (h, i)


def test_zero_bias_equals_no_bias_exactly():
    q, k, v = rand_qkv(1, 4, 2, 17, 60, 256, torch.float16, seed=35)
    for causal, window in ((False, 0), (True, 0), (True, 9)):
        a = oracle.sdpa(q, k, v, causal=causal, window=window)
        z = torch.zeros(1, 1, 1, 60, dtype=torch.float16)
        assert np.array_equal(a, oracle.sdpa(q, k, v, causal=causal, window=window, bias=z))


@pytest.mark.parametrize("window", [0, 7])
def test_inf_bias_pattern_equals_the_mask_flags(window):
    """A 0/-inf bias holding the bottom-right causal (and window) pattern, on a
    call without flags, gives the flagged call's result exactly."""
    Lq, Lk = 13, 50
    q, k, v = rand_qkv(1, 2, 1, Lq, Lk, 256, torch.bfloat16, seed=36)
    m = mask_matrix(Lq, Lk, True, window)
    bias = torch.zeros(1, 1, Lq, Lk).masked_fill(~m, -math.inf).to(torch.bfloat16)
    want = oracle.sdpa(q, k, v, causal=True, window=window)
    assert np.array_equal(oracle.sdpa(q, k, v, causal=False, bias=bias), want)


def test_row_constant_bias_cancels():
    """Softmax is invariant to a constant added across a row: a bias constant
    along keys (different per head and row) leaves the result unchanged."""
    q, k, v = rand_qkv(1, 4, 2, 8, 30, 256, torch.float16, seed=37)
    c = torch.tensor([0.5, -3.0, 8.0, 1.25]).view(1, 4, 1, 1) * torch.ones(1, 4, 8, 30)
    c = c + torch.arange(8).view(1, 1, 8, 1) * 0.25
    a = oracle.sdpa(q, k, v, causal=True)
    b = oracle.sdpa(q, k, v, causal=True, bias=c.to(torch.float16))
    assert np.max(np.abs(a - b)) < 1e-12


def test_log_weight_bias_with_zero_query_gives_weighted_mean():
    """With q = 0 every score is the bias, so a bias of log w_j makes the output
    the w-weighted mean of the values: sum_j w_j v_j / sum_j w_j."""
    Lk, D = 24, 256
    _, k, v = rand_qkv(1, 1, 1, 1, Lk, D, torch.float16, seed=38)
    q = torch.zeros(1, 1, 1, D, dtype=torch.float16)
    logw = torch.linspace(-2.0, 2.0, Lk).to(torch.float16)
    w = np.exp(logw.double().numpy())
    got = oracle.sdpa(q, k, v, causal=False, bias=logw.view(1, 1, 1, Lk))
    want = (w[:, None] * v[0, 0].double().numpy()).sum(0) / w.sum()
    assert np.max(np.abs(got[0, 0, 0] - want)) < 1e-12


def test_fully_hidden_rows_output_zeros():
    q, k, v = rand_qkv(1, 2, 1, 4, 10, 256, torch.float16, seed=39)
    bias = torch.zeros(1, 2, 4, 10, dtype=torch.float16)
    bias[0, 0, 1] = -math.inf
    bias[0, 1, 3, 5:] = -math.inf        # with causal, row 3 sees keys 0..9; keep 0..4
    bias[0, 1, 0, :7] = -math.inf        # row 0 sees keys 0..6 under causal: all hidden
    got = oracle.sdpa(q, k, v, causal=True, bias=bias)
    assert np.all(got[0, 0, 1] == 0.0) and np.all(got[0, 1, 0] == 0.0)
    assert np.any(got[0, 1, 3] != 0.0)


def test_bias_rows_subset_matches_full_call():
    q, k, v = rand_qkv(2, 4, 2, 7, 33, 256, torch.bfloat16, seed=40)
    bias = rand_bias((2, 1, 7), 33, torch.bfloat16, seed=41)
    full = oracle.sdpa(q, k, v, causal=True, window=4, bias=bias).reshape(-1, 256)
    ids = np.array([0, 5, 13, 27, 55], dtype=np.int64)
    assert np.array_equal(oracle.sdpa(q, k, v, causal=True, window=4, bias=bias, rows=ids),
                          full[ids])


@pytest.mark.parametrize("bad", [(1, 1, 1, 39), (3, 1, 1, 40), (1, 3, 1, 40), (1, 1, 2, 40),
                                 (1, 40)])
def test_rejects_bias_that_does_not_broadcast(bad):
    q, k, v = rand_qkv(2, 4, 2, 9, 40, 256, torch.float16, seed=42)
    with pytest.raises(ValueError):
        oracle.sdpa(q, k, v, bias=torch.zeros(*bad, dtype=torch.float16))


def test_rejects_bias_of_another_dtype():
    q, k, v = rand_qkv(1, 2, 1, 4, 8, 256, torch.float16, seed=43)
    with pytest.raises(ValueError):
        oracle.sdpa(q, k, v, bias=torch.zeros(1, 1, 1, 8, dtype=torch.bfloat16))
