"""Seeded synthetic inputs and the named workload shapes.

This module holds no attention arithmetic: it only draws Q/K/V tensors from a
seeded generator and names the workload shapes.  Both the CUDA path's tests
and the CPU oracle's tests consume what it produces.

Recipe: Q, K, V are drawn i.i.d. N(0, 1) in fp32, in the order q, k, v, from one
``torch.Generator`` seeded with the workload's seed, multiplied by the
workload's ``amp`` and cast to its dtype (round to nearest even).  On a CUDA
device a CUDA generator is used (same recipe, different stream of numbers);
every comparison reads the cast values back, so either is reproducible.

Shapes follow the pages' workloads: "Fused SDPA full-attention for
head_dim=192/256" (MLX PR #3660, Microbenchmarks: n_q=16, n_kv=8, head_dim 256,
qL 1024/2048 over kL 32768..131072), "fix: add head_dim=256 to fused SDPA full
attention kernel" (MLX PR #3293, Benchmark: H=64, D=256, L=16384) and
"fix: Gemma 4 MTP never engages on CUDA (GB10)" (mlxcel issue #2160, Current
Behavior: 16/8 heads at head_dim 256 with window 1024, 1 KV head at 512;
32/16 sliding and 32/4 full layers).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    D: int
    dtype: torch.dtype
    causal: bool
    window: int
    seed: int
    amp: float = 1.0
    kind: str = "prefill"  # "prefill" or "decode"
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / float(self.D) ** 0.5

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The named workloads (B = 1 throughout).
TINY = Workload("tiny_causal_hd256", 1, 2, 1, 128, 128, 256, torch.float16, True, 0, 1)
TINY_W32 = TINY.with_(name="tiny_causal_w32_hd256", window=32)
LONGKV = Workload("longkv_gqa_prefill_hd256", 1, 16, 8, 1024, 32768, 256, torch.float16,
                  True, 0, 2, note="queries at positions 31744..32767")
SELF16K = Workload("causal_self_hd256_L16k", 1, 64, 8, 16384, 16384, 256, torch.bfloat16,
                   True, 0, 3, amp=0.5)
SLIDING32K = Workload("gemma_sliding_w1024_hd256_L32k", 1, 32, 16, 32768, 32768, 256,
                      torch.bfloat16, True, 1024, 41)
FULL512 = Workload("gemma_full_hd512_L32k", 1, 32, 4, 32768, 32768, 512, torch.bfloat16,
                   True, 0, 42)
PREFILL128K = Workload("longctx_prefill_hd256_q2k_k128k", 1, 16, 8, 2048, 131072, 256,
                       torch.float16, True, 0, 51)
DECODE_SLIDING = Workload("decode_sliding_w1024_hd256_k128k", 1, 16, 8, 1, 131072, 256,
                          torch.float16, True, 1024, 52, kind="decode")
DECODE_FULL512 = Workload("decode_full_hd512_k128k", 1, 16, 1, 1, 131072, 512,
                          torch.float16, True, 0, 53, kind="decode")

# head_dim 192, which "Fused SDPA full-attention for head_dim=192/256" (MLX PR
# #3660) serves alongside 256, and 128 as a regression shape: the long-KV GQA
# geometry above at those head dims.
LONGKV_HD192 = LONGKV.with_(name="longkv_gqa_prefill_hd192", D=192, seed=61)
LONGKV_HD128 = LONGKV.with_(name="longkv_gqa_prefill_hd128", D=128, seed=62)
DECODE_SLIDING_HD192 = DECODE_SLIDING.with_(name="decode_sliding_w1024_hd192_k128k", D=192,
                                            seed=63)

PREFILL_WORKLOADS = [TINY, TINY_W32, LONGKV, SELF16K, SLIDING32K, FULL512, PREFILL128K,
                     LONGKV_HD192, LONGKV_HD128]
DECODE_WORKLOADS = [DECODE_SLIDING, DECODE_FULL512, DECODE_SLIDING_HD192]
DECODE_LQ = (1, 2, 4, 8)


def make_qkv(w: Workload, device="cpu", seed: int | None = None):
    """Draw (q, k, v) for workload ``w`` on ``device`` following the module recipe."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    shapes = [(w.B, w.Hq, w.Lq, w.D), (w.B, w.Hkv, w.Lk, w.D), (w.B, w.Hkv, w.Lk, w.D)]
    out = []
    for shp in shapes:
        t = torch.randn(shp, generator=gen, device=device, dtype=torch.float32)
        if w.amp != 1.0:
            t.mul_(w.amp)
        out.append(t.to(w.dtype))
        del t
    return tuple(out)


def sample_rows(w: Workload, n_uniform: int = 32, heads=None, seed: int = 0):
    """Flat row ids (b * Hq + h) * Lq + i checked at full size.

    Rows {0, 1, Lq-2, Lq-1}, rows on either side of the 128-row tile edges
    {127, 128, 255, 256}, rows around the window edge, plus ``n_uniform``
    seeded uniform rows; for the heads given (default: every head when Hq <= 16,
    else 8 heads including both heads of one query group and the last head).
    """
    g = torch.Generator().manual_seed(1000 + seed)
    if heads is None:
        if w.Hq <= 16:
            heads = list(range(w.Hq))
        else:
            G = w.Hq // w.Hkv
            pick = {0, 1 % w.Hq, G, G + 1, w.Hq - 1}
            extra = torch.randperm(w.Hq, generator=g).tolist()
            for h in extra:
                if len(pick) >= 8:
                    break
                pick.add(h)
            heads = sorted(pick)
    fixed = {0, 1, w.Lq - 2, w.Lq - 1, 127, 128, 255, 256}
    if w.window:
        for c in (w.window - 1, w.window, w.window + 1):
            fixed.add(c)
    rows = [i for i in fixed if 0 <= i < w.Lq]
    rows += torch.randint(0, w.Lq, (n_uniform,), generator=g).tolist()
    rows = sorted(set(rows))
    ids = []
    for b in range(w.B):
        for h in heads:
            for i in rows:
                ids.append((b * w.Hq + h) * w.Lq + i)
    return ids
