"""Benchmark of the fused attention hot path on GB300.

One step = one sdpa_prefill call (C ABI) over the long-KV GQA prefill
workload: B=1, Hq=16, Hkv=8, head_dim 256, fp16, 1024 queries at positions
31744..32767 over 32768 keys, bottom-right causal.  Inputs are synthetic
(seeded N(0,1)), resident in HBM; L2 is flushed before every timed step.

Printed: one JSON line with the step metric (causal-adjusted TFLOP/s), the
roofline of the attention kernel, an end-to-end figure through host buffers,
the oracle on the host cores as a CPU baseline, SM clocks sampled during the
timed region and a per-workload suite (every prefill workload in TFLOP/s,
decode in GB/s, transient device memory against kL).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-suite]
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from attention_sm_flash_attn_gb300 import inputs as wl  # noqa: E402

METRIC = "prefill attention TFLOP/s (D=256/512) and % of GB300 bf16 tensor peak; decode GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- workload arithmetic

def visible_pairs(Lq, Lk, causal, window):
    """Visible (query, key) pairs per query head (bottom-right causal, window W)."""
    if not causal:
        return Lq * Lk
    p = np.arange(Lk - Lq, Lk, dtype=np.int64)
    n = p + 1
    if window:
        n = np.minimum(n, window)
    return int(n.sum())


def prefill_flops(w):
    return 4.0 * w.B * w.Hq * w.D * visible_pairs(w.Lq, w.Lk, w.causal, w.window)


def decode_bytes(w):
    """K+V bytes of the keys some row of each kv head sees, plus Q and O."""
    lo = max(0, w.Lk - w.Lq - w.window + 1) if (w.causal and w.window) else 0
    keys = w.Lk - lo
    esz = 2
    kv = 2 * w.B * w.Hkv * keys * w.D * esz
    qo = 2 * w.B * w.Hq * w.Lq * w.D * esz
    return kv + qo


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBs")
            bf = d.get("bf16_tflops")
            bfs = d.get("bf16_tflops_sustained", bf)
            if hbm and bf:
                return float(hbm), float(bf), float(bfs), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ---------------------------------------------------------------- ncu traffic

TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "attn_fwd_duoq_longkv_gqa_prefill_hd256.txt")


def strip_comments(src: str) -> str:
    """C/C++ source without // and /* */ comments, trailing blanks and empty
    lines (string and character literals are kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def kernel_sources_digest() -> str:
    """sha256 over the code (comments stripped) of the CUDA sources and the public
    header, in name order: a comment edit leaves the digest, and so the profiled
    traffic, in force; any code change retires it."""
    files = sorted(glob.glob(os.path.join(ROOT, "attention_sm_flash_attn_gb300", "csrc", "*.cu*"))
                   + glob.glob(os.path.join(ROOT, "include", "*.h")))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per launch of the timed kernel from the committed ncu summary,
    or None when that summary was taken on other kernel sources."""
    keys = ("kernel_sources_sha256", "dram_bytes_per_launch")
    try:
        fields = dict(line.split(":", 1) for line in open(TRAFFIC_SUMMARY)
                      if line.split(":", 1)[0] in keys)
    except OSError:
        return None
    digest = fields.get("kernel_sources_sha256", "").strip()
    if digest != kernel_sources_digest():
        return None
    try:
        return int(fields["dram_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="sdpa_clocks_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        with open(self.path) as fh:
            lines = fh.readlines()
        os.unlink(self.path)
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- timing helpers

class L2Flush:
    def __init__(self, device, nbytes=512 << 20):
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self):
        self.buf.fill_(1)


def time_calls(fn, steps, warmup, flush, stream):
    """Per-call device time (ms) with CUDA events on `stream`, L2 flushed before each call."""
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


L2_BYTES = 129 << 20


def steady_decode(gb, w, q, k, v, out, ws, cap_bytes=40 << 30):
    """Per-call device time (ms) of a decode loop's steady state: back-to-back
    calls captured in one CUDA graph over n rotating copies of K/V, no flush in
    between; the copies are chosen so that the bytes the n calls read add up
    to more than 3x L2 (every call reads keys no recent call has touched).
    Returns (ms, n)."""
    kvb = decode_bytes(w)
    per = (k.numel() + v.numel()) * k.element_size()
    n = max(2, min(64, (3 * L2_BYTES) // max(1, kvb) + 1))
    n = max(2, min(n, cap_bytes // max(1, per)))
    ks = [k] + [k.clone() for _ in range(n - 1)]
    vs = [v] + [v.clone() for _ in range(n - 1)]

    def call(i):
        gb.sdpa_decode(q, ks[i], vs[i], out, scale=w.scale, causal=w.causal, window=w.window,
                       workspace=ws)

    torch.cuda.synchronize()
    cs = torch.cuda.Stream()  # graphs are captured on a stream of their own
    with torch.cuda.stream(cs):
        for i in range(n):
            call(i)
        cs.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for i in range(n):
                call(i)
        g.replay()
        cs.synchronize()
        ts = []
        for _ in range(10):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(cs)
            g.replay()
            b.record(cs)
            cs.synchronize()
            ts.append(a.elapsed_time(b) / n)
    torch.cuda.synchronize()
    del g, ks, vs
    return statistics.median(ts), n


# ---------------------------------------------------------------- CPU baseline (oracle)

def cpu_baseline(w, q, k, v, budget_s=12.0, max_rows=None):
    """Time the fp64 oracle on sampled query rows of workload w; TFLOP/s of visible pairs."""
    import oracle
    oracle.build()
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    R = w.B * w.Hq * w.Lq
    rng = np.random.default_rng(0)
    order = rng.permutation(R)

    def row_flops(ids):
        i = np.asarray(ids) % w.Lq
        p = w.Lk - w.Lq + i
        n = (p + 1) if w.causal else np.full_like(p, w.Lk)
        if w.window:
            n = np.minimum(n, w.window)
        return float(4.0 * w.D * n.sum())

    n = 32
    t0 = time.perf_counter()
    oracle.sdpa(qc, kc, vc, scale=w.scale, causal=w.causal, window=w.window,
                rows=order[:n].tolist())
    dt = time.perf_counter() - t0
    n2 = int(min(R, max(n, n * budget_s / max(dt, 1e-3))))
    if max_rows:
        n2 = min(n2, max_rows)
    ids = order[:n2].tolist()
    t0 = time.perf_counter()
    oracle.sdpa(qc, kc, vc, scale=w.scale, causal=w.causal, window=w.window, rows=ids)
    dt = time.perf_counter() - t0
    return {"value": row_flops(ids) / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"{n2} of {R} query rows of {w.name} (uniform, seed 0), fp64, all visible keys"}


# ---------------------------------------------------------------- the suite

def suite(gb, device, flush, stream, hbm, bf16_peak):
    res = {}
    for w in [wl.LONGKV, wl.SELF16K, wl.SLIDING32K, wl.FULL512, wl.PREFILL128K,
              wl.LONGKV_HD192, wl.LONGKV_HD128]:
        q, k, v = wl.make_qkv(w, device=device)
        out = torch.empty_like(q)
        ws = torch.empty(max(1, gb.prefill_workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D,
                                                           w.causal, w.window)),
                         dtype=torch.uint8, device=device)
        fn = lambda: gb.sdpa_prefill(q, k, v, out, scale=w.scale, causal=w.causal,
                                     window=w.window, workspace=ws)
        steps = 5 if w is wl.FULL512 else 10
        ts = time_calls(fn, steps, 3, flush, stream)
        ms = statistics.median(ts)
        tf = prefill_flops(w) / ms / 1e9
        res[w.name] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                       "frac_of_bf16_peak": round(tf / bf16_peak, 4), "flop": prefill_flops(w)}
        del q, k, v, out, ws
        torch.cuda.empty_cache()
    for w0 in wl.DECODE_WORKLOADS:
        for Lq in wl.DECODE_LQ:
            w = w0.with_(Lq=Lq)
            q, k, v = wl.make_qkv(w, device=device)
            out = torch.empty_like(q)
            ws = torch.empty(gb.decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.D),
                             dtype=torch.uint8, device=device)
            fn = lambda: gb.sdpa_decode(q, k, v, out, scale=w.scale, causal=w.causal,
                                        window=w.window, workspace=ws)
            ts = time_calls(fn, 20, 5, flush, stream)
            ms = statistics.median(ts)
            gbs = decode_bytes(w) / ms / 1e6
            sms, ncopy = steady_decode(gb, w, q, k, v, out, ws)
            sgbs = decode_bytes(w) / sms / 1e6
            res[f"{w.name}_Lq{Lq}"] = {"us": round(ms * 1e3, 2), "GBps": round(gbs, 1),
                                       "frac_of_hbm": round(gbs / hbm, 4),
                                       "bytes": decode_bytes(w),
                                       "steady_us": round(sms * 1e3, 2),
                                       "steady_GBps": round(sgbs, 1),
                                       "steady_frac_of_hbm": round(sgbs / hbm, 4),
                                       "steady_copies": ncopy}
            del q, k, v, out, ws
            torch.cuda.empty_cache()
    # additive bias (mask array): one [Lq, Lk] mask shared by all heads in prefill,
    # one row per (head, query) in decode; entries N(0, 1) with a quarter -inf
    g = torch.Generator(device=device).manual_seed(5)
    for w, decode in ((wl.LONGKV, False), (wl.DECODE_WORKLOADS[0].with_(Lq=1), True)):
        q, k, v = wl.make_qkv(w, device=device)
        out = torch.empty_like(q)
        shape = (1, w.Hq, w.Lq, w.Lk) if decode else (1, 1, w.Lq, w.Lk)
        bias = torch.randn(shape, generator=g, device=device)
        bias = bias.masked_fill(torch.rand(shape, generator=g, device=device) < 0.25,
                                float("-inf")).to(q.dtype)
        if decode:
            ws = torch.empty(gb.decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.D),
                             dtype=torch.uint8, device=device)
            fn = lambda: gb.sdpa_decode(q, k, v, out, scale=w.scale, causal=w.causal,
                                        window=w.window, workspace=ws, bias=bias)
            ms = statistics.median(time_calls(fn, 20, 5, flush, stream))
            byts = decode_bytes(w) + w.B * w.Hq * w.Lq * min(w.Lk, w.window or w.Lk) * 2
            res[f"{w.name}_Lq1_bias"] = {"us": round(ms * 1e3, 2),
                                         "GBps": round(byts / ms / 1e6, 1), "bytes": byts}
        else:
            ws = torch.empty(max(1, gb.prefill_workspace_bytes(
                w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, w.causal, w.window)),
                dtype=torch.uint8, device=device)
            fn = lambda: gb.sdpa_prefill(q, k, v, out, scale=w.scale, causal=w.causal,
                                         window=w.window, workspace=ws, bias=bias)
            ms = statistics.median(time_calls(fn, 10, 3, flush, stream))
            tf = prefill_flops(w) / ms / 1e9
            res[f"{w.name}_bias"] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                                     "frac_of_bf16_peak": round(tf / bf16_peak, 4),
                                     "bias_bytes": bias.numel() * 2}
        del q, k, v, out, ws, bias
        torch.cuda.empty_cache()
    # transient device memory against kL at the long-KV GQA head geometry
    trans = {}
    for qL, kL in ((1024, 32768), (2048, 65536), (2048, 131072)):
        w = wl.LONGKV.with_(Lq=qL, Lk=kL)
        q, k, v = wl.make_qkv(w, device=device)
        out = torch.empty_like(q)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        gb.sdpa_prefill(q, k, v, out, scale=w.scale, causal=True)
        torch.cuda.synchronize()
        peak = torch.cuda.max_memory_allocated() - base
        free1 = torch.cuda.mem_get_info()[0]
        trans[f"qL{qL}_kL{kL}"] = {"transient_bytes": int(peak),
                                   "unaccounted_free_delta": int(free0 - free1),
                                   "inputs_MiB": (q.numel() + k.numel() + v.numel()) * 2 / 2**20}
        del q, k, v, out
        torch.cuda.empty_cache()
    res["transient_memory"] = trans
    return res


# ---------------------------------------------------------------- profiling runs

def profile_run(args):
    """Run one workload through the C ABI `--warmup + --steps` times, no timing."""
    import attention_sm_flash_attn_gb300 as gb
    from attention_sm_flash_attn_gb300 import build as gbbuild
    gbbuild.build()
    name, lq = args.profile, None
    with_bias = name.endswith("_bias")
    if with_bias:
        name = name[:-len("_bias")]
    if "_Lq" in name:
        name, lq = name.rsplit("_Lq", 1)
    table = {w.name: w for w in wl.PREFILL_WORKLOADS + wl.DECODE_WORKLOADS}
    w = table[name]
    if lq is not None:
        w = w.with_(Lq=int(lq))
    if args.profile_len:
        # a shorter case of the same kernel: Lk = N, and Lq = N when the
        # workload's queries span all of its keys
        n_len = args.profile_len
        w = w.with_(Lk=n_len, Lq=n_len if w.Lq == w.Lk else min(w.Lq, n_len))
    q, k, v = wl.make_qkv(w, device="cuda")
    out = torch.empty_like(q)
    bias = None
    if with_bias:
        # the suite's bias: one [Lq, Lk] mask for all heads in prefill, one row
        # per (head, query) in decode; N(0, 1) entries, a quarter of them -inf
        g = torch.Generator(device="cuda").manual_seed(5)
        shape = (1, w.Hq, w.Lq, w.Lk) if w.kind == "decode" else (1, 1, w.Lq, w.Lk)
        bias = torch.randn(shape, generator=g, device="cuda")
        bias = bias.masked_fill(torch.rand(shape, generator=g, device="cuda") < 0.25,
                                float("-inf")).to(q.dtype)
    if w.kind == "decode":
        ws = torch.empty(gb.decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.D),
                         dtype=torch.uint8, device="cuda")
        fn = lambda: gb.sdpa_decode(q, k, v, out, scale=w.scale, causal=w.causal,
                                    window=w.window, workspace=ws, bias=bias)
    else:
        nb = gb.prefill_workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, w.causal, w.window)
        ws = torch.empty(max(1, nb), dtype=torch.uint8, device="cuda")
        fn = lambda: gb.sdpa_prefill(q, k, v, out, scale=w.scale, causal=w.causal,
                                     window=w.window, workspace=ws, bias=bias)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    st = gb.device_status()
    print(json.dumps({"profile": w.name, "Lq": w.Lq, "Lk": w.Lk, "bias": with_bias,
                      "calls": args.warmup + args.steps,
                      "device_status": st[0]}))
    return 0 if st[0] == 0 else 1


# ---------------------------------------------------------------- routing study

def routing_study():
    """The pages route kL <= 16384 to an unfused path (matmul, softmax, matmul)
    because their fused kernel lost there ("Fused SDPA full-attention for
    head_dim=192/256", the routing discussion under "Microbenchmarks").  Here:
    the fused call against that unfused path built from torch (cuBLAS GEMMs, a
    dense mask and softmax), at the long-KV GQA head geometry, queries at the
    end of the keys, for kL from 512 to 16384.  Measurement only."""
    import attention_sm_flash_attn_gb300 as gb
    from attention_sm_flash_attn_gb300 import build as gbbuild
    gbbuild.build()
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = L2Flush(device)
    rows = []
    for kL in (512, 1024, 2048, 4096, 8192, 16384):
        w = wl.LONGKV.with_(Lq=min(1024, kL), Lk=kL)
        q, k, v = wl.make_qkv(w, device=device)
        out = torch.empty_like(q)
        nb = gb.prefill_workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, True, 0)
        ws = torch.empty(max(1, nb), dtype=torch.uint8, device=device)
        G = w.Hq // w.Hkv
        i = torch.arange(w.Lq, device=device).view(-1, 1) + (w.Lk - w.Lq)
        visible = torch.arange(w.Lk, device=device).view(1, -1) <= i

        def fused():
            gb.sdpa_prefill(q, k, v, out, scale=w.scale, causal=True, workspace=ws)

        def unfused():
            kk = k.repeat_interleave(G, dim=1)
            vv = v.repeat_interleave(G, dim=1)
            s = torch.matmul(q, kk.transpose(-1, -2)).float() * w.scale
            s.masked_fill_(~visible, float("-inf"))
            p = torch.softmax(s, dim=-1).to(q.dtype)
            return torch.matmul(p, vv)

        err = float((unfused().float() - (fused() or out).float()).abs().max())
        tf = statistics.median(time_calls(fused, 10, 3, flush, stream))
        tu = statistics.median(time_calls(unfused, 10, 3, flush, stream))
        rows.append({"kL": kL, "qL": w.Lq, "fused_ms": round(tf, 4), "unfused_ms": round(tu, 4),
                     "unfused_over_fused": round(tu / tf, 2),
                     "fused_tflops": round(prefill_flops(w) / tf / 1e9, 1),
                     "max_abs_diff": round(err, 5)})
        del q, k, v, out, ws, visible
        torch.cuda.empty_cache()
    print(json.dumps({"routing_study": "fused vs unfused prefill, Hq=16, Hkv=8, D=256, fp16, "
                                       "bottom-right causal", "rows": rows}), flush=True)
    return 0


# ---------------------------------------------------------------- ranks

def max_over_ranks(value: float, dist, device) -> float:
    """The largest `value` over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- main

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (torch.cuda.is_available() and args.impl != "reference") else "gloo"
        dist.init_process_group(backend)
        return world, rank, local, dist
    return 1, 0, 0, None


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = wl.LONGKV
    q, k, v = wl.make_qkv(w, device="cpu")
    vals = []
    cb = None
    for step in range(args.warmup + args.steps):
        cb = cpu_baseline(w, q, k, v,
                          budget_s=args.cpu_budget if step >= args.warmup else args.cpu_budget / 6)
        if step >= args.warmup:
            vals.append(cb["value"])
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": prefill_flops(w) / (value * 1e9), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "Lq": w.Lq, "Lk": w.Lk, "causal": "bottom-right"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cb["cores"],
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "note": "the fp64 CPU oracle on the host cores, per step a bounded row sample; "
                    "ms_per_step extrapolates its rate to the whole workload"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-suite", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=6.0,
                    help="seconds of oracle work per timed step of the reference arm")
    ap.add_argument("--profile", default=None,
                    help="run one named workload --steps times (for ncu) and exit; decode "
                         "workloads take a _LqN suffix, and a _bias suffix adds the suite's "
                         "additive bias")
    ap.add_argument("--profile-len", type=int, default=0,
                    help="with --profile: run the workload at Lk = N (and Lq = N when its "
                         "queries span all keys), for a smaller capture of the same kernel")
    ap.add_argument("--routing", action="store_true",
                    help="fused vs unfused (cuBLAS matmul + softmax + matmul) prefill time over "
                         "kL, one JSON line, and exit")
    args = ap.parse_args()
    if args.profile:
        return profile_run(args)
    if args.routing:
        return routing_study()
    args.warmup = max(3, args.warmup)
    world, rank, local, dist = dist_setup(args)
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
        if dist is not None:
            dist.destroy_process_group()
        return rc

    import attention_sm_flash_attn_gb300 as gb
    from attention_sm_flash_attn_gb300 import build as gbbuild
    gbbuild.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    hbm, bf16_peak, bf16_sust, peak_src = peaks()
    w = wl.LONGKV
    q, k, v = wl.make_qkv(w, device=device)
    out = torch.empty_like(q)
    ws_bytes = gb.prefill_workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, w.causal, w.window)
    ws = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device=device)
    launches_per_call = gb.prefill_launches(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, w.causal, w.window,
                                            ws.numel())
    fn = lambda: gb.sdpa_prefill(q, k, v, out, scale=w.scale, causal=w.causal, window=w.window,
                                 workspace=ws)
    flush = L2Flush(device)
    flops = prefill_flops(w)

    # --- timed region (device-resident inputs)
    for _ in range(args.warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    ts = time_calls(fn, args.steps, 0, flush, stream)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(ts), dist, device)
    status = gb.device_status()
    ms_per_step = total_ms / args.steps
    value = world * flops * args.steps / (total_ms * 1e9)  # TFLOP/s, all ranks
    per_launch_tf = flops / (statistics.mean(ts) * 1e9)

    # --- end to end through host buffers (pinned), copies inside the timed region
    hq, hk, hv = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        dq = hq.to(device, non_blocking=True)
        dk = hk.to(device, non_blocking=True)
        dv = hv.to(device, non_blocking=True)
        do = torch.empty_like(dq)
        gb.sdpa_prefill(dq, dk, dv, do, scale=w.scale, causal=w.causal, window=w.window,
                        workspace=ws)
        hout.copy_(do, non_blocking=True)

    e2e_ts = time_calls(e2e_step, max(3, args.steps // 2), 2, flush, stream)
    e2e_val = world * flops / (statistics.mean(e2e_ts) * 1e9)
    h2d = (q.numel() + k.numel() + v.numel()) * q.element_size()
    d2h = out.numel() * out.element_size()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "Lq": w.Lq, "Lk": w.Lk, "causal": "bottom-right",
                   "query_positions": f"{w.Lk - w.Lq}..{w.Lk - 1}",
                   "l2": "flushed (512 MiB write) before every timed step",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(per_launch_tf, 2),
                     "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(per_launch_tf / bf16_peak, 4),
                     "traffic": profiled_traffic() if launches_per_call == 1 else None,
                     "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum of one "
                                       "ncu capture of this kernel build (profiles/), per launch",
                     "peak_source": f"{peak_src} bf16 dense burst (fp16 rate taken equal)",
                     "timed": "whole sdpa_prefill call on its stream (attention kernel"
                              + (" + combine kernel)" if launches_per_call == 2 else ")")},
        "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_call * args.steps,
        "clocks": clk,
        "device_status": status[0],
    }
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, q, k, v)
    if rank == 0 and not args.no_suite:
        del hq, hk, hv, hout
        line["suite"] = suite(gb, device, flush, stream, hbm, bf16_peak)
        line["suite_timing"] = ("ms / us: median CUDA-event time of one call, L2 flushed "
                                "(512 MiB write) before each; decode steady_us: per-call time "
                                "of back-to-back calls in one CUDA graph over rotating K/V "
                                "copies (more than 3x L2 read per pass), no flush")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
