#!/usr/bin/env python3
"""Benchmark: split-KV paged GQA decode attention on GB300.

One step = one pass of the decode attention hot path over one batch of the
Flint-shaped workload: B=64 requests, Hq=64, Hkv=8, head_dim 128, bf16 HND
pages of 16 tokens, log-uniform lengths in [1, 32768], per-head sinks, and the
workload's two layer types -- a full-attention layer and a sliding-window
(128) layer, each with its own KV cache -- so two library calls per step.

Prints one JSON line (rank 0).  `value` is KV-cache GB/s over the step
(algorithmic bytes: attended tokens x Hkv x 512 B) with inputs resident in HBM
and no L2 flush (each step streams 797 MB of KV, over six times the 129 MB L2),
from K steps run back to back with events only around the loop; `e2e` repeats the measurement through the same C ABI call with the step's
inputs copied from pinned host memory and the outputs copied back inside the
timed region.  `roofline` covers the dominant
kernel (the full-attention layer) against the measured HBM copy bandwidth; its
launch time comes from a second pass of K steps with an event pair around
every launch.
`cpu_baseline` is the fp64 CPU oracle timed on this host on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV-cache read GB/s (% of GB300 HBM peak) and attention calls/sec at 1 GPU"
UNIT = "GB/s"
WORKLOAD = ("flint_gqa_b64: B=64, Hq=64, Hkv=8, head_dim=128, bf16 HND pages of 16 tokens, "
            "seq_lens log-uniform in [1,32768], random block tables, fp32 sinks; one "
            "full-attention layer + one sliding-window-128 layer per step")
FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2
KERNEL_SOURCES = ["paged_kv_cache_30_gb300/csrc/gqa_decode.cu",
                  "paged_kv_cache_30_gb300/csrc/ptx.cuh"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_bf16_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def profiled_traffic():
    """DRAM bytes per launch of the full-layer kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "gqa_decode_flint_b64_full.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_hash") == kernel_hash():
            return d.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


# ------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        if not inside and rows:
            inside = [min(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        mx = [num(p[3]) for _, p in inside if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in inside for i in range(4)
                          if p[6 + i].lower().startswith("active")})
        pw = [num(p[4]) for _, p in inside if num(p[4]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------ workload ----
def make_layers(seed: int):
    """The step's batch: one set of requests (lengths, block tables) and two
    layers, each with its own KV cache, queries and sinks."""
    from paged_kv_cache_30_gb300 import workloads as W
    full = W.flint_gqa(seed, window=0)
    slide = W.GQAProblem(
        q=W.normal(full.q.shape, seed * 7919 + 101),
        kv_cache=W.normal(full.kv_cache.shape, seed * 7919 + 102),
        block_table=full.block_table, seq_lens=full.seq_lens,
        sinks=W.normal(full.sinks.shape, seed * 7919 + 103, dtype=full.sinks.dtype),
        window=128, scale=full.scale, page_size=16, name="flint_gqa_b64_w128")
    return [full, slide]


def oracle_baseline(layers, budget_s: float, threads: int):
    """Time the fp64 oracle on a bounded sample: whole (request, kv head)
    groups of the full layer, longest requests first, round-robin over the
    layer (again from the start once every group is done), until ~budget_s of
    work."""
    import numpy as np
    import oracle
    full = layers[0]
    B, Hq, _ = full.q.shape
    Hkv = full.kv_cache.shape[1]
    L = full.seq_lens.numpy().astype(np.int64)
    order = np.argsort(-L)  # longest first: representative bytes per second
    done_bytes, t_used, groups = 0, 0.0, 0
    i = 0
    while t_used < budget_s:
        b = int(order[(i // Hkv) % B])
        kvh = i % Hkv
        rows = np.arange(b * Hq + kvh * 8, b * Hq + kvh * 8 + 8, dtype=np.int64)
        t = time.perf_counter()
        oracle.gqa_decode(full.q, full.kv_cache, full.block_table, full.seq_lens, full.sinks, 0,
                          full.scale, 16, rows=rows, nthreads=threads)
        t_used += time.perf_counter() - t
        done_bytes += int(L[b]) * 512
        groups += 1
        i += 1
    return done_bytes / t_used / 1e9, t_used, groups


def oracle_single_thread(budget_s: float):
    """The oracle on one host thread on the tiny GQA batch (whole calls) and on
    the B = 32 qlen 4 MLA verify batch (whole (row, head) pairs of the longest
    request, until ~budget_s of work): a reported baseline beside the all-core
    figure."""
    import numpy as np
    import oracle
    from paged_kv_cache_30_gb300 import workloads as W
    tiny = W.tiny_gqa(0)
    n, t_used = 0, 0.0
    while t_used < budget_s or n < 3:
        t = time.perf_counter()
        oracle.gqa_decode(tiny.q, tiny.kv_cache, tiny.block_table, tiny.seq_lens, tiny.sinks,
                          tiny.window, tiny.scale, tiny.page_size, nthreads=1)
        t_used += time.perf_counter() - t
        n += 1
    res = {"tiny_gqa_b4": {"calls_per_s": n / t_used, "calls": n, "cores": 1}}
    mla = W.mla_verify(0)
    R, H, _ = mla.q.shape
    b = int(np.argmax(mla.seq_lens.numpy()))
    L = int(mla.seq_lens[b])
    Lr = int(mla.real_seq_lens[b]) if mla.real_seq_lens is not None else L
    flops, t_used, done = 0.0, 0.0, 0
    pairs = np.arange(b * mla.qlen * H, (b + 1) * mla.qlen * H, dtype=np.int64)
    while t_used < budget_s and done < len(pairs):
        rows = pairs[done:done + 16]
        t = time.perf_counter()
        oracle.mla_verify(mla.q, mla.latent_cache, mla.block_table, mla.seq_lens,
                          mla.real_seq_lens, mla.qlen, mla.scale, mla.page_size, rows=rows,
                          nthreads=1)
        t_used += time.perf_counter() - t
        for x in rows:
            tok = int(x) // H - b * mla.qlen
            flops += 2.0 * max(min(L - mla.qlen + 1 + tok, Lr), 0) * (576 + 512)
        done += len(rows)
    res["mla_verify_b32_q4"] = {"GFLOP_per_s": flops / t_used / 1e9, "row_heads": done,
                                "cores": 1}
    return res


# ---------------------------------------------------- the other workloads ---
def mla_flops(prob) -> float:
    """Algorithmic MLA flops: every (row, head) attends lim keys with a 576-wide
    Q.K and a 512-wide P.V (2 flops per multiply-add).  The row limit is the
    verify page's max(min(L - qlen + 1 + t, L_real), 0), restated here for the
    count."""
    import numpy as np
    L = prob.seq_lens.numpy().astype(np.int64)
    Lr = L if prob.real_seq_lens is None else prob.real_seq_lens.numpy().astype(np.int64)
    tot = 0
    for t in range(prob.qlen):
        lim = np.maximum(np.minimum(L - prob.qlen + 1 + t, Lr), 0)
        tot += int(lim.sum())
    return float(tot) * 128 * 2 * (576 + 512)


class L2Flush:
    """Evicts L2 between timed calls, outside the timed events: a 512 MiB write
    (the eviction), then a read of another 512 MiB buffer so that the lines L2
    holds afterwards are clean.  After the write alone the next kernel pays the
    write-back of the flush's ~129 MB of dirty lines: the Flint full layer took
    146.9 us after a write-only flush, 133.5 us after this one and 134.1 us
    with no flush at all (its 777 MB exceed L2), and a per-CTA trace showed it
    reading at 5.3 TB/s for its first 40 us after the write-only flush against
    7.0 TB/s after this one."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, s: int = 0):
        import torch
        self.w.fill_(float(s & 7))
        torch.amax(self.r, dim=0, out=self.sink)


def time_events(fn, flush, steps, warmup=3):
    import torch
    for _ in range(warmup):
        fn()
        flush(1)
    ev = []
    for s in range(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        flush(s)
        ev.append((a, b))
    torch.cuda.synchronize()
    ms = sorted(x.elapsed_time(y) for x, y in ev)
    return statistics.median(ms), statistics.mean(ms)


def _tiny(dev, flush, steps, tiny, gqa_entry):
    import torch
    import paged_kv_cache_30_gb300 as pkv
    d, (prob, out, lse) = gqa_entry(tiny, [4])
    t = dict(q=tiny.q.to(dev), kv=tiny.kv_cache.to(dev), bt=tiny.block_table.to(dev),
             sl=tiny.seq_lens.to(dev))
    s = torch.cuda.Stream()
    call = lambda: pkv.paged_decode_attn(t["q"], t["kv"], t["bt"], t["sl"], None, 0, tiny.scale,
                                         16, 4, out, lse, stream=s)
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(100):
            call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):  # replay and both events on one stream
        g.replay()
        a.record(s)
        for _ in range(10):
            g.replay()
        b.record(s)
    torch.cuda.synchronize()
    d["graph_replay_calls_per_s"] = 1000 / (a.elapsed_time(b) * 1e-3)  # 10 x 100 calls
    d["eager_calls_per_s"] = 1e6 / d["cap_4"]["us"]
    return d


def other_workloads(dev, flush, peak_hbm, peak_tf, steps, only=None, sampler=None):
    """Every other workload of the pages' problem, timed the same way (inputs
    resident, L2 flushed between calls by L2Flush, CUDA events): the tiny decode batch,
    the 131072-token long context at B=1 and B=8 across split caps, the two
    MLA verify workloads (bf16 and FP8 latent caches) and the paged KV append
    that precedes a decode or verify call.  With a running ClockSampler, each
    entry gets the clock record of its own timed calls."""
    import torch
    import paged_kv_cache_30_gb300 as pkv
    from paged_kv_cache_30_gb300 import workloads as W
    res = {}
    t_mark = [time.time()]

    def stamp(*names):
        """Attach the clocks sampled since the last stamp to these entries."""
        t_end = time.time()
        if sampler is not None:
            c = sampler.summary(t_mark[0], t_end)
            for n in names:
                if isinstance(res.get(n), dict):
                    res[n]["clocks"] = c
        t_mark[0] = t_end

    def start():
        torch.cuda.synchronize()
        t_mark[0] = time.time()

    def gqa_entry(prob, caps):
        t = dict(q=prob.q.to(dev), kv=prob.kv_cache.to(dev), bt=prob.block_table.to(dev),
                 sl=prob.seq_lens.to(dev),
                 sk=None if prob.sinks is None else prob.sinks.to(dev))
        out = torch.empty_like(t["q"])
        lse = torch.empty(t["q"].shape[:2], device=dev)
        nbytes = prob.kv_bytes()
        out_d = {"kv_bytes": nbytes}
        for cap in caps:
            fn = lambda: pkv.paged_decode_attn(t["q"], t["kv"], t["bt"], t["sl"], t["sk"],
                                               prob.window, prob.scale, prob.page_size, cap, out,
                                               lse)
            med, _ = time_events(fn, flush, steps)
            out_d[f"cap_{cap}"] = {"us": 1e3 * med, "GBps": nbytes / (med * 1e-3) / 1e9,
                                   "hbm_frac_of_measured": nbytes / (med * 1e-3) / 1e9 / peak_hbm}
        del t
        return out_d, (prob, out, lse)

    want = (lambda k: only is None or k in only)
    # tiny decode batch: latency-bound, report calls/s eager and as CUDA-graph replay
    if want("tiny"):
        tiny = W.tiny_gqa(0)
        start()
        res["tiny_gqa_b4"] = _tiny(dev, flush, steps, tiny, gqa_entry)
        stamp("tiny_gqa_b4")
    for B in (1, 8):
        if not want(f"long{B}"):
            continue
        prob = W.long_context(0, B=B)
        start()
        res[f"long_ctx_b{B}"], _ = gqa_entry(prob, [0, 1, 8, 32, 132])
        stamp(f"long_ctx_b{B}")
        del prob

    for key, name, mk in (("mla", "mla_verify_b32_q4", W.mla_verify),
                          ("mla_fp8", "mla_fp8_b128", W.mla_fp8)):
        if not want(key):
            continue
        prob = mk(0)
        tq = prob.q.to(dev)
        tc = prob.latent_cache.to(dev)
        tbt, tsl = prob.block_table.to(dev), prob.seq_lens.to(dev)
        trl = None if prob.real_seq_lens is None else prob.real_seq_lens.to(dev)
        ks = None if prob.k_scale is None else torch.tensor(prob.k_scale, device=dev)
        out = torch.empty((tq.shape[0], 128, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((tq.shape[0], 128), device=dev)
        fn = lambda: pkv.mla_verify_attn(tq, tc, tbt, tsl, trl, prob.qlen, prob.scale,
                                         prob.page_size, ks, out, lse, prob.num_kv_splits)
        start()
        med, _ = time_events(fn, flush, steps)
        fl = mla_flops(prob)
        nbytes = prob.kv_bytes()
        res[name] = {"us": 1e3 * med, "TFLOPs": fl / (med * 1e-3) / 1e12,
                     "tensor_frac_of_measured_bf16": fl / (med * 1e-3) / 1e12 / peak_tf,
                     "GBps": nbytes / (med * 1e-3) / 1e9, "flops": fl, "kv_bytes": nbytes,
                     "cap": prob.num_kv_splits}
        stamp(name)
        if key == "mla_fp8" and want("native"):
            # the same workload on the native-FP8 path: query quantised to e4m3
            # per (row, head) inside the timed call, S on kind::f8f6f4 MMAs
            q8 = torch.empty(tq.shape, dtype=torch.float8_e4m3fn, device=dev)
            qs = torch.empty(tq.shape[:2], dtype=torch.float32, device=dev)

            def fn_native():
                pkv.mla_quantize_q(tq, q8, qs)
                pkv.mla_verify_attn_fp8_native(q8, qs, tc, tbt, tsl, trl, prob.qlen, prob.scale,
                                               prob.page_size, ks, out, lse, prob.num_kv_splits)
            start()
            med_n, _ = time_events(fn_native, flush, steps)
            res["mla_fp8_native_b128"] = {
                "us": 1e3 * med_n, "TFLOPs": fl / (med_n * 1e-3) / 1e12,
                "tensor_frac_of_measured_bf16": fl / (med_n * 1e-3) / 1e12 / peak_tf,
                "GBps": nbytes / (med_n * 1e-3) / 1e9, "flops": fl, "kv_bytes": nbytes,
                "cap": prob.num_kv_splits,
                "note": "query quantised to e4m3 (an opt-in numerics change); the quantisation "
                        "kernel is inside the timed call"}
            stamp("mla_fp8_native_b128")
            del q8, qs
        del tq, tc
    if want("append"):
        # the cache write before each call: the Flint batch's current tokens
        # (64 x 8 kv heads x 512 B) and the MLA verify rows (32 x 4 x 1152 B)
        prob = W.flint_gqa(0, 0)
        B, Hq = prob.q.shape[:2]
        k = W.normal((B, Hq // 8, 128), 91).to(dev)
        v = W.normal((B, Hq // 8, 128), 92).to(dev)
        kv, bt, sl = prob.kv_cache.to(dev), prob.block_table.to(dev), prob.seq_lens.to(dev)
        fn = lambda: pkv.gqa_kv_append(k, v, kv, bt, sl, prob.page_size)
        start()
        med, _ = time_events(fn, flush, steps)
        nbytes = 2 * int((prob.seq_lens > 0).sum()) * (Hq // 8) * 512  # read + written
        res["kv_append_flint_b64"] = {"us": 1e3 * med, "GBps": nbytes / (med * 1e-3) / 1e9,
                                      "rows": int((prob.seq_lens > 0).sum()) * (Hq // 8)}
        del kv
        mp = W.mla_verify(0)
        lat = W.normal((mp.q.shape[0], 576), 93).to(dev)
        cache, mbt, msl = mp.latent_cache.to(dev), mp.block_table.to(dev), mp.seq_lens.to(dev)
        stamp("kv_append_flint_b64")
        fn = lambda: pkv.mla_kv_append(lat, cache, mbt, msl, mp.qlen, mp.page_size)
        start()
        med, _ = time_events(fn, flush, steps)
        nbytes = 2 * mp.q.shape[0] * 1152
        res["kv_append_mla_b32_q4"] = {"us": 1e3 * med, "GBps": nbytes / (med * 1e-3) / 1e9,
                                       "rows": int(mp.q.shape[0])}
        stamp("kv_append_mla_b32_q4")
        del cache
    assert pkv.check_errors(dev.index or 0) == 0
    return res


# ------------------------------------------------------------- reference ---
def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: same workload, metric and
    unit; each step a bounded sample (whole kv-head groups of the full layer)."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    oracle.build()
    layers = make_layers(args.seed)
    full = layers[0]
    B, Hq, _ = full.q.shape
    Hkv = full.kv_cache.shape[1]
    L = full.seq_lens.numpy().astype(np.int64)
    threads = os.cpu_count() or 1
    total_steps = args.steps + args.warmup
    per_step = min(4.0, 150.0 / max(1, total_steps))
    rng = np.random.default_rng(args.seed)
    cand = [(b, k) for b in range(B) for k in range(Hkv)]

    def one_step():
        t0 = time.perf_counter()
        nbytes = 0
        while True:
            b, kvh = cand[int(rng.integers(len(cand)))]
            rows = np.arange(b * Hq + kvh * 8, b * Hq + kvh * 8 + 8, dtype=np.int64)
            oracle.gqa_decode(full.q, full.kv_cache, full.block_table, full.seq_lens,
                              full.sinks, 0, full.scale, 16, rows=rows, nthreads=threads)
            nbytes += int(L[b]) * 512
            if time.perf_counter() - t0 >= per_step:
                return nbytes, time.perf_counter() - t0

    for _ in range(args.warmup):
        one_step()
    tot_b, tot_t = 0, 0.0
    for _ in range(args.steps):
        nb, dt = one_step()
        tot_b += nb
        tot_t += dt
    value = tot_b / tot_t / 1e9
    sample = (f"random (request, kv head) groups of the full-attention layer, all 8 query "
              f"heads each, ~{per_step:.2f} s of oracle work per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 64, "seed": args.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- main arm --
# ------------------------------------------------- ranks (weak scaling) ---
def rank_seed(seed: int, rank: int) -> int:
    """Each rank runs its own batch: same shapes and length law, its own draw."""
    return seed + 7919 * rank


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's value (all ranks receive it); x itself on one rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, step_bytes: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch
    import paged_kv_cache_30_gb300 as pkv
    from paged_kv_cache_30_gb300 import build as pkv_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pkv_build.build()
    pkv.load_library()
    pkv.init(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    if args.only:
        # profiling aid: time only the named other workloads
        flush = L2Flush(dev)
        peak, _ = measured_peaks()
        res = other_workloads(dev, flush, peak, measured_bf16_tflops(), args.extra_steps,
                              only=set(args.only.split(",")))
        if rank == 0:
            print(json.dumps({"other_workloads": res}), flush=True)
        return

    # weak scaling: every rank runs its own batch of 64 requests
    layers = make_layers(rank_seed(args.seed, rank))
    kv_bytes = [p.kv_bytes() for p in layers]
    step_bytes = sum(kv_bytes)
    stream = torch.cuda.current_stream(dev)
    d = []
    bt_dev = layers[0].block_table.to(dev)
    sl_dev = layers[0].seq_lens.to(dev)
    for p in layers:
        d.append(dict(q=p.q.to(dev), kv=p.kv_cache.to(dev), bt=bt_dev, sl=sl_dev,
                      sinks=p.sinks.to(dev), out=torch.empty_like(p.q, device=dev),
                      lse=torch.empty(p.q.shape[:2], device=dev)))
    flush = L2Flush(dev)  # for the other workloads; the step loop needs none

    def call(i):
        p, t = layers[i], d[i]
        pkv.paged_decode_attn(t["q"], t["kv"], t["bt"], t["sl"], t["sinks"], p.window, p.scale,
                              16, 0, t["out"], t["lse"])

    def barrier():
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    # ---------------- device-resident timing ----------------
    for _ in range(args.warmup):
        call(0); call(1)
    assert pkv.check_errors(local_rank) == 0
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    # The steps as a user runs them: the two layers back to back with no
    # stream operation between them, so the window layer's launch overlaps the
    # full layer's tail (programmatic dependent launch).  Only this loop's time
    # gives `value`.
    e_a = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    barrier()
    t0 = time.time()
    e_a[0].record(stream)
    for s in range(args.steps):
        call(0)
        call(1)
        # no flush: the full layer's 777 MB of KV evict the window layer's 20 MB
        # between its calls, and each step streams over six times the L2
    e_a[1].record(stream)
    barrier()
    t1 = time.time()
    total_ms = max_over_ranks(e_a[0].elapsed_time(e_a[1]), dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_value(world, step_bytes, ms_per_step)
    calls_per_s = world * 2 / (ms_per_step * 1e-3)
    assert pkv.check_errors(local_rank) == 0

    # The same steps again with an event around every launch, to time the
    # full-layer kernel alone for the roofline.  The event between the layers
    # stops the overlap, so these steps are slower than the loop above.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier()
    for s in range(args.steps):
        e = ev[s]
        e[0].record(stream)
        call(0)
        e[1].record(stream)
        call(1)
        e[2].record(stream)
    barrier()
    t2 = time.time()
    full_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    step_ms_evented = statistics.mean(ev[s][0].elapsed_time(ev[s][2]) for s in range(args.steps))
    full_mean = statistics.mean(full_ms)
    achieved = kv_bytes[0] / (full_mean * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    assert pkv.check_errors(local_rank) == 0

    # ---------------- end to end through the same call, host buffers ----------------
    # Every step copies its inputs (q of both layers, block table, seq_lens)
    # from pinned host memory and reads its results (out, lse of both layers)
    # back; the copies run on two copy streams, double-buffered, so step s+1's
    # upload and step s's download overlap step s's kernels.  No flush inside
    # this loop: each step streams 777 MB of KV, more than the 129 MB L2.
    # one pinned upload buffer per step: [q of layer 0 | q of layer 1 | block table |
    # seq_lens]; one download buffer: [out 0 | out 1 | lse 0 | lse 1]
    def carve(buf, specs):
        views, off = [], 0
        for shape, dtype in specs:
            nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
            views.append(buf[off:off + nbytes].view(dtype).view(shape))
            off += (nbytes + 255) // 256 * 256
        return views
    in_specs = [(tuple(p.q.shape), torch.bfloat16) for p in layers] + [
        (tuple(layers[0].block_table.shape), torch.int32), (tuple(layers[0].seq_lens.shape), torch.int32)]
    out_specs = [(tuple(p.q.shape), torch.bfloat16) for p in layers] + [
        (tuple(p.q.shape[:2]), torch.float32) for p in layers]
    def size_of(specs):
        return sum((int(np.prod(sh)) * torch.tensor([], dtype=dt).element_size() + 255) // 256 * 256
                   for sh, dt in specs)
    h_in = torch.empty(size_of(in_specs), dtype=torch.uint8).pin_memory()
    hv = carve(h_in, in_specs)
    for i in range(2):
        hv[i].copy_(layers[i].q)
    hv[2].copy_(layers[0].block_table)
    hv[3].copy_(layers[0].seq_lens)
    d_in = [torch.empty_like(h_in, device=dev) for _ in range(2)]
    dv = [carve(x, in_specs) for x in d_in]
    h_out = [torch.empty(size_of(out_specs), dtype=torch.uint8).pin_memory() for _ in range(2)]
    hov = [carve(x, out_specs) for x in h_out]
    d_out = [torch.empty_like(h_out[0], device=dev) for _ in range(2)]
    dov = [carve(x, out_specs) for x in d_out]
    h2d = sum(int(np.prod(sh)) * torch.tensor([], dtype=dt).element_size() for sh, dt in in_specs)
    d2h = sum(int(np.prod(sh)) * torch.tensor([], dtype=dt).element_size() for sh, dt in out_specs)
    # uploads and read-backs on separate copy streams: on one stream the upload
    # of step s+1 would queue behind the read-back of step s, which waits for
    # step s's kernels, and no copy would overlap a kernel
    upload, download = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    up = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer b uploaded
    done = [torch.cuda.Event() for _ in range(2)]    # kernels of buffer b finished
    down = [torch.cuda.Event() for _ in range(2)]    # outputs of buffer b read back

    def e2e_step(s):
        b = s & 1
        with torch.cuda.stream(upload):
            if s >= 2:
                upload.wait_event(done[b])           # step s-2 no longer reads buffer b
            d_in[b].copy_(h_in, non_blocking=True)
            up[b].record(upload)
        stream.wait_event(up[b])
        if s >= 2:
            stream.wait_event(down[b])               # step s-2's results are read back
        for i in range(2):
            p = layers[i]
            pkv.paged_decode_attn(dv[b][i], d[i]["kv"], dv[b][2], dv[b][3], d[i]["sinks"],
                                  p.window, p.scale, 16, 0, dov[b][i], dov[b][2 + i],
                                  stream=stream)
        done[b].record(stream)
        with torch.cuda.stream(download):
            download.wait_event(done[b])
            h_out[b].copy_(d_out[b], non_blocking=True)
            down[b].record(download)

    for s in range(3):  # warm the copy path
        e2e_step(s)
    torch.cuda.synchronize()
    barrier()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for s in range(args.steps):
        e2e_step(s)
    stream.wait_stream(download)                     # the last read-back is inside the region
    e_end.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), dist, dev)
    e2e_value = job_value(world, step_bytes, e2e_ms / args.steps)
    # the last step's results reached the host intact: the kernels are
    # deterministic, so they equal the device-resident loop's (same inputs)
    last = (args.steps - 1) & 1
    for i in range(2):
        assert torch.equal(hov[last][i].view(torch.int16), d[i]["out"].cpu().view(torch.int16))
    assert pkv.check_errors(local_rank) == 0

    if dist:
        dist.barrier()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    # ---------------- CPU baseline: the oracle on this host ----------------
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = os.cpu_count() or 1
        v, t_used, groups = oracle_baseline(layers, args.cpu_budget, threads)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{groups} (request, kv head) groups of the full-attention layer "
                         f"(longest requests first, all 8 query heads each, "
                         f"{groups / (layers[0].q.shape[0] * layers[0].kv_cache.shape[1]):.1f} "
                         f"passes over the layer), {t_used:.1f} s of fp64 oracle work on "
                         f"{threads} threads"}
        cpu["single_thread"] = oracle_single_thread(2.0)

    extra = None
    try:
        if world == 1 and not args.no_extra:
            extra = other_workloads(dev, flush, peak, measured_bf16_tflops(), args.extra_steps,
                                    sampler=sampler)
        time.sleep(0.2)
    finally:
        sampler.stop()
    clocks = sampler.summary(t0, t2)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 64 * world, "seed": args.seed,
                   "kv_bytes_per_step": step_bytes, "kv_bytes_full_layer": kv_bytes[0],
                   "l2": "inputs larger than L2: no flush between steps (797 MB of KV per "
                         "step, L2 129 MB); e2e loop the same, copies double-buffered on "
                         "two copy streams; other_workloads: L2 flushed between calls (512 MiB "
                         "write, then a 512 MiB read so L2 is left clean)",
                   "parallelism": f"{world} independent ranks" if world > 1 else "single GPU"},
        "calls_per_s": calls_per_s,
        "hbm_frac_of_measured": value / peak,
        "hbm_frac_of_nominal_8tbs": value / 8000.0,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "kernel": "gqa_decode_kernel<16, 0> (persistent mode, full-attention layer)",
                     "peak_source": f"{peak_kind} hbm_gbs", "launch_ms": full_mean,
                     "timing": "mean of one event pair around each full-layer launch over "
                               "K steps timed after the value loop (those steps: "
                               f"{step_ms_evented:.4f} ms each)"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "like the value loop, no event between the two layers: the window "
                        "layer's launch overlaps the full layer's tail (programmatic "
                        "dependent launch)"},
        "gpu_launches": 2 * args.steps,
        "other_workloads": extra,
        "clocks": clocks,
        "kernel_hash": kernel_hash(),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads (tiny, long context, MLA)")
    ap.add_argument("--extra-steps", type=int, default=30)
    ap.add_argument("--only", default="",
                    help="comma list of tiny,long1,long8,mla,mla_fp8,native (with mla_fp8),append: time only "
                         "these (no headline)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world > 1:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
