#!/usr/bin/env python3
"""Benchmark of absorbed MLA decode over a paged latent cache on GB300.

A step is one pass of the hot path over one batch: mla_cache_append of the tokens each request
adds (quantised into the cache) followed by mla_decode of the whole batch (page gather, FP8
dequantisation, scores, online softmax, weighted latent sum, split-KV merge).  The headline
workload is the largest one that fits one GPU: the FP8 mixed cache, B=64 requests of 32,768
positions each (32,704 prefilled + 64 appended per step), H=128, 64-token pages shuffled,
scale 1/sqrt(192).  The same run measures the other four workloads (tiny dense, batched paged,
long context, top-k sparse) and reports them under "configs".

Timing: W warm-up steps, then exactly K steps bracketed by a barrier and a device synchronise,
timed with CUDA events on the launching stream, max over ranks.  Each step is a CUDA graph of
the two library calls (the calls take about as long as the kernels, so eager launches would
time the host).  The inputs rotate over identical pool replicas whose touched bytes exceed L2
three times, so every step reads its cache from HBM; the tiny workload is also timed with L2
flushed before every call.  The decode call alone is timed over at least a second of
back-to-back calls for the roofline figures.

One JSON line on stdout (rank 0).  ``--impl reference`` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode KV GB/s, TFLOP/s and % of GB300 roofline; decode tokens/s at B×ctx"
UNIT = "KV GB/s"
L2_BYTES = 126 * 2 ** 20

# DRAM bytes (read + write) per launch of each workload's dominant kernel from an ncu capture,
# keyed by the sha256 of the code (comments excluded) of the sources that kernel is built from and
# the workload; any change to that code makes the entry stale (traffic = null).
_HEADERS = ["mla_latent_kv_decode_gb300/csrc/decode_common.cuh",
            "mla_latent_kv_decode_gb300/csrc/mla_internal.cuh",
            "mla_latent_kv_decode_gb300/csrc/tc_ptx.cuh",
            "include/mla.h"]
KERNEL_SOURCES = {
    "decode_tc": ["mla_latent_kv_decode_gb300/csrc/decode_tc.cu"] + _HEADERS,
    "decode_gather": ["mla_latent_kv_decode_gb300/csrc/decode_gather.cu",
                      "mla_latent_kv_decode_gb300/csrc/decode_gather.cuh"] + _HEADERS,
    "indexer_score": ["mla_latent_kv_decode_gb300/csrc/indexer.cu"] + _HEADERS,
    "proj": ["mla_latent_kv_decode_gb300/csrc/proj.cu"] + _HEADERS,
}
WORKLOAD_KERNEL = {"tiny_dense": "decode_tc", "paged_batch": "decode_tc", "long_context": "decode_tc",
                   "fp8_batch": "decode_gather", "topk_sparse": "decode_gather",
                   "v4_batch": "decode_gather", "v41_batch": "decode_gather",
                   "indexer_topk": "indexer_score", "value_project": "proj", "value_project_merged": "proj"}
NCU_TRAFFIC = {
    ("a6a81cb6175a2d16", "tiny_dense"): 4_939_008,
    ("a6a81cb6175a2d16", "paged_batch"): 176_497_152,
    ("a6a81cb6175a2d16", "long_context"): 154_273_024,
    ("4c1171a7fa215234", "fp8_batch"): 1_412_164_096,
    ("4c1171a7fa215234", "topk_sparse"): 120_542_080,
    ("4c1171a7fa215234", "v4_batch"): 1_263_980_032,
    ("4c1171a7fa215234", "v41_batch"): 641_302_016,
    ("509e33095508b7b4", "indexer_topk"): 1_142_835_200,
    ("46f7feafc1c08056", "value_project"): 224_005_632,
    ("46f7feafc1c08056", "value_project_merged"): 682_509_184,
}


def _code_only(text: str) -> str:
    """The source without its comments and blank lines (a comment edit leaves the kernel as it
    was; any change to code or constants does not)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def _sources_hash(workload: str) -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[WORKLOAD_KERNEL[workload]]:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic(workload: str):
    return NCU_TRAFFIC.get((_sources_hash(workload), workload))


def max_over_ranks(ms: float, dist, device: str = "cuda") -> float:
    """The slowest rank's time (every rank gets it), so that a job's value is the units all ranks
    processed divided by the time the whole job took.  dist is torch.distributed or None."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: each of `world` ranks processes `units_per_rank` in `seconds` (the
    max over ranks); replicas only, so per-rank work is fixed as ranks are added (weak scaling)."""
    return world * units_per_rank / seconds


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------------
# Reference arm / CPU baseline: the fp64 oracle on the host cores
# ----------------------------------------------------------------------------------------------

_POOLS = {}


def _request_pool(w, b: int):
    """Request b's rows in a one-request oracle pool (built once per run: drawing and encoding the
    rows is set-up, not the oracle's decode)."""
    import oracle
    from mla_latent_kv_decode_gb300 import synth
    key = (w.name, w.seed, b)
    if key not in _POOLS:
        n = int(w.seq_lens[b])
        pool = oracle.new_pool(w.fmt, (n + 63) // 64)
        c, r = synth.kv_rows(w.seed, b, 0, n)
        oracle.cache_append(w.fmt, pool, c, r, np.arange(n, dtype=np.int32))
        _POOLS[key] = pool
    return _POOLS[key]


def _oracle_requests(w, budget_s: float, nthreads: int):
    import oracle
    ql, qr = w.queries()
    done, tokens, spent = 0, 0, 0.0
    b = 0
    while b < w.B and (spent < budget_s or done == 0):
        n = int(w.seq_lens[b])
        pages = (n + 63) // 64
        pool = _request_pool(w, b)
        bt = np.arange(pages, dtype=np.int32)[None]
        pairs = [(0, h) for h in range(w.H)]
        t0 = time.perf_counter()
        oracle.mla_decode(w.fmt, pool, ql[b:b + 1], qr[b:b + 1], bt, w.seq_lens[b:b + 1], w.scale,
                          pairs=pairs, nthreads=nthreads)
        spent += time.perf_counter() - t0
        tokens += n
        done += 1
        b += 1
    return tokens, spent, done


def cpu_baseline(w, budget_s: float = 12.0):
    import oracle
    nth = os.cpu_count() or 1
    oracle.build()
    tokens, spent, done = _oracle_requests(w, budget_s, nth)
    rb = 1152 if w.fmt == 0 else 656
    return {"value": round(tokens * rb / spent / 1e9, 6), "unit": UNIT, "cores": nth,
            "kind": "oracle",
            "sample": f"{done} of {w.B} requests of the {w.name} workload, all {w.H} heads, "
                      f"{tokens} attended positions, {spent:.1f} s of fp64 oracle time "
                      f"({nth} OpenMP threads)"}


def _reference_replicas(w):
    """The replica count and pool size our arm uses for this workload (for an identical config)."""
    rb = 1152 if w.fmt == 0 else 656
    one_pool = w.num_pages * 64 * rb
    kv = w.attended() * rb
    need = -(-3 * L2_BYTES // max(kv, 1))
    rep = 1 if need <= 1 else int(max(1, min(need + 1, 96, POOL_BUDGET // max(one_pool, 1))))
    return rep, one_pool


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from mla_latent_kv_decode_gb300 import synth
    import oracle
    oracle.build()
    w = synth.make_workload(args.workload)
    nth = os.cpu_count() or 1
    rb = 1152 if w.fmt == 0 else 656
    budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_requests(w, budget / 4, nth)
    tok, sec, req = 0, 0.0, 0
    for _ in range(args.steps):
        t, s, d = _oracle_requests(w, budget, nth)
        tok, sec, req = tok + t, sec + s, req + d
    value = tok * rb / sec / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, *_reference_replicas(w)),
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": nth, "kind": "oracle",
                             "sample": f"each step: whole requests of the {w.name} workload "
                                       f"(all heads) for ~{budget:.1f} s; {req} requests, {tok} "
                                       f"positions in total"},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_indexer_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from mla_latent_kv_decode_gb300 import synth
    import oracle
    oracle.build()
    w = synth.make_index_workload()
    nth = os.cpu_count() or 1
    budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_indexer_requests(w, budget / 4, nth)
    keys, sec, req = 0, 0.0, 0
    for _ in range(args.steps):
        k, s_, d = _oracle_indexer_requests(w, budget, nth)
        keys, sec, req = keys + k, sec + s_, req + d
    value = keys * 132 / sec / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "search-key GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "topk": w.K, "description": w.description},
            "cpu_baseline": {"value": round(value, 6), "unit": "search-key GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: whole queries of the {w.name} workload for ~{budget:.1f} s; "
                                       f"{req} queries, {keys} keys in total"},
            "e2e": {"value": round(value, 6), "unit": "search-key GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------------------------

HEADLINE = "fp8_batch"
CONFIG_ORDER = ["tiny_dense", "paged_batch", "long_context", "fp8_batch", "topk_sparse", "v4_batch", "v41_batch"]
SHARED_WORKLOADS = ("v4_batch", "v41_batch")
KV_FORMAT_NAMES = {0: "bf16", 1: "fp8_mixed", 2: "v4_fp8_584B", 3: "v41_fp4_288B"}
POOL_BUDGET = 48 << 30        # device bytes the pool replicas of one workload may take


def workload_config(w, replicas: int, one_pool: int, world: int = 1) -> dict:
    """The config object of a workload's line (the same for both arms)."""
    topk = 0 if w.topk_idx is None else int(w.topk_idx.shape[1])
    return {"workload": w.name, "B": w.B, "H": w.H, "kv_format": KV_FORMAT_NAMES[w.fmt],
            "description": w.description, "topk": topk, "page_tokens": 64, "scale": w.scale,
            "step": "cache_append of the tokens each request adds + mla_decode of the batch",
            "l2": f"inputs larger than L2: {replicas} rotating pool replicas of {one_pool / 2**20:.0f} MiB"
                  if replicas > 1 else "one pool, larger than L2",
            "parallelism": f"replicas x{world}"}


def _replicas(w, mla, kv_bytes: int) -> int:
    """Pool replicas whose touched record bytes exceed L2 three times (within POOL_BUDGET)."""
    one_pool = mla.pool_bytes(w.fmt, w.num_pages)
    need = -(-3 * L2_BYTES // max(kv_bytes, 1))
    if need <= 1:
        return 1
    return int(max(1, min(need + 1, 96, POOL_BUDGET // max(one_pool, 1))))


def _roofline(dw, dec_ms: float, peaks: dict, burst: bool) -> dict:
    """Roofline of one mla_decode call: its algorithmic bytes (or flops, where the flops at the
    tensor peak take longer than the bytes at the HBM peak) over its measured duration."""
    alg_bytes = dw.algorithmic_bytes()
    flops = dw.flops()
    dec_s = dec_ms / 1e3
    tpeak = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
    tensor_bound = flops / (tpeak * 1e12) > alg_bytes / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:
        r = {"bound": "tensor", "achieved": round(flops / dec_s / 1e12, 2), "peak": tpeak, "unit": "TFLOP/s",
             "frac": round(flops / dec_s / 1e12 / tpeak, 4),
             "peak_kind": "burst bf16 (graph of back-to-back calls timed alone)" if burst else "sustained bf16"}
    else:
        achieved = alg_bytes / dec_s / 1e9
        r = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": round(achieved / peaks["hbm_gbs"], 4)}
    r.update({"traffic": _traffic(dw.w.name), "peak_source": peaks["source"], "kernel": "mla_decode call",
              "ms_per_launch": round(dec_ms, 6), "bytes_per_launch": alg_bytes, "flops_per_launch": flops,
              "hbm_frac": round(alg_bytes / dec_s / 1e9 / peaks["hbm_gbs"], 4),
              "tensor_frac": round(flops / dec_s / 1e12 / tpeak, 4)})
    return r


class _Bench:
    """One workload on the device: pool replicas, CUDA graphs of the step (append + decode) and
    of back-to-back decode calls, and the timed legs."""

    def __init__(self, name, args, torch, mla, harness, synth, stream, barrier, dist, replicas=None):
        self.torch, self.mla, self.stream, self.barrier, self.dist = torch, mla, stream, barrier, dist
        shared = name in SHARED_WORKLOADS
        w = synth.make_shared_workload(name) if shared else synth.make_workload(name)
        self.w = w
        kv = int(w.attended() * mla.record_bytes(w.fmt))
        self.replicas = replicas if replicas is not None else (
            _replicas(w, mla, kv) if args.replicas == 0 else args.replicas)
        self.one_pool = mla.pool_bytes(w.fmt, w.num_pages)
        if shared:
            self.dw = dw = harness.SharedDeviceWorkload(w, replicas=self.replicas, appended=1)
        else:
            skip = 1 if w.appended == 0 else w.appended
            self.dw = dw = harness.DeviceWorkload(w, replicas=self.replicas, prefill_skip_last=skip)
        dw.alloc_outputs()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):      # eager warm-up (also sets kernel attributes)
            for r in range(self.replicas):
                dw.step(r)
        stream.synchronize()
        rc = mla.check_status()
        if rc != 0:
            raise mla.MlaError(rc, f"warm-up {name}")
        self.graphs = []
        for r in range(self.replicas):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                dw.step(r)
            self.graphs.append(g)
        self.reps = 20
        self.dec_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.dec_graph, stream=stream):
            for i in range(self.reps):
                dw.decode(i % self.replicas)

    def _timed(self, fn):
        torch = self.torch
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            fn()
            e1.record(self.stream)
        self.barrier()
        return e0.elapsed_time(e1)

    def steps(self, k: int, warmup: int) -> float:
        """ms of exactly k steps after `warmup` untimed ones (max over ranks)."""
        def run(n):
            for i in range(n):
                self.graphs[i % self.replicas].replay()
        with self.torch.cuda.stream(self.stream):
            run(warmup)
        self.barrier()
        return max_over_ranks(self._timed(lambda: run(k)), self.dist)

    def decode_ms(self, min_seconds: float) -> float:
        """Average ms of one decode call over graphs of back-to-back calls lasting at least
        min_seconds (the estimate of one replay sizes the loop)."""
        one = self._timed(lambda: self.dec_graph.replay())
        n = max(10, int(min_seconds * 1e3 / max(one, 1e-3)) + 1)
        def run():
            for _ in range(n):
                self.dec_graph.replay()
        return self._timed(run) / (n * self.reps)

    def cold_decode_ms(self, calls: int = 50) -> float:
        """Average ms of one decode call with L2 flushed before each (a buffer twice the size of
        L2 is written between calls; only the call itself is inside the events)."""
        torch = self.torch
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=self.dw.device)
        total = 0.0
        for _ in range(calls):
            with torch.cuda.stream(self.stream):
                flush.fill_(1)
            total += self._timed(lambda: self.dw.decode(0, self.stream))
        del flush
        return total / calls

    def free(self):
        del self.graphs, self.dec_graph, self.dw
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def measure_value_project(args, torch, mla, harness, stream, barrier, peaks, merged=False):
    """The value up-projection and output projection of a decode batch (B=64, 128 heads, d_v 128,
    hidden 5,120; Fig. 6 (2), or (3) with the merged weight): the call alone over >= the kernel
    leg's seconds of back-to-back calls alternating two weight replicas (370 MB, or 1.3 GB merged,
    larger than L2), and end to end with U copied in from pinned host memory and Y copied back."""
    B, H, D = 64, 128, 5120
    reps = [harness.ProjInputs(B, H, D, seed=0x4D4C41 + 7 + i, merged=merged) for i in range(2)]
    z = torch.empty((2, B, H * mla.D_V), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")

    def call(p):
        if merged:
            mla.value_project_merged(p.u, p.w_hat_t, y=y)
        else:
            mla.value_project(p.u, p.w_uv_t, p.w_o_t, z=z, y=y)

    with torch.cuda.stream(stream):
        for p in reps:
            call(p)
    stream.synchronize()
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "value projection warm-up")
    n_in = 20
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_in):
            call(reps[i % 2])

    def timed(fn):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            fn()
            e1.record(stream)
        barrier()
        return e0.elapsed_time(e1)

    one = timed(g.replay)
    n = max(10, int(args.kernel_seconds * 1e3 / max(one, 1e-3)) + 1)

    def loop():
        for _ in range(n):
            g.replay()
    ms = timed(loop) / (n * n_in)
    # end to end: U in from pinned host memory, the call, Y back, each step
    u_h = reps[0].u.cpu().pin_memory()
    y_h = torch.empty(y.shape, dtype=y.dtype).pin_memory()

    def e2e_step(i):
        p = reps[i % 2]
        p.u.copy_(u_h, non_blocking=True)
        call(p)
        y_h.copy_(y, non_blocking=True)
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    barrier()
    k = 50

    def e2e_loop():
        for i in range(k):
            e2e_step(i)
    e2e_ms = timed(e2e_loop) / k
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "value projection timed region")
    p = reps[0]
    alg = p.algorithmic_bytes()
    flops = p.flops()
    gbs = alg / (ms / 1e3) / 1e9
    entry = {"ms_per_call": round(ms, 6), "B": B, "H": H, "d_v": mla.D_V, "D": D,
             "form": "merged weight (Fig. 6 (3))" if merged else "two products (Fig. 6 (2))",
             "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": round(gbs / peaks["hbm_gbs"], 4),
                          "traffic": _traffic("value_project_merged" if merged else "value_project"),
                          "peak_source": peaks["source"], "bytes_per_launch": alg, "flops_per_launch": flops,
                          "tensor_frac": round(flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4)},
             "e2e": {"value": round(alg / (e2e_ms / 1e3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                     "h2d_bytes_per_step": int(u_h.numel() * 2), "d2h_bytes_per_step": int(y_h.numel() * 2),
                     "steps": k},
             "l2": "two weight replicas alternate (inputs larger than L2)"}
    del reps, z, y, g
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_value_project(args):
    """The value up-projection and output projection alone (one line, for profiling it): the
    measurement of measure_value_project, with the clocks of its run."""
    import torch
    import mla_latent_kv_decode_gb300 as mla
    from mla_latent_kv_decode_gb300 import harness
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    mla.load()
    stream = torch.cuda.Stream()
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    sampler.start()
    entry = measure_value_project(args, torch, mla, harness, stream, torch.cuda.synchronize, _peaks(),
                                  merged=args.workload == "value_project_merged")
    entry["clocks"] = sampler.stop()
    print(json.dumps({"metric": METRIC, "workload": args.workload, **entry}), flush=True)
    return 0


def run_ours(args):
    import torch
    import mla_latent_kv_decode_gb300 as mla
    from mla_latent_kv_decode_gb300 import harness, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    mla.load()
    peaks = _peaks()
    stream = torch.cuda.Stream()
    sampler = ClockSampler(local)
    sampler.start()
    headline = args.workload
    others = [] if args.no_configs else [n for n in CONFIG_ORDER if n != headline]

    # ---- the headline workload: exactly K timed steps, then the decode call alone ----
    bh = _Bench(headline, args, torch, mla, harness, synth, stream, barrier, dist)
    w, dw = bh.w, bh.dw
    ms = bh.steps(args.steps, args.warmup)
    dec_ms = bh.decode_ms(args.kernel_seconds)
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "timed region")
    e2e = run_e2e(args, dw, torch, mla, stream, barrier, dist)

    kv_bytes = dw.kv_bytes()
    flops = dw.flops()
    step_s = ms / 1e3 / args.steps
    value = job_value(world, kv_bytes, step_s) / 1e9
    topk = 0 if w.topk_idx is None else int(w.topk_idx.shape[1])
    launches_per_step = 1 + int(mla.load().mla_decode_launches(w.fmt, w.B, w.H, w.max_seq_len, topk))
    roofline = _roofline(dw, dec_ms, peaks, burst=True)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, bh.replicas, bh.one_pool, world),
        "decode_tokens_per_s": round(world * w.B / step_s, 1),
        "tflops": round(world * flops / step_s / 1e12, 3),
        "attended_tokens": w.attended(),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
    }
    bh.free()

    # ---- the other workloads: the same legs, reported under "configs" ----
    configs = {}
    for name in others:
        b = _Bench(name, args, torch, mla, harness, synth, stream, barrier, dist)
        k = max(args.steps, 20)
        c_ms = b.steps(k, max(args.warmup, 3))
        c_dec = b.decode_ms(args.kernel_seconds)
        rc = mla.check_status()
        if rc != 0:
            raise mla.MlaError(rc, f"timed region {name}")
        c_e2e = run_e2e(args, b.dw, torch, mla, stream, barrier, dist)
        entry = {"ms_per_step": round(c_ms / k, 6), "steps": k,
                 "value": round(job_value(world, b.dw.kv_bytes(), c_ms / 1e3 / k) / 1e9, 3), "unit": UNIT,
                 "ms_per_call": round(c_dec, 6),
                 "decode_tokens_per_s": round(world * b.w.B / (c_dec / 1e3), 1),
                 "roofline": _roofline(b.dw, c_dec, peaks, burst=True),
                 "e2e": c_e2e,
                 "config": workload_config(b.w, b.replicas, b.one_pool, world)}
        b.free()
        if name == "tiny_dense":
            # 4.7 MB fits in L2: the figure above is hot (one pool, back-to-back); cold = L2
            # flushed before every call
            hot = _Bench(name, args, torch, mla, harness, synth, stream, barrier, dist, replicas=1)
            cold_ms = hot.cold_decode_ms()
            hot_ms = hot.decode_ms(min(args.kernel_seconds, 0.5))
            entry["l2_hot"] = {"ms_per_call": round(hot_ms, 6), "roofline": _roofline(hot.dw, hot_ms, peaks, True),
                               "how": "one pool, back-to-back calls (the 4.7 MB cache stays in L2)"}
            entry["l2_cold"] = {"ms_per_call": round(cold_ms, 6), "roofline": _roofline(hot.dw, cold_ms, peaks, True),
                                "how": f"{2 * L2_BYTES / 2**20:.0f} MiB written before each call, outside the events"}
            hot.free()
        configs[name] = entry
    if not args.no_configs:
        configs["value_project"] = measure_value_project(args, torch, mla, harness, stream, barrier, peaks)
        configs["value_project_merged"] = measure_value_project(args, torch, mla, harness, stream, barrier, peaks,
                                                                merged=True)
        r = measure_indexer(args, torch, mla, stream, barrier, dist, world, peaks)
        configs["indexer_topk"] = {"ms_per_step": round(r["ms"], 6), "steps": r["steps"], "value": r["value"],
                                   "unit": r["unit"], "queries_per_s": r["queries_per_s"],
                                   "roofline": r["roofline"], "e2e": r["e2e"], "config": r["config"]}
    if configs:
        line["configs"] = configs
    line["clocks"] = sampler.stop()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def measure_indexer(args, torch, mla, stream, barrier, dist, world, peaks, sampler=None):
    """The DSA lightning-indexer step (search-key scores of every cached position, then top-k per
    query) on the indexer_topk workload: one graph of mla_indexer_score + mla_topk_select.
    Returns the workload, the step time and the line's figures; the device buffers are freed."""
    from mla_latent_kv_decode_gb300 import synth

    w = synth.make_index_workload(B=args.index_batch)
    pool = torch.zeros(mla.index_pool_bytes(w.num_pages), dtype=torch.uint8, device="cuda")
    chunk = 1 << 15
    kbuf = torch.empty((chunk, mla.INDEX_DIM), dtype=torch.bfloat16, device="cuda")
    for b in range(w.B):
        n = int(w.seq_lens[b])
        for t0 in range(0, n, chunk):
            t1 = min(n, t0 + chunk)
            synth.gpu_normal_bf16(kbuf.data_ptr(), t1 - t0, w.seed, synth.STREAM_IDX_K,
                                  (b * synth.KV_ROW_STRIDE + t0) * mla.INDEX_DIM, mla.INDEX_DIM, mla.INDEX_DIM)
            slot = torch.from_numpy(w.slots(b, t0, t1)).cuda()
            mla.index_append(pool, w.num_pages, kbuf[:t1 - t0], slot)
    del kbuf
    q = torch.from_numpy(synth.index_queries(w.seed, w.B).view(np.int16)).cuda().view(torch.bfloat16)
    wt = torch.from_numpy(synth.index_weights(w.seed, w.B)).cuda()
    bt = torch.from_numpy(w.block_table).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    ld = w.max_seq_len
    scores = torch.empty((w.B, ld), dtype=torch.float32, device="cuda")
    idx = torch.empty((w.B, w.K), dtype=torch.int32, device="cuda")

    def step():
        mla.indexer_score(pool, w.num_pages, q, wt, bt, sl, ld, scores=scores)
        mla.topk_select(scores, sl, w.K, topk_idx=idx)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "indexer warm-up")
    graphs = {}
    for name, fn in (("step", step),
                     ("score", lambda: mla.indexer_score(pool, w.num_pages, q, wt, bt, sl, ld, scores=scores)),
                     ("topk", lambda: mla.topk_select(scores, sl, w.K, topk_idx=idx))):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs[name] = g
    if sampler is not None:
        sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graphs["step"].replay()
    barrier()

    def timed(g, n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                g.replay()
            e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / n

    steps = min(args.steps, 500)
    ms = timed(graphs["step"], steps)
    ms = max_over_ranks(ms, dist)
    score_ms = timed(graphs["score"], max(10, steps // 2))
    topk_ms = timed(graphs["topk"], max(10, steps // 2))
    clocks = sampler.stop() if sampler is not None else None
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "indexer timed region")

    # end to end: queries, weights, tables host -> device, the step, the picks device -> host
    host = {k: v.cpu().pin_memory() for k, v in (("q", q), ("w", wt), ("bt", bt), ("sl", sl))}
    dev = {"q": q, "w": wt, "bt": bt, "sl": sl}
    idx_h = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = idx_h.numel() * idx_h.element_size()

    def one():
        for k in dev:
            dev[k].copy_(host[k], non_blocking=True)
        step()
        idx_h.copy_(idx, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
    barrier()
    e_steps = max(3, min(steps, 100))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e_steps):
            one()
        e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    del graphs, pool, q, wt, bt, sl, scores, idx
    torch.cuda.empty_cache()

    keys = int(w.seq_lens.astype(np.int64).sum())
    key_bytes = keys * 132
    alg_bytes = (key_bytes + w.B * 64 * 128 * 2 + w.B * 64 * 4 + w.B * w.K * 4 + w.block_table.size * 4
                 + w.B * 4)
    flops = 2 * 64 * 128 * keys
    s = ms / 1e3
    tensor_bound = flops / (peaks["bf16_tflops_sustained"] * 1e12) > alg_bytes / (peaks["hbm_gbs"] * 1e9)
    achieved = alg_bytes / s / 1e9
    if tensor_bound:
        roofline = {"bound": "tensor", "achieved": round(flops / s / 1e12, 2), "peak": peaks["bf16_tflops_sustained"],
                    "unit": "TFLOP/s", "frac": round(flops / s / 1e12 / peaks["bf16_tflops_sustained"], 4)}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4)}
    roofline.update({"traffic": _traffic(w.name), "peak_source": peaks["source"],
                     "kernel": "mla_indexer_score + mla_topk_select", "ms_per_launch": round(ms, 6),
                     "bytes_per_launch": alg_bytes, "flops_per_launch": flops,
                     "score_ms": round(score_ms, 6), "topk_ms": round(topk_ms, 6),
                     "score_frac_of_hbm": round(key_bytes / (score_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)})
    return {
        "w": w, "steps": steps, "ms": ms, "clocks": clocks,
        "value": round(world * key_bytes / s / 1e9, 3), "unit": "search-key GB/s",
        "config": {"workload": w.name, "B": w.B, "indexer_heads": 64, "indexer_dim": 128, "topk": w.K,
                   "description": w.description, "step": "mla_indexer_score + mla_topk_select",
                   "l2": f"inputs larger than L2: a {key_bytes / 2**30:.2f} GiB search-key pool",
                   "parallelism": f"replicas x{world}"},
        "queries_per_s": round(world * w.B / s, 1),
        "roofline": roofline,
        "e2e": {"value": round(world * key_bytes / (e2e_ms / 1e3) / 1e9, 3), "unit": "search-key GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e_steps,
                "ms_per_step": round(e2e_ms, 4)},
    }


def run_indexer(args):
    """The indexer_topk workload as its own JSON line (scores + top-k, with the oracle's CPU
    baseline)."""
    import torch
    import mla_latent_kv_decode_gb300 as mla

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    mla.load()
    r = measure_indexer(args, torch, mla, torch.cuda.Stream(), barrier, dist, world, _peaks(),
                        sampler=ClockSampler(local))
    w = r["w"]
    line = {
        "metric": METRIC, "value": r["value"], "unit": r["unit"],
        "n_gpus": world, "steps": r["steps"], "warmup": args.warmup, "ms_per_step": round(r["ms"], 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": r["config"],
        "queries_per_s": r["queries_per_s"],
        "roofline": r["roofline"],
        "clocks": r["clocks"],
        "e2e": r["e2e"],
        "gpu_launches": r["steps"] * 2,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = indexer_cpu_baseline(w, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def _oracle_indexer_requests(w, budget_s: float, nthreads: int):
    """The oracle's scores and top-k of whole requests of the indexer workload until the budget."""
    import oracle
    from mla_latent_kv_decode_gb300 import synth
    q = synth.index_queries(w.seed, w.B)
    wt = synth.index_weights(w.seed, w.B)
    done, keys, spent = 0, 0, 0.0
    while done < w.B and (spent < budget_s or done == 0):
        b = done
        n = int(w.seq_lens[b])
        pages = (n + 63) // 64
        pool = oracle.new_index_pool(pages)
        oracle.index_append(pool, synth.index_keys(w.seed, b, 0, n), np.arange(n, dtype=np.int32))
        bt = np.arange(pages, dtype=np.int32)[None]
        t0 = time.perf_counter()
        sc = oracle.indexer_scores(pool, q[b:b + 1], wt[b:b + 1], bt, w.seq_lens[b:b + 1], n, nthreads)
        oracle.topk(sc, w.seq_lens[b:b + 1], w.K, nthreads)
        spent += time.perf_counter() - t0
        keys += n
        done += 1
    return keys, spent, done


def indexer_cpu_baseline(w, budget_s: float = 12.0):
    import oracle
    nth = os.cpu_count() or 1
    oracle.build()
    keys, spent, done = _oracle_indexer_requests(w, budget_s, nth)
    return {"value": round(keys * 132 / spent / 1e9, 6), "unit": "search-key GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {w.B} queries of the {w.name} workload (scores of all {keys} keys, top-{w.K}), "
                      f"{spent:.1f} s of fp64 oracle time (one thread per query)"}


def _pack(torch, tensors, device):
    """One pinned host buffer and one device buffer holding `tensors` at 256-byte aligned offsets:
    (host buffer, device buffer, device views with the tensors' dtypes and shapes)."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev = torch.empty(total, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        host[o:o + n].copy_(t.detach().contiguous().view(torch.uint8).reshape(-1).cpu())
        views.append(dev[o:o + n].view(t.dtype).view(t.shape))
    return host, dev, views


def run_e2e(args, dw, torch, mla, stream, barrier, dist):
    """Same metric through the public API with pinned host buffers, as a serving loop runs it:
    every step's inputs (queries, block table, seq_lens, new rows and slots, packed in one pinned
    buffer) go host->device in one copy and its out + lse (one device buffer) come back in one
    copy, on a copy stream, while the compute stream runs append + decode of the step before
    (two input and two output buffers; events keep each buffer's writer after its last reader).
    Every copy of every step is inside the timed region."""
    names = [k for k in ("q_lat", "q_rope", "q", "sink", "rope_cs", "block_table", "seq_lens", "new_c", "new_r",
                         "new_e", "new_slot") if getattr(dw, k, None) is not None]
    saved = {k: getattr(dw, k) for k in names + ["out", "lse"]}
    ins = [_pack(torch, [saved[k] for k in names], dw.device) for _ in range(2)]
    outs = [_pack(torch, [saved["out"], saved["lse"]], dw.device) for _ in range(2)]
    h2d = ins[0][0].numel()
    d2h = outs[0][0].numel()
    steps = max(3, min(args.steps, 200))
    # one copy stream for both directions: a second one (measured) helped the batch workloads by
    # ~1.5 % and cost the long-context one ~10 % in host overhead
    hstream = dstream = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]     # inputs of the slot landed
    in_free = [ev(), ev()]      # the compute that read the slot's inputs is done
    out_ready = [ev(), ev()]    # the compute that wrote the slot's outputs is done
    out_free = [ev(), ev()]     # the copy that read the slot's outputs is done

    def run(n):
        with torch.cuda.stream(hstream):
            ins[0][1].copy_(ins[0][0], non_blocking=True)
            in_ready[0].record(hstream)
        for i in range(n):
            sl = i % 2
            stream.wait_event(in_ready[sl])
            if i >= 2:
                stream.wait_event(out_free[sl])
            for k, v in zip(names, ins[sl][2]):
                setattr(dw, k, v)
            dw.out, dw.lse = outs[sl][2]
            with torch.cuda.stream(stream):
                dw.step(i % dw.replicas)
            in_free[sl].record(stream)
            out_ready[sl].record(stream)
            if i + 1 < n:
                o = 1 - sl
                if i >= 1:
                    hstream.wait_event(in_free[o])
                with torch.cuda.stream(hstream):
                    ins[o][1].copy_(ins[o][0], non_blocking=True)
                    in_ready[o].record(hstream)
            dstream.wait_event(out_ready[sl])
            with torch.cuda.stream(dstream):
                outs[sl][0].copy_(outs[sl][1], non_blocking=True)
                out_free[sl].record(dstream)
        stream.wait_stream(hstream)

    try:
        run(3)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        hstream.wait_stream(stream)
        run(steps)
        e1.record(stream)
        barrier()
    finally:
        for k, v in saved.items():
            setattr(dw, k, v)
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, dist)
    world = 1 if dist is None else dist.get_world_size()
    value = job_value(world, dw.kv_bytes(), ms / 1e3 / steps) / 1e9
    return {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(ms / steps, 4),
            "overlap": "inputs of step i+1 and outputs of step i copied while step i+1 / i compute"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["tiny_dense", "paged_batch", "long_context", "fp8_batch", "topk_sparse",
                             "indexer_topk", "v4_batch", "v41_batch", "value_project", "value_project_merged"])
    ap.add_argument("--index-batch", type=int, default=64,
                    help="indexer_topk: queries per step (64 is the workload; smaller for profiling)")
    ap.add_argument("--replicas", type=int, default=0, help="pool replicas (0 = enough to exceed L2 3x)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="measure the headline workload only")
    ap.add_argument("--kernel-seconds", type=float, default=1.0,
                    help="minimum length of the back-to-back decode timing of each workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        if args.workload in SHARED_WORKLOADS or args.workload.startswith("value_project"):
            ap.error("the reference arm times the MLA workloads and the indexer")
        if args.workload == "indexer_topk":
            return run_indexer_reference(args)
        return run_reference(args)
    if args.workload == "indexer_topk":
        return run_indexer(args)
    if args.workload in ("value_project", "value_project_merged"):
        return run_value_project(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
