#!/usr/bin/env python3
"""Benchmark of absorbed MLA decode over a paged latent cache on GB300.

A step is one pass of the hot path over one batch: mla_cache_append of the newest token of
every request (bf16 record) followed by mla_decode of the whole batch (page gather, scores,
online softmax, weighted latent sum, split-KV merge).  Default workload: the batched paged
decode (B=32, H=128, seq_lens uniform in [1024, 8192], 64-token pages shuffled in a shared pool,
bf16 cache, scale 1/sqrt(192)).

Timing: W warm-up steps, then exactly K steps bracketed by a barrier and a device synchronise,
timed with CUDA events on the launching stream, max over ranks.  Each step is a CUDA graph of
the two library calls (the calls take about as long as the kernels, so eager launches would
time the host).  The inputs rotate over several identical pool replicas whose total exceeds L2,
so every step reads its cache from HBM.

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
# the workload; any change to that code makes the entry stale (traffic = null).  Captures: profiles/decode_tc_paged_batch.md,
# profiles/decode_gather_fp8_batch.md, profiles/indexer_score_indexer_topk.md.
_HEADERS = ["mla_latent_kv_decode_gb300/csrc/decode_common.cuh",
            "mla_latent_kv_decode_gb300/csrc/mla_internal.cuh",
            "mla_latent_kv_decode_gb300/csrc/tc_ptx.cuh",
            "include/mla.h"]
KERNEL_SOURCES = {
    "decode_tc": ["mla_latent_kv_decode_gb300/csrc/decode_tc.cu"] + _HEADERS,
    "decode_gather": ["mla_latent_kv_decode_gb300/csrc/decode_gather.cu"] + _HEADERS,
    "indexer_score": ["mla_latent_kv_decode_gb300/csrc/indexer.cu"] + _HEADERS,
}
WORKLOAD_KERNEL = {"tiny_dense": "decode_tc", "paged_batch": "decode_tc", "long_context": "decode_tc",
                   "fp8_batch": "decode_gather", "topk_sparse": "decode_gather",
                   "indexer_topk": "indexer_score"}
NCU_TRAFFIC = {
    ("c9436f9a11212c15", "paged_batch"): 178_121_984,
    ("c9436f9a11212c15", "long_context"): 155_761_152,
    ("317d8c4c452e69fa", "fp8_batch"): 1_414_574_592,
    ("317d8c4c452e69fa", "topk_sparse"): 122_382_592,
    ("a650593e7d15f670", "indexer_topk"): 1_144_615_680,
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

def _oracle_requests(w, budget_s: float, nthreads: int):
    import oracle
    from mla_latent_kv_decode_gb300 import synth
    ql, qr = w.queries()
    done, tokens, spent = 0, 0, 0.0
    b = 0
    while b < w.B and (spent < budget_s or done == 0):
        n = int(w.seq_lens[b])
        pages = (n + 63) // 64
        pool = oracle.new_pool(w.fmt, pages)
        c, r = synth.kv_rows(w.seed, b, 0, n)
        oracle.cache_append(w.fmt, pool, c, r, np.arange(n, dtype=np.int32))
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
            "config": {"workload": w.name, "B": w.B, "H": w.H, "kv_format": "bf16" if w.fmt == 0 else "fp8_mixed",
                       "description": w.description},
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
    w = synth.make_workload(args.workload)
    one_pool = mla.pool_bytes(w.fmt, w.num_pages)
    replicas = max(1, min(8, -(-3 * L2_BYTES // max(one_pool, 1)) + 1)) if args.replicas == 0 else args.replicas
    skip = 1 if w.appended == 0 else w.appended
    dw = harness.DeviceWorkload(w, replicas=replicas, prefill_skip_last=skip)
    dw.alloc_outputs()
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    # eager warm-up (also sets kernel attributes before capture)
    with torch.cuda.stream(stream):
        for r in range(replicas):
            dw.step(r)
    stream.synchronize()
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "warm-up")

    # one graph per replica: append + decode
    graphs = []
    for r in range(replicas):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            dw.step(r)
        graphs.append(g)
    dec_graphs = []
    reps = 20
    for r in range(replicas):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                dw.decode((r + i) % replicas)
        dec_graphs.append(g)

    sampler = ClockSampler(local)
    sampler.start()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % replicas].replay()
    barrier()

    # ---- timed region: exactly K steps ----
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            graphs[i % replicas].replay()
        ev1.record(stream)
    barrier()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, dist)

    # ---- decode-kernel timing (roofline): graphs of `reps` back-to-back decode calls ----
    n_dec = max(10, min(200, args.steps // reps + 1))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(n_dec):
            dec_graphs[i % replicas].replay()
        e1.record(stream)
    barrier()
    dec_ms = e0.elapsed_time(e1) / (n_dec * reps)
    clocks = sampler.stop()
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "timed region")

    # ---- end to end through the public API with host buffers ----
    e2e = run_e2e(args, dw, torch, mla, stream, barrier, dist)

    kv_bytes = dw.kv_bytes()
    alg_bytes = dw.algorithmic_bytes()
    flops = dw.flops()
    step_s = ms / 1e3 / args.steps
    value = job_value(world, kv_bytes, step_s) / 1e9
    peaks = _peaks()
    dec_s = dec_ms / 1e3
    achieved = alg_bytes / dec_s / 1e9
    traffic = _traffic(w.name)
    topk = 0 if w.topk_idx is None else int(w.topk_idx.shape[1])
    launches_per_step = 1 + int(mla.load().mla_decode_launches(w.fmt, w.B, w.H, w.max_seq_len, topk))
    # the bound of the call: HBM unless its flops at the dense bf16 peak take longer than its
    # bytes at the HBM peak (the FP8 batch: q stays bf16, the cache bytes halve)
    tensor_bound = flops / (peaks["bf16_tflops_sustained"] * 1e12) > alg_bytes / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:
        roofline = {"bound": "tensor", "achieved": round(flops / dec_s / 1e12, 2),
                    "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                    "frac": round(flops / dec_s / 1e12 / peaks["bf16_tflops_sustained"], 4)}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
    roofline.update({"traffic": traffic, "peak_source": peaks["source"], "kernel": "mla_decode call",
                     "ms_per_launch": round(dec_ms, 6), "bytes_per_launch": alg_bytes,
                     "flops_per_launch": flops})
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "kv_format": "bf16" if w.fmt == 0 else "fp8_mixed",
                   "seq_lens": "uniform in [1024, 8192]" if w.name == "paged_batch" else w.description,
                   "attended_tokens": w.attended(), "page_tokens": 64, "scale": w.scale,
                   "step": "cache_append of each request's newest token + mla_decode of the batch",
                   "l2": f"inputs larger than L2: {replicas} rotating pool replicas of "
                         f"{one_pool / 2**20:.0f} MiB", "parallelism": f"replicas x{world}"},
        "decode_tokens_per_s": round(world * w.B / step_s, 1),
        "tflops": round(world * flops / step_s / 1e12, 3),
        "step_frac_of_hbm_roofline": round((alg_bytes / (peaks['hbm_gbs'] * 1e9)) / step_s, 4),
        "roofline": roofline,
        "tensor_util": {"achieved_tflops": round(flops / dec_s / 1e12, 2),
                        "peak": peaks["bf16_tflops_sustained"],
                        "frac": round(flops / dec_s / 1e12 / peaks["bf16_tflops_sustained"], 4)},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_indexer(args):
    """The DSA lightning-indexer step (search-key scores of every cached position, then top-k per
    query) on the indexer_topk workload: one graph of mla_indexer_score + mla_topk_select."""
    import torch
    import mla_latent_kv_decode_gb300 as mla
    from mla_latent_kv_decode_gb300 import synth

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
    q = torch.from_numpy(synth.index_queries(w.seed, w.B).view(np.int16)).cuda().view(torch.bfloat16)
    wt = torch.from_numpy(synth.index_weights(w.seed, w.B)).cuda()
    bt = torch.from_numpy(w.block_table).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    ld = w.max_seq_len
    scores = torch.empty((w.B, ld), dtype=torch.float32, device="cuda")
    idx = torch.empty((w.B, w.K), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        mla.indexer_score(pool, w.num_pages, q, wt, bt, sl, ld, scores=scores)
        mla.topk_select(scores, sl, w.K, topk_idx=idx)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "warm-up")
    graphs = {}
    for name, fn in (("step", step),
                     ("score", lambda: mla.indexer_score(pool, w.num_pages, q, wt, bt, sl, ld, scores=scores)),
                     ("topk", lambda: mla.topk_select(scores, sl, w.K, topk_idx=idx))):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs[name] = g
    sampler = ClockSampler(local)
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
    clocks = sampler.stop()
    rc = mla.check_status()
    if rc != 0:
        raise mla.MlaError(rc, "timed region")

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

    keys = int(w.seq_lens.astype(np.int64).sum())
    key_bytes = keys * 132
    alg_bytes = (key_bytes + w.B * 64 * 128 * 2 + w.B * 64 * 4 + w.B * w.K * 4 + w.block_table.size * 4
                 + w.B * 4)
    flops = 2 * 64 * 128 * keys
    peaks = _peaks()
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
    line = {
        "metric": METRIC, "value": round(world * key_bytes / s / 1e9, 3), "unit": "search-key GB/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "indexer_heads": 64, "indexer_dim": 128, "topk": w.K,
                   "description": w.description, "step": "mla_indexer_score + mla_topk_select",
                   "l2": f"inputs larger than L2: a {key_bytes / 2**30:.2f} GiB search-key pool",
                   "parallelism": f"replicas x{world}"},
        "queries_per_s": round(world * w.B / s, 1),
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": round(world * key_bytes / (e2e_ms / 1e3) / 1e9, 3), "unit": "search-key GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e_steps,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": steps * 2,
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
    names = [k for k in ("q_lat", "q_rope", "block_table", "seq_lens", "new_c", "new_r", "new_slot")
             if getattr(dw, k) is not None]
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
    ap.add_argument("--workload", default="paged_batch",
                    choices=["tiny_dense", "paged_batch", "long_context", "fp8_batch", "topk_sparse",
                             "indexer_topk"])
    ap.add_argument("--index-batch", type=int, default=64,
                    help="indexer_topk: queries per step (64 is the workload; smaller for profiling)")
    ap.add_argument("--replicas", type=int, default=0, help="pool replicas (0 = enough to exceed L2 3x)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        if args.workload == "indexer_topk":
            return run_indexer_reference(args)
        return run_reference(args)
    if args.workload == "indexer_topk":
        return run_indexer(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
