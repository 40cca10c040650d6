#!/usr/bin/env python
"""Benchmark of the paged-KV decode hot path on GB300.

A step is one pass of the whole hot path over one batch: the cache write of
every sequence's new token (pa_reshape_and_cache), the copy-on-write block
copies when the workload has any (pa_copy_blocks), and paged decode
attention over the pool (pa_decode: main kernel + log-sum-exp reduce).

Default workload: a Qwen2.5-7B-like decode layer -- 28 query / 4 KV heads,
head_dim 128, block 16, fp16 KV, batch 64 with lengths uniform in [100, 8192]
over a shuffled 40,000-block pool (0.54 GB of K+V, larger than the 129 MB L2,
so every step streams the pool from HBM).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs the full
workload on its own GPU (independent sequences, no data exchange: weak
scaling); the value is all ranks' tokens over the slowest rank's time.
``--impl reference`` times the CPU oracle (the plain single-threaded
restatement of the pages' method) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import glob
import hashlib
import json
import math
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention tokens/s and achieved KV HBM GB/s (% of 8 TB/s) on 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def make_workload(name: str, seed: int, device: str):
    from paged_kv_cache_69_gb300 import inputs
    gd = device
    table = {
        "qwen7b_fp16": lambda: inputs.qwen7b_fp16(seed=seed, gen_device=gd),
        "short_mix_bf16_bs16": lambda: inputs.short_mix_bf16(seed=seed + 1, block_size=16, gen_device=gd),
        "short_mix_bf16_bs8": lambda: inputs.short_mix_bf16(seed=seed + 1, block_size=8, gen_device=gd),
        "prefix_share_fp16": lambda: inputs.prefix_share_fp16(seed=seed + 2, prompt_len=2048, gen_device=gd),
        "prefix_share_cow_fp16": lambda: inputs.prefix_share_fp16(seed=seed + 2, prompt_len=2040, gen_device=gd),
        "long_ctx_bf16": lambda: inputs.long_ctx("bf16", seed=seed + 3, gen_device=gd),
        "long_ctx_fp8": lambda: inputs.long_ctx("fp8_e4m3", seed=seed + 3, gen_device=gd),
        "long_ctx_fp8_e5m2": lambda: inputs.long_ctx("fp8_e5m2", seed=seed + 3, gen_device=gd),
        "tiny_fp32": lambda: inputs.tiny_fp32(seed=seed - 1),
    }
    return table[name]()


def workload_config(wl, extra=None) -> dict:
    cfg = {"workload": wl.name, "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
           "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
           "num_blocks": wl.num_blocks, "kv_dtype": wl.kv_dtype, "q_dtype": wl.q_dtype,
           "total_tokens": int(wl.seq_lens.sum()), "max_seq_len": int(wl.seq_lens.max())}
    if extra:
        cfg.update(extra)
    return cfg


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources the decode kernels (main + merge) and their launch code are built from
DECODE_SOURCES = ("pa_api.cu", "pa_common.h", "pa_decode_e4m3.cu", "pa_decode_kernel.cuh", "pa_decode_simt.cu",
                  "pa_decode_tc.cu", "pa_device.cuh", "pa_kernels.h")


def _code_only(text: str) -> str:
    """C/C++ source without comments or trailing blanks: the digest follows
    what is compiled, not the prose around it."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def source_digest() -> str:
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_69_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profile_name(workload: str, partition_tokens: int = 0, q_per_seq: int = 1, simt: bool = False) -> str:
    """File stem of the committed ncu summary of one bench configuration."""
    stem = f"pa_attention_{workload}_q{q_per_seq}" if q_per_seq > 1 else f"pa_decode_{workload}"
    return stem + ("_simt" if simt else "") + (f"_p{partition_tokens}" if partition_tokens else "")


def profile_traffic(name: str):
    """DRAM bytes per decode launch from the committed ncu summary `name`,
    when it was taken from the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{name}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    s = re.search(r"source_sha256:\s*([0-9a-f]+)", txt)
    if m and s and s.group(1) == source_digest():
        return int(m.group(1))
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML read-only queries)
# ---------------------------------------------------------------------------
def max_over_ranks(values, device, world):
    """Each value's maximum over all ranks: the slowest rank sets the job's
    time.  One all-reduce of a float64 vector (NCCL on GPUs, gloo on CPUs)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(units_per_rank_step, world, steps, ms_total):
    """Units all ranks processed per second over the max-over-ranks time."""
    return units_per_rank_step * world * steps / (ms_total / 1e3)


def capture_graph(fn):
    """fn's launches captured as one CUDA graph, or None (with a note on
    stderr) when capture fails; the eager launches are then timed instead."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            fn()
        torch.cuda.synchronize()
        return g
    except Exception as e:  # noqa: BLE001 -- any capture failure falls back to eager timing
        torch.cuda.synchronize()
        print(f"bench: CUDA graph capture failed ({e}); timing eager launches", file=sys.stderr)
        return None


class ClockSampler:
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, interval_s: float = 0.005):
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        self._interval = interval_s
        try:
            import torch
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
                if self.nvml.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.handle)) != 0:
                    return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.ok = True
        except Exception:
            self.ok = False

    def _sample(self):
        mhz = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        r1 = self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz))
        r2 = self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle, ctypes.byref(reasons))
        if r1 == 0:
            self.samples.append((int(mhz.value), int(reasons.value) if r2 == 0 else 0))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self._interval)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self) -> dict | None:
        if not self.ok:
            return None
        self._stop.set()
        self._thread.join()
        if not self.samples:
            self._sample()
        mhz = [s[0] for s in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if bits & b], "samples": len(mhz)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def host_cpu() -> dict:
    """The host's logical CPU count and CPU model name."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            import subprocess
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return {"nproc": os.cpu_count(), "cpu_model": model}



def oracle_inputs(wl):
    import oracle
    k = oracle.as_raw(wl.k_cache).copy()
    v = oracle.as_raw(wl.v_cache).copy()
    return k, v


def oracle_step(wl, k, v, seqs):
    """The oracle's cache write of the sampled sequences' new tokens, then
    their decode attention over every query head."""
    import numpy as np
    import oracle
    kvd, sd = oracle.DTYPE_CODES[wl.kv_dtype], oracle.DTYPE_CODES[wl.src_dtype]
    idx = np.array(seqs)
    oracle.reshape_and_cache(k, v, kvd, oracle.as_raw(wl.new_key)[idx], oracle.as_raw(wl.new_value)[idx], sd,
                             oracle.as_raw(wl.slot_mapping)[idx], wl.num_kv_heads, wl.head_dim,
                             wl.block_size, wl.num_blocks, wl.k_scale, wl.v_scale)
    prob = oracle.Problem(wl.q, oracle.DTYPE_CODES[wl.q_dtype], k, v, kvd, wl.block_tables, wl.seq_lens,
                          wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_blocks,
                          wl.scale, wl.k_scale, wl.v_scale)
    for i in seqs:
        for h in range(wl.num_q_heads):
            oracle.attend_one(prob, i, h)


def time_oracle(wl, budget_s: float = 15.0):
    """Sequences per second of the oracle over a bounded sample: sequences in
    workload order until ~budget_s of CPU work."""
    k, v = oracle_inputs(wl)
    done, t0 = [], time.perf_counter()
    for i in range(wl.num_seqs):
        oracle_step(wl, k, v, [i])
        done.append(i)
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return len(done) / el, len(done), el


# ---------------------------------------------------------------------------
def run_reference(args) -> dict:
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = make_workload(args.workload, 1, dev)
    wl = wl.to("cpu")
    k, v = oracle_inputs(wl)
    # a step: the oracle on a bounded sample of the workload (as many
    # sequences as fit in ~1.5 s, measured on the first one)
    t0 = time.perf_counter()
    oracle_step(wl, k, v, [0])
    one = time.perf_counter() - t0
    per_step = max(1, min(wl.num_seqs, int(1.5 / max(one, 1e-6))))
    seqs = list(range(per_step))
    for _ in range(args.warmup):
        oracle_step(wl, k, v, seqs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, k, v, seqs)
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    sample = (f"first {per_step} of {wl.num_seqs} sequences per step (all {wl.num_q_heads} query heads, "
              f"cache write + decode), oracle in plain C, one thread")
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, {"sample_seqs_per_step": per_step}),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample,
                             **host_cpu()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ours(args, rank, world, local) -> dict | None:
    import torch
    import torch.distributed as dist
    import paged_kv_cache_69_gb300 as pa
    from paged_kv_cache_69_gb300 import sizing

    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    pa.build()
    wl = make_workload(args.workload, 1, device)
    d = wl.to(device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    fill = None
    for kind, payload in d.setup:
        if kind == "copy":
            pa.pa_copy_blocks(d.k_cache, d.v_cache, payload, err_flag=err)
        else:
            # the pool's history arrives through the cache write: time the large fills
            fa, fb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            fa.record()
            pa.pa_reshape_and_cache(d.k_cache, d.v_cache, payload.key, payload.value, payload.slots,
                                    k_scale=d.k_scale, v_scale=d.v_scale, err_flag=err)
            fb.record()
            torch.cuda.synchronize()
            T = payload.slots.numel()
            if T >= 100000:
                nbytes = T * wl.num_kv_heads * wl.head_dim * 2 * (payload.key.element_size() +
                                                                  sizing.ELEM_BYTES[wl.kv_dtype])
                fill = {"tokens": T, "us": fa.elapsed_time(fb) * 1e3,
                        "gbs": nbytes / (fa.elapsed_time(fb) / 1e3) / 1e9}
    out = torch.empty_like(d.q)
    MB = d.block_tables.shape[1]
    ws = pa.alloc_workspace(d.num_seqs, d.num_q_heads, MB * d.block_size, d.head_dim, args.partition_tokens,
                            device=device)
    NQ = max(1, args.q_per_seq)
    if NQ > 1:
        # speculative-decoding step: the last NQ tokens of every sequence are queries (causal)
        gq = torch.Generator(device=device)
        gq.manual_seed(17)
        q_mq = torch.randn(d.num_seqs * NQ, d.num_q_heads, d.head_dim, generator=gq, device=device).to(d.q.dtype)
        out_mq = torch.empty_like(q_mq)
        qs_mq = torch.arange(0, d.num_seqs * NQ + 1, NQ, dtype=torch.int32, device=device)
        ws = torch.empty(pa.pa_attention_workspace_size(d.num_seqs, NQ, d.num_q_heads, MB * d.block_size, d.head_dim,
                                                        args.partition_tokens), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    pairs = d.cow_pairs if (d.cow_pairs is not None and d.cow_pairs.numel()) else None

    def write(q_, key_, val_, slots_):
        pa.pa_reshape_and_cache(d.k_cache, d.v_cache, key_, val_, slots_, k_scale=d.k_scale,
                                v_scale=d.v_scale, err_flag=err)

    def decode(q_, bt_, sl_, out_):
        if NQ > 1:
            pa.pa_attention(out_mq, q_mq, d.k_cache, d.v_cache, bt_, sl_, qs_mq, d.scale, NQ, k_scale=d.k_scale,
                            v_scale=d.v_scale, partition_tokens=args.partition_tokens, workspace=ws, err_flag=err)
            return
        pa.pa_decode(out_, q_, d.k_cache, d.v_cache, bt_, sl_, d.scale, k_scale=d.k_scale, v_scale=d.v_scale,
                     partition_tokens=args.partition_tokens, workspace=ws, err_flag=err, simt=args.simt)

    def step(q_, key_, val_, slots_, bt_, sl_, out_):
        if pairs is not None:
            pa.pa_copy_blocks(d.k_cache, d.v_cache, pairs, err_flag=err)
        write(q_, key_, val_, slots_)
        decode(q_, bt_, sl_, out_)

    dev_args = (d.q, d.new_key, d.new_value, d.slot_mapping, d.block_tables, d.seq_lens, out)
    for _ in range(args.warmup):
        step(*dev_args)
    torch.cuda.synchronize()
    # The step as one CUDA graph: replaying it keeps host launch gaps out of
    # the step time (the kernels and their order are those of the eager step).
    graph = None if args.eager else capture_graph(lambda: step(*dev_args))
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(local)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.start()
    t_start.record(stream)
    ew = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    ec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if graph is not None:
        # K steps replayed back to back: the step time
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t_start.record(stream)
        for _ in range(K):
            graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        g_start, g_end = t_start, t_end
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
    # Eager steps with events around each kernel: the per-kernel times (and
    # the step time when no graph is used).  Per-call times are medians over
    # at least 200 calls and about 0.5 s of work, so the clock sampler sees
    # the GPU under load for many samples.
    n_eager = K
    if graph is not None:
        step_ms = max(g_start.elapsed_time(g_end), 1e-3) / K
        n_eager = int(min(20000, max(K, 200, math.ceil(500.0 / step_ms))))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_eager)]
        ew = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_eager)]
        ec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_eager)]
    for i in range(n_eager):
        if pairs is not None:
            ec[i][0].record(stream)
            pa.pa_copy_blocks(d.k_cache, d.v_cache, pairs, err_flag=err)
            ec[i][1].record(stream)
        ew[i][0].record(stream)
        write(d.q, d.new_key, d.new_value, d.slot_mapping)
        ew[i][1].record(stream)
        ev[i][0].record(stream)
        decode(d.q, d.block_tables, d.seq_lens, out)
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms_total = g_start.elapsed_time(g_end) if graph is not None else t_start.elapsed_time(t_end)
    dec_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    write_us = statistics.median(a.elapsed_time(b) for a, b in ew) * 1e3
    copy_us = statistics.median(a.elapsed_time(b) for a, b in ec) * 1e3 if pairs is not None else None
    ms_total, dec_ms = max_over_ranks([ms_total, dec_ms], device, world)
    if err.item() != 0:
        raise RuntimeError(f"device error flag {err.item()} during the benchmark")

    # ---- end to end: host buffers, copies inside the timed region ----
    e2e = None
    if not args.no_e2e and NQ == 1:
        host = [x.cpu().pin_memory() for x in (d.q, d.new_key, d.new_value, d.slot_mapping, d.block_tables,
                                                d.seq_lens)]
        stage = [torch.empty_like(x) for x in (d.q, d.new_key, d.new_value, d.slot_mapping, d.block_tables,
                                               d.seq_lens)]
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in host)
        d2h = out_h.numel() * out_h.element_size()

        def e2e_step():
            for s_, h_ in zip(stage, host):
                s_.copy_(h_, non_blocking=True)
            step(stage[0], stage[1], stage[2], stage[3], stage[4], stage[5], out)
            out_h.copy_(out, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        g_e2e = None if args.eager else capture_graph(e2e_step)
        run_e2e = g_e2e.replay if g_e2e is not None else e2e_step
        for _ in range(args.warmup):
            run_e2e()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            run_e2e()
        b.record(stream)
        torch.cuda.synchronize()
        (te,) = max_over_ranks([a.elapsed_time(b)], device, world)
        e2e = {"value": job_throughput(wl.num_seqs, world, K, te), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    if rank != 0:
        return None
    lens = wl.seq_lens.tolist()
    alg = sizing.decode_algorithmic_bytes(lens, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.kv_dtype,
                                          wl.q_dtype)
    # queries and outputs of the extra query tokens
    alg += (NQ - 1) * wl.num_seqs * wl.num_q_heads * wl.head_dim * 2 * sizing.ELEM_BYTES[wl.q_dtype]
    if wl.meta.get("unique_tokens"):
        # shared prefix blocks are read once from HBM: count each unique token once
        alg = (wl.meta["unique_tokens"] * wl.num_kv_heads * wl.head_dim * sizing.ELEM_BYTES[wl.kv_dtype] * 2 +
               wl.num_seqs * wl.num_q_heads * wl.head_dim * 2 * sizing.ELEM_BYTES[wl.q_dtype])
    peak, peak_src = measured_peak()
    achieved = alg / (dec_ms / 1e3) / 1e9
    value = job_throughput(wl.num_seqs * NQ, world, K, ms_total)
    res = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
           "warmup": args.warmup, "ms_per_step": ms_total / K, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": wl.kv_dtype, "data": "synthetic",
           "config": workload_config(wl, {"l2": "inputs larger than L2 (K+V pool streamed each step)",
                                          "decode_variant": "cuda-core" if args.simt else "tensor-core",
                                          "partition_tokens": args.partition_tokens,
                                          "query_tokens_per_seq": NQ,
                                          "launch": "cuda_graph" if graph is not None else "eager",
                                          "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}),
           "kv_gbs": achieved, "pct_of_8tbs": 100.0 * achieved / NOMINAL_HBM_GBS,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                        "frac": achieved / peak, "peak_source": peak_src,
                        "kernel": "pa_decode (main + reduce)" if NQ == 1 else "pa_attention (main + reduce)",
                        "algorithmic_bytes_per_launch": alg,
                        "launch_ms": dec_ms, "launch_ms_stat": f"median of {n_eager} eager calls",
                        "traffic": profile_traffic(profile_name(args.workload, args.partition_tokens, NQ, args.simt)),
                        "profile": f"profiles/{profile_name(args.workload, args.partition_tokens, NQ, args.simt)}.md"},
           "gpu_launches": K * (3 + (1 if pairs is not None else 0)),
           "clocks": clk, "e2e": e2e,
           "cache_write_us_per_step": write_us,
           "copy_blocks_us_per_step": copy_us,
           "copy_blocks_pairs": int(pairs.shape[0]) if pairs is not None else 0}
    if fill is not None:
        res["cache_fill"] = fill
    if not args.no_cpu_baseline and world == 1:
        rate, n, el = time_oracle(wl.to("cpu"), budget_s=args.cpu_budget)
        res["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                               "sample": f"first {n} of {wl.num_seqs} sequences (all {wl.num_q_heads} query "
                                         f"heads, cache write + decode), {el:.1f} s, one thread",
                               **host_cpu()}
    return res


# ---------------------------------------------------------------------------
# host block manager (the allocator that feeds the GPU calls)
# ---------------------------------------------------------------------------
def _bm_trace(n_req: int, bs: int, seed: int):
    """Prompt token lists of a short-mix batch whose prompts start with one of
    four shared 256-token system prompts (prefix-cache hits)."""
    import random
    from paged_kv_cache_69_gb300 import inputs
    rnd = random.Random(seed)
    systems = [[rnd.randrange(150000) for _ in range(256)] for _ in range(4)]
    lens = inputs.short_mix_lens(seed, n_req)
    return [systems[i % 4] + [rnd.randrange(150000) for _ in range(L)] for i, L in enumerate(lens)]


def _bm_run(make, hash_fn, prompts, bs, decode_steps, reqs_cap=None):
    """Admit every prompt (prefix lookup + allocation), then decode_steps
    steps of one token per request with the step's block tables; returns
    (admit seconds, seconds per decode step, requests admitted)."""
    import numpy as np
    from paged_kv_cache_69_gb300 import block_manager as hbm
    m = make()
    prompts = prompts[:reqs_cap] if reqs_cap else prompts
    t0 = time.perf_counter()
    for r, p in enumerate(prompts):
        m.allocate(r, len(p), hash_fn(p, bs))
    t1 = time.perf_counter()
    reqs = np.arange(len(prompts), dtype=np.int64)
    maxb = max(-(-(len(p) + decode_steps) // bs) for p in prompts)
    tables = hbm.BlockTableBuffer(len(prompts), maxb) if hasattr(m, "append_slots") else None
    for _ in range(decode_steps):
        if tables is not None:
            m.append_slots(reqs)
            tables.update(m, reqs)
        else:
            for r in reqs.tolist():
                m.append_slot(r)
            np.array([m.block_table(r) + [-1] * (maxb - len(m.block_table(r))) for r in reqs.tolist()], np.int32)
    t2 = time.perf_counter()
    return t1 - t0, (t2 - t1) / decode_steps, len(prompts)


def run_block_manager(args) -> dict:
    from oracle import block_pool as obp
    from paged_kv_cache_69_gb300 import block_manager as hbm
    n_req, bs, steps = 1024, 16, max(args.steps, 10)
    prompts = _bm_trace(n_req, bs, 2)
    nb = sum(-(-(len(p) + steps) // bs) for p in prompts) + 64
    # warm-up, then the timed run
    _bm_run(lambda: hbm.HostBlockManager(nb, bs), hbm.block_hashes, prompts, bs, 2)
    admit, step, n = _bm_run(lambda: hbm.HostBlockManager(nb, bs), hbm.block_hashes, prompts, bs, steps)
    # the oracle on a bounded sample of the same trace
    o_admit, o_step, o_n = _bm_run(lambda: obp.BlockManager(nb, bs), obp.chain_hashes, prompts, bs, 5,
                                   reqs_cap=256)
    return {"metric": "host block manager: decode step (one token for each of 1024 requests + block tables)",
            "component": "block_manager", "value": step * 1e6, "unit": "us", "higher_is_better": False,
            "steps": steps, "config": {"workload": "short mix prompts behind 4 shared 256-token system prompts",
                                       "requests": n, "block_size": bs, "num_blocks": nb},
            "admit_us_per_request": admit / n * 1e6, "tokens_per_s": n / step,
            "cpu_baseline": {"value": o_step * (n / o_n) * 1e6, "unit": "us", "cores": 1, "kind": "oracle",
                             "sample": f"first {o_n} requests, 5 steps, scaled to {n} requests"}}


# ---------------------------------------------------------------------------
# block copies: all-layer copy-on-write and swap through pinned host memory
# ---------------------------------------------------------------------------
def run_block_copy(args) -> dict:
    import torch
    import paged_kv_cache_69_gb300 as pa
    torch.cuda.set_device(0)
    dev = "cuda"
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps * 1e-3          # seconds per call

    # swap: 4096 scattered blocks of the 7B-like layer (16 x 4 x 128 fp16 = 16 KB each for K and V)
    NB, NH, bs, Hkv, D, P = 40000, 4096, 16, 4, 128, 4096
    g = torch.Generator().manual_seed(0)
    dk = torch.randn(NB, bs, Hkv, D, device=dev, dtype=torch.float16)
    dv = torch.randn(NB, bs, Hkv, D, device=dev, dtype=torch.float16)
    hk = torch.empty(NH, bs, Hkv, D, dtype=torch.float16).pin_memory()
    hv = torch.empty(NH, bs, Hkv, D, dtype=torch.float16).pin_memory()
    src = torch.randperm(NB, generator=g)[:P]
    out_pairs = torch.stack([src, torch.arange(P)], 1).to(dev)
    in_pairs = torch.stack([torch.arange(P), torch.randperm(NB, generator=g)[:P]], 1).to(dev)
    block_bytes = bs * Hkv * D * 2
    moved = 2 * P * block_bytes                                   # K and V
    t_out = timed(lambda: pa.pa_swap_blocks(hk, hv, dk, dv, out_pairs), 20)
    t_in = timed(lambda: pa.pa_swap_blocks(dk, dv, hk, hv, in_pairs), 20)
    flat_d = torch.empty(moved // 2, dtype=torch.float16, device=dev)
    flat_h = torch.empty(moved // 2, dtype=torch.float16).pin_memory()
    t_flat_out = timed(lambda: flat_h.copy_(flat_d, non_blocking=True), 20)
    t_flat_in = timed(lambda: flat_d.copy_(flat_h, non_blocking=True), 20)
    del dk, dv, hk, hv, flat_d, flat_h
    torch.cuda.empty_cache()
    # all-layer copy-on-write: 96 pairs (the prefix-sharing COW step) in 28
    # layers of 2048-block pools (1.8 GB on the device)
    L, NB2, pairs_n = 28, 2048, 96
    ks = [torch.randn(NB2, bs, Hkv, D, device=dev, dtype=torch.float16) for _ in range(L)]
    vs = [torch.randn(NB2, bs, Hkv, D, device=dev, dtype=torch.float16) for _ in range(L)]
    perm = torch.randperm(NB2, generator=g)
    cow = torch.stack([perm[:pairs_n], perm[pairs_n:2 * pairs_n]], 1).to(dev)
    t_cow = timed(lambda: pa.pa_copy_blocks_layers(ks, vs, cow), 50)
    cow_bytes = L * pairs_n * 2 * block_bytes * 2                 # K and V, read + write
    # the same kernel on 1024 pairs x 28 layers (1.8 GB moved, far beyond L2)
    pairs_l = 1024
    cow_l = torch.stack([perm[:pairs_l], perm[pairs_l:2 * pairs_l]], 1).to(dev)
    t_cow_l = timed(lambda: pa.pa_copy_blocks_layers(ks, vs, cow_l), 10)
    cow_l_bytes = L * pairs_l * 2 * block_bytes * 2
    peak, src_peak = measured_peak()
    return {"metric": "block copies: swap through pinned host memory and all-layer copy-on-write",
            "component": "block_copy", "unit": "GB/s", "higher_is_better": True,
            "value": moved / t_out / 1e9,
            "config": {"workload": "4096 scattered 32 KB blocks (K+V, 7B-like layer) out to pinned host and back; "
                                   "96 COW pairs x 28 layers", "block_bytes_k_or_v": block_bytes},
            "swap_out_gbs": moved / t_out / 1e9, "swap_in_gbs": moved / t_in / 1e9,
            "contiguous_d2h_gbs": moved / t_flat_out / 1e9, "contiguous_h2d_gbs": moved / t_flat_in / 1e9,
            "swap_out_frac_of_contiguous": t_flat_out / t_out, "swap_in_frac_of_contiguous": t_flat_in / t_in,
            "cow_all_layers_us": t_cow * 1e6, "cow_all_layers_gbs": cow_bytes / t_cow / 1e9,
            "copy_1024_pairs_28_layers_us": t_cow_l * 1e6, "copy_1024_pairs_28_layers_gbs": cow_l_bytes / t_cow_l / 1e9,
            "copy_1024_pairs_28_layers_frac": cow_l_bytes / t_cow_l / 1e9 / peak,
            "roofline": {"bound": "hbm", "kernel": "block_copy_kernel (28-layer COW)",
                         "achieved": cow_bytes / t_cow / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": cow_bytes / t_cow / 1e9 / peak, "peak_source": src_peak, "traffic": None}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen7b_fp16")
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--simt", action="store_true", help="time the CUDA-core decode variant")
    ap.add_argument("--q-per-seq", type=int, default=1,
                    help="query tokens per sequence (>1: speculative-decoding step through pa_attention)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time the step as eager launches instead of a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--component", choices=["decode", "block_manager", "block_copy"], default="decode",
                    help="block_manager: the host allocator; block_copy: swap and all-layer copies")
    args = ap.parse_args()
    if args.component != "decode":
        if int(os.environ.get("RANK", "0")) == 0:
            run = run_block_manager if args.component == "block_manager" else run_block_copy
            print(json.dumps(run(args)))
        return
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local)
    if res is not None:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
