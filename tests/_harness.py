"""Replay a workload on the GPU (through the C-ABI binding) and on the CPU
oracle, and compare.  Test infrastructure: the oracle side never sees a value
produced by the GPU side."""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import inputs

# tolerances: pass iff |gpu - ref| <= atol + rtol*|ref| element-wise, and the
# normalised RMS error ||gpu - ref|| / ||ref|| stays under nrms
TOL = {"f32": dict(atol=1e-5, rtol=0.0, nrms=1e-5),
       "f16": dict(atol=2e-2, rtol=2e-2, nrms=1e-2),
       "bf16": dict(atol=2e-2, rtol=2e-2, nrms=1e-2),
       "fp8_e4m3": dict(atol=6e-2, rtol=6e-2, nrms=3e-2),
       "fp8_e5m2": dict(atol=6e-2, rtol=6e-2, nrms=3e-2)}


def oracle_caches(wl: inputs.Workload):
    """The pool after the workload's setup and this step's write, by the oracle."""
    k = oracle.as_raw(wl.k_cache).copy()
    v = oracle.as_raw(wl.v_cache).copy()
    kvd, sd = oracle.DTYPE_CODES[wl.kv_dtype], oracle.DTYPE_CODES[wl.src_dtype]
    args = (wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_blocks)
    for kind, payload in wl.setup:
        if kind == "copy":
            oracle.copy_blocks(k, v, kvd, oracle.as_raw(payload), *args)
        else:
            oracle.reshape_and_cache(k, v, kvd, oracle.as_raw(payload.key), oracle.as_raw(payload.value), sd,
                                     oracle.as_raw(payload.slots), *args, wl.k_scale, wl.v_scale)
    oracle.reshape_and_cache(k, v, kvd, oracle.as_raw(wl.new_key), oracle.as_raw(wl.new_value), sd,
                             oracle.as_raw(wl.slot_mapping), *args, wl.k_scale, wl.v_scale)
    return k, v


def oracle_problem(wl: inputs.Workload, k, v, block_tables=None, seq_lens=None) -> oracle.Problem:
    return oracle.Problem(wl.q, oracle.DTYPE_CODES[wl.q_dtype], k, v, oracle.DTYPE_CODES[wl.kv_dtype],
                          wl.block_tables if block_tables is None else block_tables,
                          wl.seq_lens if seq_lens is None else seq_lens,
                          wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_blocks,
                          wl.scale, wl.k_scale, wl.v_scale)


def oracle_decode_threaded(prob: oracle.Problem, threads: int = 0) -> np.ndarray:
    """oracle.decode's result, computed as one oracle.attend_one call per
    (sequence, head) spread over host threads.  The oracle itself stays
    single-threaded; its C calls release the GIL, so independent calls run
    side by side.  Longest sequences go first so the threads finish together."""
    out = np.zeros((prob.num_seqs, prob.num_q_heads, prob.head_dim), dtype=np.float64)
    lens = prob.seq_lens.astype(np.int64)
    pairs = sorted(((i, h) for i in range(prob.num_seqs) for h in range(prob.num_q_heads)),
                   key=lambda ih: -int(lens[ih[0]]))

    def one(ih):
        out[ih[0], ih[1]] = oracle.attend_one(prob, ih[0], ih[1])

    with ThreadPoolExecutor(max_workers=threads or max(1, min(32, os.cpu_count() or 1))) as ex:
        list(ex.map(one, pairs))
    return out


class GpuStep:
    """Device copies of a workload; ``run`` replays setup + step write + decode."""

    def __init__(self, wl: inputs.Workload, device="cuda"):
        self.wl = wl
        self.dev = wl.to(device)
        # private pools: GPU writes must never reach the tensors the oracle reads
        self.dev.k_cache = self.dev.k_cache.clone()
        self.dev.v_cache = self.dev.v_cache.clone()
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.out = torch.empty(wl.q.shape, dtype=wl.q.dtype, device=device)

    def setup(self):
        d = self.dev
        for kind, payload in d.setup:
            if kind == "copy":
                pa.pa_copy_blocks(d.k_cache, d.v_cache, payload, err_flag=self.err)
            else:
                pa.pa_reshape_and_cache(d.k_cache, d.v_cache, payload.key, payload.value, payload.slots,
                                        k_scale=d.k_scale, v_scale=d.v_scale, err_flag=self.err)

    def write_step(self):
        d = self.dev
        pa.pa_reshape_and_cache(d.k_cache, d.v_cache, d.new_key, d.new_value, d.slot_mapping,
                                k_scale=d.k_scale, v_scale=d.v_scale, err_flag=self.err)

    def decode(self, simt=False, partition_tokens=0, workspace=None, block_tables=None, seq_lens=None,
               out=None):
        d = self.dev
        out = self.out if out is None else out
        pa.pa_decode(out, d.q, d.k_cache, d.v_cache, d.block_tables if block_tables is None else block_tables,
                     d.seq_lens if seq_lens is None else seq_lens, d.scale, k_scale=d.k_scale,
                     v_scale=d.v_scale, partition_tokens=partition_tokens, workspace=workspace,
                     err_flag=self.err, simt=simt)
        return out

    def run(self, simt=False, partition_tokens=0):
        self.setup()
        self.write_step()
        out = self.decode(simt=simt, partition_tokens=partition_tokens)
        torch.cuda.synchronize()
        return out


def compare(got: torch.Tensor, ref: np.ndarray, kv_dtype: str, what: str = ""):
    """Element-wise tolerance + normalised RMS; returns the stats dict."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    t = TOL[kv_dtype]
    err = np.abs(g - ref)
    bound = t["atol"] + t["rtol"] * np.abs(ref)
    bad = ~(err <= bound)
    nrms = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    stats = dict(max_abs=float(err.max()) if err.size else 0.0,
                 max_rel=float((err / np.maximum(np.abs(ref), 1e-30)).max()) if err.size else 0.0,
                 nrms=nrms, n_bad=int(bad.sum()), n=int(err.size))
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    assert stats["n_bad"] == 0, f"{what}: {stats['n_bad']} of {stats['n']} outside tolerance {t}; {stats}"
    assert nrms <= t["nrms"], f"{what}: normalised RMS {nrms:.3g} > {t['nrms']}; {stats}"
    return stats


def assert_caches_equal(step: GpuStep, k_ref: np.ndarray, v_ref: np.ndarray):
    kg = oracle.as_raw(step.dev.k_cache)
    vg = oracle.as_raw(step.dev.v_cache)
    assert np.array_equal(kg.view(np.uint8), k_ref.view(np.uint8)), "K pool differs from the oracle's"
    assert np.array_equal(vg.view(np.uint8), v_ref.view(np.uint8)), "V pool differs from the oracle's"
