#!/usr/bin/env python
"""Benchmark of the GQA-over-preallocated-KV-cache hot path on one GB300.

Default workload: Llama-3.1-8B-shaped single-layer decode (B=32, Hq=32,
Hkv=8, d=128, bf16 cache [32, 8, 8192, 128], initial lengths uniform in
[1024, 7936], T=1, one appended token per row per step).  A step is one pass
of the whole path: the in-place append of the step's K/V and the attention of
the step's queries (libkvc kernels, one launch each).  The headline metric is
KV-read GB/s: live K/V bytes the attention must read (sum over rows of
lens * Hkv * d * 2 (K and V) * 2 B) divided by the step time.

Other workloads (--workload): verify (B=64, S=4096, T=4), prefill (B=4,
Hkv=8, chunk T=512 on priors that are multiples of 512; metric attention
TFLOP/s over visible pairs), longctx (32 layers of [4, 8, 131072, 128]).

--impl reference times the CPU float64 oracle (the only reference this
method has) on a bounded sample of the same workload, on the host cores.
Multi-GPU: replicas only (each rank runs its own independent cache; no
collective), weak scaling, max time over ranks.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")  # the CPU baseline runs on one thread, stated as cores = 1

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gqa_attention_preallocated_gb300 import workloads as wl  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples go to a temporary file; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"kvc_bench_clocks_gpu{index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Workload set-up (inputs resident in HBM before timing starts)
# ---------------------------------------------------------------------------


def kv_bytes(lens, Hkv, d, esize=2):
    return int(np.sum(lens)) * Hkv * d * 2 * esize


def visible_pairs(priors, n_new):
    # sum over rows of sum_{t < n} (prior + t + 1)
    return int(sum(int(n) * int(p) + int(n) * (int(n) + 1) // 2 for p, n in zip(priors, n_new)))


FP8_SCALE = 4.0 / 448  # N(0,1) content: 4 sigma maps to the largest E4M3 value


def _fill_fp8_(dst: torch.Tensor, seed: int, stream: int, chunk: int = 1 << 26) -> None:
    """Synthetic FP8 cache content: codes of normal(seed, stream) / FP8_SCALE (clamped to +-448)."""
    flat = dst.view(-1)
    for start in range(0, flat.numel(), chunk):
        stop = min(flat.numel(), start + chunk)
        idx = torch.arange(start, stop, dtype=torch.int64, device=dst.device)
        x = wl.normal_at(seed, stream, idx).to(torch.float32) / FP8_SCALE
        flat[start:stop] = x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)


def make_cache(shape, layers, lens0, seed, kv_dtype="bf16"):
    from gqa_attention_preallocated_gb300 import KVCache

    fp8 = kv_dtype == "fp8"
    cache = KVCache(layers, shape.B, shape.Hkv, shape.max_len, shape.d,
                    dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16, device="cuda")
    for layer in range(layers):
        if fp8:
            sc = np.full(shape.Hkv, FP8_SCALE, dtype=np.float32)
            cache.set_kv_scales(layer, sc, sc)
            _fill_fp8_(cache.k[layer], seed, wl.STREAM_CACHE_K + 16 * layer)
            _fill_fp8_(cache.v[layer], seed, wl.STREAM_CACHE_V + 16 * layer)
        else:
            wl.fill_normal_(cache.k[layer], seed, wl.STREAM_CACHE_K + 16 * layer)
            wl.fill_normal_(cache.v[layer], seed, wl.STREAM_CACHE_V + 16 * layer)
        cache.set_lens(layer, lens0)
    return cache


def step_inputs(shape, Hq, T, n_distinct, seed, device="cuda"):
    q = [wl.to_storage(wl.normal(seed, 5000 + i, (shape.B, Hq, T, shape.d), device=device), torch.bfloat16)
         for i in range(n_distinct)]
    k = [wl.to_storage(wl.normal(seed, 1000 + 2 * i, (shape.B, shape.Hkv, T, shape.d), device=device), torch.bfloat16)
         for i in range(n_distinct)]
    v = [wl.to_storage(wl.normal(seed, 1001 + 2 * i, (shape.B, shape.Hkv, T, shape.d), device=device), torch.bfloat16)
         for i in range(n_distinct)]
    return q, k, v


class Workload:
    """One named workload: set-up, one step, and the step's algorithmic work."""

    def __init__(self, name, seed=0, verify_t=4, verify_g=4, kv_dtype="bf16", prefill_ragged=False, head_dim=128):
        self.name = name
        self.ragged = False
        self.seed = seed
        self.kv_dtype = kv_dtype  # "bf16", or "fp8": E4M3 cache with one scale per KV head
        self.esize = 1 if kv_dtype == "fp8" else 2
        if head_dim not in (64, 128) or (head_dim == 64 and (name != "decode8b" or kv_dtype != "bf16")):
            raise SystemExit("--head-dim 64 applies to the bf16 decode8b workload")
        if name == "decode8b":
            s = self.shape = wl.DECODE_8B
            if head_dim == 64:  # the same decode shape with 64-wide heads
                s = self.shape = wl.Shape("decode_b32_hq32_hkv8_d64_len8192_bf16", B=32, Hq=32, Hkv=8, d=64,
                                          max_len=8192, dtype="bf16")
            self.layers, self.Hq, self.T = 1, s.Hq, 1
            self.lens0 = wl.decode_lens(seed, s.B, 1024, s.max_len - 256)
            self.n_new = np.ones(s.B, dtype=np.int64)
            self.rollback_every = 256  # the workload's 256 steps, then back to the initial lengths
            self.metric, self.unit = "GQA decode KV-read HBM GB/s", "GB/s"
        elif name == "verify":
            s = self.shape = wl.VERIFY
            # the verify sweep: T drafts in {4, 8} (16 beyond it), G = Hq / Hkv in {1, 2, 4, 8} (16 beyond it)
            self.layers, self.Hq, self.T = 1, verify_g * s.Hkv, verify_t
            self.lens0 = np.full(s.B, s.max_len - self.T, dtype=np.int64)
            self.n_new = np.full(s.B, self.T, dtype=np.int64)
            self.rollback_every = 1  # speculative verify: append T, attend, truncate back
            self.metric, self.unit = "GQA speculative-verify KV-read HBM GB/s", "GB/s"
        elif name == "prefill":
            s = self.shape = wl.PREFILL
            self.layers, self.Hq, self.T = 1, s.Hq, 512
            self.lens0 = wl.prefill_priors(seed, s.B)
            self.n_new = np.full(s.B, 512, dtype=np.int64)
            if prefill_ragged:  # the ragged final chunk: T = 512 padded, n_new[b] uniform in 1..512
                self.ragged = True
                self.n_new = wl.ragged_chunk(seed, s.B)
            self.rollback_every = 1
            self.metric, self.unit = "GQA chunked-prefill attention TFLOP/s", "TFLOP/s"
        elif name == "longctx":
            s = self.shape = wl.LONGCTX
            self.layers, self.Hq, self.T = s.layers, s.Hq, 1
            self.lens0 = wl.decode_lens(seed, s.B, 32768, s.max_len - 64)
            self.n_new = np.ones(s.B, dtype=np.int64)
            self.rollback_every = 64
            self.metric, self.unit = "GQA long-context 32-layer decode KV-read HBM GB/s", "GB/s"
        else:
            raise SystemExit(f"unknown workload {name}")

    def config(self):
        s = self.shape
        name = s.name + ("_ragged_final_chunk" if self.ragged else "") + ("_fp8_cache" if self.kv_dtype == "fp8" else "")
        extra = {"n_new": [int(x) for x in self.n_new]} if self.ragged else {}
        return {"workload": name, **extra, "B": s.B, "Hq": self.Hq,
                "Hkv": s.Hkv, "d": s.d, "max_len": s.max_len,
                "layers": self.layers, "T": self.T, "dtype": "bf16",
                "kv_storage": "fp8_e4m3 (one scale per KV head)" if self.kv_dtype == "fp8" else "bf16",
                "initial_lens": {"min": int(self.lens0.min()), "max": int(self.lens0.max()),
                                 "mean": float(self.lens0.mean())},
                "l2": self.l2_statement()}

    def l2_statement(self):
        """How the timed steps meet the L2 (no flush between steps; the reason, with sizes)."""
        l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size if torch.cuda.is_available() \
            else 126 << 20
        live = kv_bytes(self.lens_at(0), self.shape.Hkv, self.shape.d, self.esize) * self.layers
        if self.unit == "TFLOP/s":
            return (f"no flush: tensor-bound (about 2,000 FLOP per K/V byte); each step reads {live / 1e6:.0f} MB "
                    f"of live K/V ({live / l2:.1f}x the {l2 / 1e6:.0f} MB L2) in about a tenth of its time")
        return (f"no flush, no rotation: each step reads all live K/V, {live / 1e6:.0f} MB "
                f"({live / l2:.1f}x the {l2 / 1e6:.0f} MB L2), in the same order as the step before, "
                f"so those lines are evicted before they are read again" + _committed_l2(self))

    def lens_at(self, i):
        """Lengths after the append of step i (steps counted from the last rollback)."""
        return self.lens0 + self.n_new * ((i % self.rollback_every) + 1)

    def work(self, i):
        """Algorithmic units of step i in the metric's unit numerator (bytes or FLOPs)."""
        s = self.shape
        if self.unit == "TFLOP/s":
            return 4 * s.d * self.Hq * visible_pairs(self.lens0, self.n_new)
        return kv_bytes(self.lens_at(i), s.Hkv, s.d, self.esize) * self.layers

    @property
    def tc_min_rows(self):
        """Query rows per KV head above which the library runs attention on the tcgen05 kernel."""
        return 32 if self.kv_dtype == "fp8" else 12

    @property
    def tensor_core(self):
        return (self.Hq // self.shape.Hkv) * self.T > self.tc_min_rows

    @property
    def kernel_name(self):
        """The dominant kernel of the timed attention call."""
        if self.tensor_core:
            rows = "128 positions per head" if self.T >= 128 else "packed rows g*T+t of a KV head"
            return f"prefill_tc_kernel (tcgen05/TMEM, {rows}; cut items merged in-kernel)"
        return "decode_splitkv_bf16_kernel (+ combine_bf16_kernel" + (", append fused in)" if self.fused else ")")

    @property
    def kernel_source(self):
        return "prefill_tc.cu" if self.tensor_core else "decode_bf16.cu"

    @property
    def fused(self):
        """The library appends inside the attention launch when the split-KV kernel runs it on one
        16-row MMA tile per KV head (up to 16 query rows)."""
        return not self.tensor_core and (self.Hq // self.shape.Hkv) * self.T <= 16

    def kernel_bytes(self, i):
        """Algorithmic bytes of the timed attention call: live K/V + q + out (+ the append when fused)."""
        s = self.shape
        qo = 2 * s.B * self.Hq * self.T * s.d * 2
        # fused append: bf16 rows read, stored rows written (K and V)
        app = 2 * int(np.sum(self.n_new)) * s.Hkv * s.d * (2 + self.esize) if self.fused else 0
        return kv_bytes(self.lens_at(i), s.Hkv, s.d, self.esize) + qo + app


def run_native(w: Workload, steps: int, warmup: int, rank: int, world: int):
    from gqa_attention_preallocated_gb300 import KVCache  # noqa: F401

    s = w.shape
    torch.cuda.synchronize()
    cache = make_cache(s, w.layers, w.lens0, w.seed + rank, w.kv_dtype)
    n_distinct = min(max(steps, 1), 16)
    q, k, v = step_inputs(s, w.Hq, w.T, n_distinct, w.seed + rank)
    out = torch.empty_like(q[0])
    ws = cache.workspace(w.Hq, w.T)
    stream = torch.cuda.current_stream()

    def one_step(i):
        # One pass of the whole path: append + attention for every layer (one
        # C-ABI call per layer; the library fuses the append into the
        # attention launch where warps own whole tiles).
        if i > 0 and i % w.rollback_every == 0:
            cache.truncate(w.lens0)
        j = i % n_distinct
        for layer in range(w.layers):
            cache.append_attention(layer, q[j], k[j], v[j], w.n_new, out=out, workspace=ws)

    for i in range(warmup):
        one_step(i)
    cache.truncate(w.lens0)
    torch.cuda.synchronize()

    # Timed region: K steps back to back, events only at its two ends.
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = cache.kernel_launches()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_wall = time.perf_counter()
        start.record(stream)
        for i in range(steps):
            one_step(i)
        stop.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    launches = cache.kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    ms = start.elapsed_time(stop)

    # Kernel time for the roofline: the average duration of the attention
    # launch when launches run back to back, as in the timed region (an event
    # pair around every call would break the chaining of consecutive launches
    # and time each launch's start-up alone).  Fused steps (the attention
    # launch also appends) are one attention launch per layer call, so the
    # timed region itself is that chain.  Otherwise the append runs once and
    # K attention-only calls of layer 0 on the same lengths are chained
    # between one event pair.
    cache.truncate(w.lens0)
    torch.cuda.synchronize()
    if w.fused:
        attn_ms = ms / (steps * w.layers)
        kbytes = [w.kernel_bytes(i) for i in range(steps)]
        kernel_timing = "timed region / (steps x layers): fused attention launches back to back"
    else:
        cache.append(0, k[0], v[0], w.n_new)
        for _ in range(2):  # warm the chain
            cache.gqa_attention(0, q[0], w.n_new, out=out, workspace=ws)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a0.record(stream)
        for i in range(steps):
            cache.gqa_attention(0, q[i % n_distinct], w.n_new, out=out, workspace=ws)
        a1.record(stream)
        torch.cuda.synchronize()
        attn_ms = a0.elapsed_time(a1) / steps
        kbytes = [w.kernel_bytes(0)] * steps
        kernel_timing = f"{steps} attention-only calls of layer 0 back to back between one event pair (append before)"
    status = cache.device_status(ws)
    work = sum(w.work(i) for i in range(steps))
    res = {
        "ms": ms, "wall_s": t_wall, "work": work, "attn_ms": attn_ms, "kernel_timing": kernel_timing,
        "kernel_bytes": kbytes, "launches": launches, "clocks": clk.summary(), "status": status,
    }
    res["e2e"] = run_e2e(w, cache, steps, q, k, v)
    if w.fused:
        res["graph"] = run_graph(w, cache, steps, q, k, v)
    return res


def run_graph(w: Workload, cache, steps: int, q, k, v):
    """The same steps as one CUDA graph replay each (lengths resident on the device).

    One step (per layer: device plan, attention with the append fused in,
    combine) is captured per distinct input set, reading that set's q / k_new
    / v_new in place (as a model's own producing kernels would leave them);
    each step is one replay.  The rollback rewrites the device lengths.
    """
    n_distinct = len(q)
    ws = cache.workspace(w.Hq, w.T)
    cache.truncate(w.lens0)
    torch.cuda.synchronize()
    dev_lens = cache.lens_to_device()
    lens0 = torch.from_numpy(w.lens0.astype(np.int32)).cuda().view(1, -1).expand(w.layers, -1)
    snn = torch.from_numpy(w.n_new.astype(np.int32)).cuda()
    sout = torch.empty_like(q[0])
    try:
        for layer in range(w.layers):  # first use outside the capture
            cache.decode_step(layer, q[0], k[0], v[0], snn, sout, ws)
        graphs = []
        l0 = cache.kernel_launches()
        for j in range(n_distinct):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for layer in range(w.layers):
                    cache.decode_step(layer, q[j], k[j], v[j], snn, sout, ws)
            graphs.append(g)
        kernels_per_step = (cache.kernel_launches() - l0) // n_distinct
        dev_lens.copy_(lens0)
        stream = torch.cuda.current_stream()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(steps):
            if i > 0 and i % w.rollback_every == 0:
                dev_lens.copy_(lens0)
            graphs[i % n_distinct].replay()
        stop.record(stream)
        torch.cuda.synchronize()
        status = cache.device_status(ws)
    finally:
        cache.lens_from_device()
    ms = start.elapsed_time(stop)
    return {"ms": ms, "work": sum(w.work(i) for i in range(steps)), "status": status,
            "kernels_per_step": kernels_per_step}


def run_e2e(w: Workload, cache, steps: int, q, k, v):
    """The end-to-end leg: one layer a step through the library's host-buffer call, several layers
    (the step's inputs feed every layer) with the copies issued around the device-buffer call."""
    if w.layers == 1:
        return _e2e_host_call(w, cache, steps, q, k, v)
    return _e2e_copies_around_device_calls(w, cache, steps, q, k, v)


def _e2e_host_call(w: Workload, cache, steps: int, q, k, v):
    """Same steps through ``append_attention_host`` (the C ABI's host-buffer call).

    Each step's q, k_new and v_new start in page-locked host memory and its out ends there.  The
    library copies positions t < n_new[b] in and out on its own two copy streams through two device
    staging slots that alternate, so neighbouring steps' copies overlap the compute between them.
    The timed region ends when the last output has reached the host.  Afterwards the last step runs
    again through the device-buffer call from the lengths it started from, on the same inputs, and its
    output is compared bit for bit with what reached the host.
    """
    n_distinct = len(q)
    hq = [t.cpu().pin_memory() for t in q]
    hk = [t.cpu().pin_memory() for t in k]
    hv = [t.cpu().pin_memory() for t in v]
    hout = [torch.zeros(q[0].shape, dtype=q[0].dtype, pin_memory=True) for _ in range(2)]
    ws = cache.workspace(w.Hq, w.T)
    stream = torch.cuda.current_stream()
    cache.truncate(w.lens0)
    cache.append_attention_host(0, hq[0], hk[0], hv[0], w.n_new, hout[0], workspace=ws)  # staging set up
    cache.host_copies_done()
    cache.truncate(w.lens0)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        if i > 0 and i % w.rollback_every == 0:
            cache.truncate(w.lens0)
        j = i % n_distinct
        cache.append_attention_host(0, hq[j], hk[j], hv[j], w.n_new, hout[i % 2], workspace=ws)
    cache.host_copies_done()
    stop.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(stop)

    last = steps - 1
    matches = None
    if steps > 0:
        cache.truncate(w.lens_at(last) - w.n_new)
        j = last % n_distinct
        check = cache.append_attention(0, q[j], k[j], v[j], w.n_new, out=torch.empty_like(q[0]), workspace=ws)
        torch.cuda.synchronize()
        matches = bool(torch.equal(check.cpu(), hout[last % 2]))
    moved = int(np.sum(w.n_new)) * w.shape.d * q[0].element_size()  # positions t < n_new[b] only
    return {"ms": ms, "work": sum(w.work(i) for i in range(steps)), "h2d": moved * (w.Hq + 2 * w.shape.Hkv),
            "d2h": moved * w.Hq, "matches_device": matches,
            "path": "kvc_append_attention_host (host buffers; copies inside the library call)"}


def _e2e_copies_around_device_calls(w: Workload, cache, steps: int, q, k, v):
    """Same steps through the public API with the step's inputs in pinned host memory.

    Per step: one host->device copy of q, k_new and v_new (laid end to end in one pinned buffer, the
    three call arguments are views of its device copy); append + attention; device->host copy of out.
    Inputs move on one copy stream and outputs on another, with double-buffered device inputs and
    outputs, so step i+1's inputs and step i's output move, in opposite directions at once, while
    step i computes (every step still moves all its bytes; the timed region ends when the last output
    has reached the host).  Afterwards the last step runs again through the device-resident path from
    the same cache state, and its output is compared bit for bit with what reached the host.
    """
    n_distinct = len(q)
    args = (q[0], k[0], v[0])
    sizes = [t.numel() for t in args]
    offs = [0]
    for n in sizes:
        offs.append(offs[-1] + (n + 127) // 128 * 128)  # every view starts 256-byte aligned

    def packed(j):
        h = torch.empty(offs[-1], dtype=torch.bfloat16, pin_memory=True)
        for t, o, n in zip((q[j], k[j], v[j]), offs, sizes):
            h[o:o + n].copy_(t.reshape(-1))
        return h

    hin = [packed(j) for j in range(n_distinct)]
    din = [torch.empty(offs[-1], dtype=torch.bfloat16, device=q[0].device) for _ in range(2)]
    views = [[din[b][o:o + n].view(t.shape) for t, o, n in zip(args, offs, sizes)] for b in range(2)]
    out = [torch.empty_like(q[0]) for _ in range(2)]
    hout = [torch.empty(q[0].shape, dtype=q[0].dtype, pin_memory=True) for _ in range(2)]
    ws = cache.workspace(w.Hq, w.T)
    stream = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, computed, out_copied = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    cache.truncate(w.lens0)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    h2d.wait_stream(stream)
    d2h.wait_stream(stream)

    def load(i):  # step i's inputs into buffer i % 2 (on the input stream)
        b = i % 2
        with torch.cuda.stream(h2d):
            din[b].copy_(hin[i % n_distinct], non_blocking=True)
            in_ready[b].record(h2d)

    def compute(b, dst):
        qb, kb, vb = views[b]
        for layer in range(w.layers):
            cache.append_attention(layer, qb, kb, vb, w.n_new, out=dst, workspace=ws)

    load(0)
    for i in range(steps):
        b = i % 2
        if i > 0 and i % w.rollback_every == 0:
            cache.truncate(w.lens0)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_copied[b])  # out[b] of step i-2 has reached the host
        compute(b, out[b])
        computed[b].record(stream)
        if i + 1 < steps:
            if i >= 1:
                h2d.wait_event(computed[1 - b])  # step i-1 no longer reads buffer 1-b
            load(i + 1)
        with torch.cuda.stream(d2h):
            d2h.wait_event(computed[b])
            hout[b].copy_(out[b], non_blocking=True)
            out_copied[b].record(d2h)
    stream.wait_stream(d2h)
    stop.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(stop)

    # The last step once more from the lengths it started from, on its device-resident inputs.
    last = steps - 1
    if steps > 0:
        cache.truncate(w.lens_at(last) - w.n_new)
        check = torch.empty_like(q[0])
        compute(last % 2, check)
        torch.cuda.synchronize()
        matches = bool(torch.equal(check.cpu(), hout[last % 2]))
    else:
        matches = None
    work = sum(w.work(i) for i in range(steps))
    h2d_bytes = offs[-1] * 2  # the packed buffer as copied (alignment gaps included)
    return {"ms": ms, "work": work, "h2d": h2d_bytes, "d2h": q[0].numel() * 2, "matches_device": matches,
            "path": "device-buffer calls, torch copies from and to pinned host memory around them"}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------


def run_oracle_sample(w: Workload, budget_s: float = 12.0):
    """Time the float64 oracle on a bounded sample of the workload (one thread).

    Sample: one row of the batch (all its query heads) per oracle call, with
    that row's real length, repeated over rows until the time budget is spent.
    Returns (value in the metric's unit, sample description).
    """
    import oracle.ref as ref

    s = w.shape
    rng = np.random.default_rng(0)
    done_work, t_total, calls, rows = 0, 0.0, 0, 0
    b = 0
    while t_total < budget_s and rows < 4096:
        L = int(w.lens_at(0)[b])
        n = int(w.n_new[b])
        c = ref.OracleCache(1, 1, s.Hkv, L, s.d)
        c.k[0][:] = rng.standard_normal(c.k[0].shape)
        c.v[0][:] = rng.standard_normal(c.v[0].shape)
        c.lens[0] = [L]
        q = rng.standard_normal((1, w.Hq, w.T, s.d))
        t0 = time.perf_counter()
        ref.gqa_attention(q, c, 0, np.array([n]))
        t_total += time.perf_counter() - t0
        rows += 1
        calls += 1
        if w.unit == "TFLOP/s":
            done_work += 4 * s.d * w.Hq * visible_pairs([L - n], [n])
        else:
            done_work += L * s.Hkv * s.d * 2 * 2
        b = (b + 1) % s.B
    scale = 1e-12 if w.unit == "TFLOP/s" else 1e-9
    value = done_work * scale / t_total
    sample = (f"{rows} rows of the batch (all {w.Hq} query heads, real lengths), one oracle call each, "
              f"{t_total:.1f} s of CPU time on one thread; value = the rows' algorithmic "
              f"{'FLOPs' if w.unit == 'TFLOP/s' else 'KV bytes (bf16 sizes)'} / that time")
    return value, sample, t_total


# ---------------------------------------------------------------------------


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=["decode8b", "verify", "prefill", "longctx"], default="decode8b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--verify-t", type=int, choices=[4, 8, 16], default=4, help="drafts per row (verify workload)")
    ap.add_argument("--verify-g", type=int, choices=[1, 2, 4, 8, 16], default=4,
                    help="query heads per KV head, Hq = G * 8 (verify workload)")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="cache storage: bf16, or FP8 E4M3 with one scale per KV head")
    ap.add_argument("--prefill-ragged", action="store_true",
                    help="prefill workload: the ragged final chunk (n_new[b] uniform in 1..512) on the same priors")
    ap.add_argument("--head-dim", type=int, choices=[64, 128], default=128,
                    help="decode8b: head dimension of the cache (64: the same shape with 64-wide heads)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode8b: skip the chunked-prefill objects added to the line")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = Workload(args.workload, verify_t=args.verify_t, verify_g=args.verify_g, kv_dtype=args.kv_dtype,
                 prefill_ragged=args.prefill_ragged, head_dim=args.head_dim)
    # The headline metric has two halves (decode KV-read GB/s; chunked-prefill
    # attention TFLOP/s): the default decode run also measures both prefill
    # cases (the full chunk and the ragged final chunk) and reports them as
    # objects of the same line.
    extra = []
    if args.workload == "decode8b" and args.head_dim == 128 and not args.no_prefill:
        extra = [("prefill", Workload("prefill", kv_dtype=args.kv_dtype)),
                 ("prefill_ragged_final_chunk", Workload("prefill", kv_dtype=args.kv_dtype, prefill_ragged=True))]

    if args.impl == "reference":
        if rank != 0:
            return
        line = reference_line(w, args)
        for key, wx in extra:
            sub = reference_line(wx, args, cpu_budget_s=6.0)
            line[key] = {k: sub[k] for k in ("metric", "value", "unit", "config", "cpu_baseline", "e2e")}
        print(json.dumps(line))
        return

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)

    line = native_line(w, args, world, rank)
    for key, wx in extra:
        sub = native_line(wx, args, world, rank, cpu_budget_s=6.0)
        line[key] = {k: sub[k] for k in ("metric", "value", "unit", "ms_per_step", "config", "roofline", "e2e",
                                          "gpu_launches", "clocks", "device_status", "cpu_baseline") if k in sub}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def reference_line(w: Workload, args, cpu_budget_s: float = 12.0) -> dict:
    """The oracle arm: the float64 oracle timed on a bounded sample of w, on the host cores."""
    value, sample, _ = run_oracle_sample(w, cpu_budget_s)
    return {"metric": w.metric, "value": value, "unit": w.unit, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "impl": "reference", "dtype": "f64",
            "data": "synthetic", "config": w.config(),
            "cpu_baseline": {"value": value, "unit": w.unit, "cores": 1, "kind": "oracle", "sample": sample,
                             "host_cpus": os.cpu_count(), "blas_threads": 1},
            "e2e": {"value": value, "unit": w.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "vs_baseline": None}


def native_line(w: Workload, args, world: int, rank: int, cpu_budget_s: float = 12.0) -> dict:
    """One workload through the library: the bench line's fields for it."""
    scale = 1e-12 if w.unit == "TFLOP/s" else 1e-9
    res = run_native(w, args.steps, args.warmup, rank, world)
    graph_ms = res["graph"]["ms"] if "graph" in res else 0.0
    ms, e2e_ms, graph_ms = max_over_ranks([res["ms"], res["e2e"]["ms"], graph_ms], world, "cuda")
    value = whole_job_value(res["work"], world, ms, scale)
    e2e_value = whole_job_value(res["e2e"]["work"], world, e2e_ms, scale)
    if res["e2e"]["matches_device"] is False:
        print(f"bench: {w.config()['workload']}: the end-to-end leg's last output differs from the "
              "device-resident run of the same step", file=sys.stderr)

    hbm, bf16, bf16_sus, peak_kind = _peaks()
    attn_ms = float(res["attn_ms"])
    kb = float(np.mean(res["kernel_bytes"]))
    if w.unit == "TFLOP/s":
        flops = w.work(0)
        roof = {"bound": "tensor", "achieved": flops / (attn_ms * 1e-3) * 1e-12, "peak": bf16, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": kb / (attn_ms * 1e-3) * 1e-9, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    roof["kernel"] = w.kernel_name
    roof["kernel_ms"] = attn_ms
    roof["kernel_timing"] = res["kernel_timing"]
    roof["traffic"] = _committed_traffic(w, kb)

    line = {
        "metric": w.metric, "value": value, "unit": w.unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.kv_dtype == "bf16" else "fp8 storage, f16 MMA, fp32 accumulate",
        "data": "synthetic (seeded counter-based generator, ~N(0,1))",
        "config": dict(w.config(), parallelism="replicas only" if world > 1 else "single GPU"),
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": w.unit, "h2d_bytes_per_step": res["e2e"]["h2d"],
                "d2h_bytes_per_step": res["e2e"]["d2h"],
                "last_output_matches_device": res["e2e"]["matches_device"], "path": res["e2e"]["path"]},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "device_status": res["status"],
    }
    if w.unit == "GB/s":
        line["tokens_per_s"] = w.shape.B * args.steps * world / (ms * 1e-3)
        line["frac_of_hbm_peak"] = value / hbm
    else:
        line["frac_of_bf16_peak"] = value / bf16
    if "graph" in res:
        gr = res["graph"]
        line["graph_replay"] = {"value": whole_job_value(gr["work"], world, graph_ms, scale), "unit": w.unit,
                                "ms_per_step": graph_ms / args.steps, "kernels_per_step": gr["kernels_per_step"],
                                "note": "lengths resident on the device; one CUDA graph replay per step",
                                "device_status": gr["status"]}
    if rank == 0 and not args.no_cpu_baseline:
        cv, sample, _ = run_oracle_sample(w, cpu_budget_s)
        line["cpu_baseline"] = {"value": cv, "unit": w.unit, "cores": 1, "kind": "oracle", "sample": sample,
                                 "host_cpus": os.cpu_count(), "blas_threads": 1}
    return line


def max_over_ranks(times_ms, world: int, device) -> list:
    """Each timing's maximum over the ranks (the job is as slow as its slowest replica)."""
    if world <= 1:
        return [float(t) for t in times_ms]
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_value(work_per_rank: float, world: int, max_ms: float, scale: float) -> float:
    """Whole-job throughput: every rank's units (replicas do equal work) over the slowest rank's time."""
    return work_per_rank * world * scale / (max_ms * 1e-3)


def _committed_l2(w: Workload) -> str:
    """The back-to-back L2 measurement of this workload's kernel, if one was taken on the current source."""
    import hashlib

    path = os.path.join(ROOT, "profiles", f"l2_{w.name}.txt")
    if w.kv_dtype != "bf16" or w.shape.d != 128 or not os.path.exists(path):
        return ""
    kv = dict(line.strip().split("=", 1) for line in open(path) if "=" in line and not line.startswith("#"))
    src = os.path.join(ROOT, "gqa_attention_preallocated_gb300", "csrc", w.kernel_source)
    if kv.get("kernel_source_sha256_16") != hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]:
        return ""
    return (f"; measured on {kv['launches']} back-to-back launches without cache control: L2 hit rate "
            f"{kv['lts_hit_rate_pct']} %, DRAM bytes {kv['dram_over_algorithmic']}x the algorithmic bytes")


def _committed_traffic(w: Workload, mean_kernel_bytes: float):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source.

    The capture is one launch; its DRAM bytes are scaled to the average timed
    launch by the ratio of algorithmic bytes (traffic grows with the live K/V).
    """
    import hashlib

    tag = ("_ragged" if w.ragged else "") + ("_fp8" if w.kv_dtype == "fp8" else "") + \
        ("_d64" if w.shape.d == 64 else "")
    path = os.path.join(ROOT, "profiles", f"traffic_{w.name}{tag}.txt")
    if not os.path.exists(path):
        return None
    kv = dict(line.strip().split("=", 1) for line in open(path) if "=" in line and not line.startswith("#"))
    src = os.path.join(ROOT, "gqa_attention_preallocated_gb300", "csrc", w.kernel_source)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if kv.get("kernel_source_sha256_16") != sha:
        return None
    dram = float(kv["dram_bytes_per_launch"])
    alg = float(kv.get("algorithmic_bytes_of_captured_launch", 0) or 0)
    return dram * (mean_kernel_bytes / alg) if alg > 0 else dram


if __name__ == "__main__":
    main()
