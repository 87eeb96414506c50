"""Benchmark of the paged-attention hot path on GB300.

One step = one call of the operator (plan, cache write, prefill, split-KV decode, merge)
over one batch of seeded synthetic inputs already resident in HBM. The headline line is
the decode batch workload (64 sequences, one new token each, history uniform in
[512, 4096], 32 query / 8 KV heads, head_size 128, 256-token pages, fp16): decode KV
GB/s = the K and V history bytes the step must read (each element once) / step time.
The other workloads (causal prefill 4 x 2048 bf16, the mixed continuous batch, long
decode with 16-token pages) are measured in the same run under "secondary".

Timing: the step time comes from K whole steps, one call each, between CUDA events on
the launching stream; the dominant kernel's time from K more steps of the same program split
into calls around that kernel (the kernel bracketed by its own events: the self-planned
decode kernel of decode-only steps, the prefill kernel of prefill steps, the two attention
kernels that run side by side in a mixed step); e2e from at least 100 pipelined steps
through the Python API with pinned host buffers (wall clock).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
N > 1 runs under torchrun, one rank per GPU, each rank on its own batch (weak scaling,
no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

MAIN = 2
SECONDARY = (3, 4, 5)
METRIC = "paged-attn decode KV GB/s & prefill TFLOP/s vs GB300 peak; packed tokens/s"


# ---- algorithmic work of one step ---------------------------------------------------------

def kv_history_bytes(p) -> int:
    """K and V of every sequence's history (past + new rows), each element read once: two
    bytes per element for 16-bit caches, one per INT8 code, half a byte per INT4 code."""
    row = p.head_size * 2 if p.kv_quant is None else (p.head_size if p.kv_quant == "int8" else p.head_size // 2)
    return int(p.kv_lens.sum()) * p.kv_num_heads * row * 2


def step_bytes(p) -> int:
    """History K/V read + new K/V rows read and written + queries read + output written."""
    N, nh, kvh, hs = p.num_tokens, p.num_heads, p.kv_num_heads, p.head_size
    written = N if p.slot_mapping is None else int((p.slot_mapping >= 0).sum())
    return kv_history_bytes(p) + N * nh * hs * 2 * 2 + (N + written) * kvh * hs * 2 * 2


def causal_flops(p, sequences=None) -> int:
    """4 * head_size * num_heads * (query, key) pairs inside the causal mask (QK^T and PV)."""
    total = 0
    for b in (range(p.batch_size) if sequences is None else sequences):
        q, past = int(p.q_lens[b]), int(p.past_seqlens[b])
        total += q * past + q * (q + 1) // 2
    return 4 * p.head_size * p.num_heads * total


def decode_sequences(p):
    G = p.num_heads // p.kv_num_heads
    return [b for b in range(p.batch_size) if 1 <= p.q_lens[b] and p.q_lens[b] * G <= 16]


def prefill_sequences(p):
    d = set(decode_sequences(p))
    return [b for b in range(p.batch_size) if p.q_lens[b] > 0 and b not in d]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---- clocks during the timed region ---------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples of the timed region (the JSON line carries their summary)
        self.path = os.path.join(ROOT, "_build", f"clocks_gpu{gpu_index}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
                except ValueError:
                    pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2][1:]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ---- the CUDA arm ---------------------------------------------------------------------------------

class Runner:
    """Holds one workload resident on the GPU and enqueues steps through the C ABI with
    pre-marshalled arguments (so host overhead stays far below the GPU time of a step)."""

    def __init__(self, p, device):
        import torch

        import varlen_paged_kv_gb300 as pa
        self.torch, self.pa, self.p = torch, pa, p
        dt = {"fp16": torch.float16, "bf16": torch.bfloat16}[p.dtype]

        def t16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(dt)

        def t32(a):
            return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

        self.host = {k: getattr(p, k) for k in ("query", "key", "value")}
        self.q, self.k, self.v = t16(p.query), (None if p.key is None else t16(p.key)), (None if p.value is None else t16(p.value))
        if p.kv_quant is None:
            self.kc, self.vc = t16(p.key_cache), t16(p.value_cache)
            self.ext = None
        else:  # integer caches: code bytes, per-channel fp32 scales through pa_extensions
            self.kc = torch.from_numpy(np.ascontiguousarray(p.key_cache)).to(device)
            self.vc = torch.from_numpy(np.ascontiguousarray(p.value_cache)).to(device)
            self.k_scale = torch.from_numpy(np.ascontiguousarray(p.k_scale, dtype=np.float32)).to(device)
            self.v_scale = torch.from_numpy(np.ascontiguousarray(p.v_scale, dtype=np.float32)).to(device)
            self.ext = pa.PaExtensions(None, None, None, self.k_scale.data_ptr(), self.v_scale.data_ptr())
        self.cum, self.past = t32(p.cumulative_sequence_length), t32(p.past_seqlens)
        self.bt, self.sm = t32(p.block_table), t32(p.slot_mapping)
        self.out = torch.empty((p.num_tokens, p.num_heads * p.head_size), dtype=dt, device=device)
        # the caller knows its batch composition: pass the bound on new tokens per sequence
        self.max_q = int(p.q_lens.max()) if p.batch_size else 0
        self.dims = pa.make_dims(p.num_tokens, p.batch_size, p.head_size, p.num_blocks, p.block_size,
                                 p.max_blocks_per_sequence, dt, max_query_len=self.max_q, kv_dtype=p.kv_quant)
        self.ws = torch.zeros(pa.workspace_size(self.dims, p.num_heads, p.kv_num_heads), dtype=torch.uint8,
                              device=device)
        self.stream = torch.cuda.current_stream(device)
        self.lib = pa.load_library()
        vp = ctypes.c_void_p

        def ptr(t):
            return None if t is None else vp(t.data_ptr())

        self.args = (ptr(self.q), ptr(self.k), ptr(self.v), ptr(self.kc), ptr(self.vc), ptr(self.cum),
                     ptr(self.past), ptr(self.bt), ptr(self.sm), p.num_heads, p.kv_num_heads,
                     ctypes.c_float(p.scale), ptr(self.out), ctypes.byref(self.dims), ptr(self.ws),
                     self.ws.numel(), vp(self.stream.cuda_stream))

    def call(self, stages):
        if stages == 0:
            return
        if self.ext is not None:  # (integer caches: pa_paged_attention_ex, its stages field)
            self.ext.stages = stages
            a = self.args
            st = self.lib.pa_paged_attention_ex(*a[:13], ctypes.byref(self.ext), *a[13:])
        else:
            st = self.lib.pa_paged_attention_stages(*self.args, stages)
        if st:
            raise RuntimeError(f"pa_paged_attention: status {st}")

    def step(self):
        self.call(self.pa.STAGE_ALL)

    def timed(self, steps, warmup, kernel_stages, clocks=None):
        """Times `steps` steps of the whole call's program, each split into three calls: the
        stages before `kernel_stages`, those stages (bracketed by their own events), the
        stages after. Returns (seconds per step, seconds per bracketed launch, launches)."""
        torch, pa = self.torch, self.pa
        stages = (pa.STAGE_PLAN, pa.STAGE_CACHE_WRITE, pa.STAGE_PREFILL, pa.STAGE_DECODE)
        low = kernel_stages & -kernel_stages
        mask_before = sum(s for s in stages if s < low)
        mask_after = sum(s for s in stages if s > kernel_stages)
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = pa.kernel_launch_count()
        if clocks is not None:
            clocks.__enter__()
        torch.cuda.synchronize()
        start.record(self.stream)
        for i in range(steps):
            self.call(mask_before)
            ev[i][0].record(self.stream)
            self.call(kernel_stages)
            ev[i][1].record(self.stream)
            self.call(mask_after)
        end.record(self.stream)
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.__exit__(None, None, None)
        launches = pa.kernel_launch_count() - n0
        total = start.elapsed_time(end) / 1e3
        kern = sum(a.elapsed_time(b) for a, b in ev) / 1e3 / steps
        return total / steps, kern, launches

    def whole(self, steps, warmup, clocks=None):
        """Times `steps` whole steps, one call each (how a caller runs the operator).
        Returns (seconds per step, launches per step)."""
        torch, pa = self.torch, self.pa
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = pa.kernel_launch_count()
        if clocks is not None:
            clocks.__enter__()
        torch.cuda.synchronize()
        start.record(self.stream)
        for _ in range(steps):
            self.step()
        end.record(self.stream)
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.__exit__(None, None, None)
        launches = pa.kernel_launch_count() - n0
        return start.elapsed_time(end) / 1e3 / steps, launches / steps

    def e2e(self, steps, warmup):
        """The public Python API with host buffers: per step, H2D of the step's inputs from
        pinned memory, the call, D2H of the output; the caches stay resident. Steps are
        pipelined as a serving loop runs them: the inputs of step i+1 travel on one copy
        stream and the output of step i on another while step i+1 computes (two sets of
        device input and output buffers), so every step's copies are inside the timed region
        but overlap other steps' compute."""
        torch, pa = self.torch, self.pa
        p = self.p
        names = ("query", "key", "value", "cum", "past", "bt", "sm")
        devs = dict(zip(names, (self.q, self.k, self.v, self.cum, self.past, self.bt, self.sm)))
        pins = {n: torch.empty(d.shape, dtype=d.dtype, pin_memory=True) for n, d in devs.items() if d is not None}
        for n, h in pins.items():
            h.copy_(devs[n].cpu())
        # two sets of device inputs and outputs (set 0 is the runner's own tensors)
        sets = [dict(devs), {n: (torch.empty_like(d) if d is not None else None) for n, d in devs.items()}]
        outs = [self.out, torch.empty_like(self.out)]
        out_host = [torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True) for _ in range(2)]
        h2d = sum(h.numel() * h.element_size() for h in pins.values())
        d2h = out_host[0].numel() * out_host[0].element_size()
        comp = torch.cuda.current_stream()
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ready = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        drained = [torch.cuda.Event() for _ in range(2)]

        def one(i):
            k = i & 1
            d = sets[k]
            with torch.cuda.stream(up):
                up.wait_event(computed[k])  # step i-2 has finished reading this set
                for n, h in pins.items():
                    d[n].copy_(h, non_blocking=True)
                ready[k].record(up)
            comp.wait_event(ready[k])
            comp.wait_event(drained[k])  # step i-2's output has left this buffer
            quant = {} if p.kv_quant is None else dict(kv_quant=p.kv_quant, k_scale=self.k_scale,
                                                          v_scale=self.v_scale)
            pa.paged_attention(d["query"], d["key"], d["value"], self.kc, self.vc, d["cum"], d["past"], d["bt"],
                               d["sm"], num_heads=p.num_heads, kv_num_heads=p.kv_num_heads, scale=p.scale,
                               output=outs[k], workspace=self.ws, max_query_len=self.max_q, **quant)
            computed[k].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[k])
                out_host[k].copy_(outs[k], non_blocking=True)
                drained[k].record(down)

        for i in range(warmup):
            one(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            one(i)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / steps, h2d, d2h


# DRAM bytes (read + write) of one launch of the dominant kernel, from one ncu capture
# (profiles/<kernel>_<workload>.md), with a hash of the kernel's sources at capture time:
# the figure is reported only while the sources are unchanged, else traffic is null.
# ("decode_kernel_self": the self-planned instantiation that decode-only steps run.)
NCU_TRAFFIC = {
    ("decode_kernel_self", "decode-b64"): (618575104 + 3658496, "a13d94cc23457e5b"),
    ("decode_kernel_self", "long-decode-b8-bs16"): (2279131904 + 3412736, "a13d94cc23457e5b"),
    ("decode_kernel_self", "decode-b64-int8"): (310088704 + 3812864, "a13d94cc23457e5b"),
    ("decode_kernel_self", "decode-b64-int4"): (155679744 + 3673856, "a13d94cc23457e5b"),
    ("decode_kernel_self", "decode-b64-hs256"): (295574784 + 4252672, "a13d94cc23457e5b"),
    ("prefill_kernel", "causal-prefill-4x2048"): (104446976 + 31610368, "438918628f0afde7"),
    ("prefill256_kernel", "causal-prefill-hs256"): (84022784 + 25982208, "b4b200812dc0f5a1"),
    # the two attention kernels of a mixed step (prefill 188.8 + 15.5 MB, decode 775.7 + 0.3 MB;
    # on INT8 caches prefill 101.0 + 8.7 MB, decode 388.2 + 0.5 MB)
    ("prefill_kernel+decode_kernel", "mixed-8x512-chunks+24-decode"): (188848640 + 15481600 + 775743232 + 322048,
                                                                        "c3f863d2415e1ed3"),
    ("prefill_kernel+decode_kernel", "mixed-8x512-chunks+24-decode-int8"): (100956672 + 8674816 + 388170240 + 463104,
                                                                             "c3f863d2415e1ed3"),
}
KERNEL_SOURCES = {"decode_kernel": ("decode.cu", "common.cuh"), "decode_kernel_self": ("decode.cu", "common.cuh"),
                  "prefill_kernel": ("prefill.cu", "common.cuh"), "prefill256_kernel": ("prefill256.cu", "common.cuh"),
                  "prefill_kernel+decode_kernel": ("prefill.cu", "decode.cu", "common.cuh")}


def source_hash(kernel):
    """Hash of the kernel's sources, line comments and trailing blanks aside (a comment edit
    does not change the kernel the counters were taken from)."""
    m = hashlib.sha1()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "varlen_paged_kv_gb300", "csrc", f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    m.update(code.encode() + b"\n")
    return m.hexdigest()[:16]


def ncu_traffic(kernel, name):
    entry = NCU_TRAFFIC.get((kernel, name))
    if entry is None or source_hash(kernel) != entry[1]:
        return None
    return entry[0]


def kernel_roofline(p, kind, seconds_per_launch, pk, kernel):
    if kind == "hbm":
        units = kv_history_bytes(p)
        achieved = units / seconds_per_launch / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": ncu_traffic(kernel, p.name),
                "peak_source": f"{pk['source']} hbm_gbs", "algorithmic_bytes_per_launch": units}
    flops = causal_flops(p, prefill_sequences(p))
    achieved = flops / seconds_per_launch / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(achieved / pk["bf16_tflops"], 4), "traffic": ncu_traffic(kernel, p.name),
            "peak_source": f"{pk['source']} bf16_tflops (burst; fp16 nominal rate equals bf16)",
            "algorithmic_flops_per_launch": flops}


def reduce_over_ranks(local_seconds: float, local_units: float):
    """max step time and summed units over ranks (identity when not distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_seconds, local_units
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def oracle_baseline(p, budget_s=10.0, max_reps=200):
    """The oracle on the whole workload, repeated until about budget_s seconds of host work
    (at most max_reps runs). Returns (seconds per run, runs, threads)."""
    import oracle
    oracle.build()
    reps = 0
    t0 = time.perf_counter()
    while reps < max_reps and (reps == 0 or time.perf_counter() - t0 < budget_s):
        oracle.paged_attention(p)
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return dt, reps, oracle.max_threads()


WORKLOAD_TEXT = {
    2: "decode batch: B=64, 1 new token each, past U[512,4096], 32/8 heads, head_size 128, 256-token pages, "
       "fp16, separate K/V, slots derived",
    3: "causal prefill: B=4 x 2048 new tokens, past 0, 32/8 heads, head_size 128, 256-token pages, bf16",
    4: "mixed continuous batch: 8 prefill chunks of 512 (past U[0,8192]) + 24 decode tokens (past "
       "U[1024,16384]), 32/8 heads, head_size 128, 256-token pages, fp16, packed [Q|K|V], 10% slots -1",
    5: "long-context decode: B=8, 1 new token each, past U[32768,131072], 32/8 heads, head_size 128, "
       "16-token pages, bf16",
    "causal-prefill-explicit-slots": "causal prefill: B=4 x 2048 new tokens, past 0, 32/8 heads, head_size 128, "
                                     "256-token pages, bf16, explicit slot_mapping (the fp16 V copy kernel runs)",
    "causal-prefill-hs256": "causal prefill: B=4 x 2048 new tokens, past 0, 16/2 heads, head_size 256, "
                            "256-token pages, bf16",
    "decode-b64-hs256": "decode batch: B=64, 1 new token each, past U[512,4096], 16/2 heads, head_size 256, "
                        "256-token pages, fp16, slots derived",
}


def quant_text(k, fmt):
    return WORKLOAD_TEXT[k].replace(", fp16,", ", fp16 queries, %s per-channel KV caches," % fmt)


def load_workload(k, kv_quant=None):
    """(problem, key) of a workload number (2..5), a variant name, or k with integer caches."""
    if k in wl.VARIANTS:
        return wl.variant(k), k
    k = int(k)
    return (wl.config_kv_quant(k, kv_quant) if kv_quant else wl.config(k)), k


def measure(r, steps, warmup, pk, clocks=None):
    """Times one workload: whole steps (one call each) for the step time, then the same
    steps split around the dominant kernel (prefill for workloads with prefill rows, else
    decode), which is bracketed by its own events. Returns (seconds per step, roofline,
    kernel launches in the whole-step timed region)."""
    q = r.p
    sec, per_step = r.whole(steps, warmup, clocks=clocks)
    pa = r.pa
    if prefill_sequences(q) and decode_sequences(q):
        # a mixed step runs its two attention kernels side by side on split SMs: time the pair
        _, kt, _ = r.timed(steps, warmup, pa.STAGE_PREFILL | pa.STAGE_DECODE)
        roof = kernel_roofline(q, "tensor", kt, pk, "prefill_kernel+decode_kernel")
        roof["kernel"] = ("prefill_kernel (tcgen05/TMEM, TMA) beside decode_kernel (split-KV) on split SMs; "
                          "achieved = the prefill rows' causal FLOPs / the pair's time")
    elif prefill_sequences(q):
        _, kt, _ = r.timed(steps, warmup, pa.STAGE_PREFILL)
        name = "prefill256_kernel" if q.head_size == 256 else "prefill_kernel"
        roof = kernel_roofline(q, "tensor", kt, pk, name)
        roof["kernel"] = name + " (tcgen05/TMEM, TMA)"
    else:
        # decode-only with the host bound: the decode kernel the whole step runs (self-planned
        # up to 256 sequences, 64 at head_size 256)
        _, kt, _ = r.timed(steps, warmup, pa.STAGE_DECODE)
        self_planned = q.batch_size <= (64 if q.head_size == 256 else 256)
        roof = kernel_roofline(q, "hbm", kt, pk, "decode_kernel_self" if self_planned else "decode_kernel")
        roof["kernel"] = ("decode_kernel (%ssplit-KV, TMA + mma.sync%s)"
                          % ("self-planned, " if self_planned else "",
                             "" if q.kv_quant is None else ", on %s codes" % q.kv_quant))
    roof["ms_per_launch"] = round(kt * 1e3, 4)
    # The bracketing events serialise the bracketed launches with the rest of the stream; in
    # back-to-back steps a kernel's prologue overlaps its predecessor (programmatic dependent
    # launch), so a launch can take longer than the step period. The rate over the whole step:
    units = roof.get("algorithmic_bytes_per_launch") or roof.get("algorithmic_flops_per_launch")
    roof["achieved_over_step"] = round(units / sec / (1e9 if roof["bound"] == "hbm" else 1e12), 1)
    return sec, roof, per_step * steps


def headline(q, sec):
    """(value, unit) of a workload's own metric: decode KV GB/s for decode-only batches,
    causal TFLOP/s for prefill-only batches, packed tokens/s for mixed ones."""
    if not prefill_sequences(q):
        return kv_history_bytes(q) / sec / 1e9, "GB/s"
    if not decode_sequences(q):
        return causal_flops(q) / sec / 1e12, "TFLOP/s"
    return q.num_tokens / sec, "tokens/s"


def run_cuda(args):
    import torch
    import torch.distributed as dist
    from varlen_paged_kv_gb300 import build as _build
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    pk = peaks()

    if rank == 0 or args.kv_quant or args.workload in wl.VARIANTS:
        p, k = load_workload(args.workload, args.kv_quant)
    else:
        k = int(args.workload)
        p = wl.make_problem(**_rank_recipe(k, rank))
    r = Runner(p, device)
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sec, roof, launches = measure(r, args.steps, args.warmup, pk, clocks=sampler)
    value, unit = headline(p, sec)
    sec_max, value_all = reduce_over_ranks(sec, value * sec)   # units of work summed over ranks
    value = value_all / sec_max
    e2e_sec, h2d, d2h = r.e2e(max(args.steps // 4, 100), args.warmup)
    e2e_max, e2e_units = reduce_over_ranks(e2e_sec, headline(p, e2e_sec)[0] * e2e_sec)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec_max * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": p.dtype, "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[k] if not args.kv_quant else quant_text(k, args.kv_quant),
                   "name": p.name, "num_tokens": p.num_tokens,
                   "batch_size": p.batch_size, "num_blocks": p.num_blocks,
                   "kv_history_bytes_per_step": kv_history_bytes(p),
                   "causal_flops_per_step": causal_flops(p),
                   "l2": ("inputs larger than L2: each step streams %.0f MB of K/V history (L2 129 MB)"
                          % (kv_history_bytes(p) / 1e6)) if k != 3 else
                         "compute-bound workload; its %.0f MB of K/V fit in L2" % (kv_history_bytes(p) / 1e6),
                   "parallelism": f"replicas x{world} (one batch per GPU)"},
        "roofline": roof,
        "e2e": {"value": round(e2e_units / e2e_max, 1), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_max * 1e3, 4)},
        "gpu_launches": int(launches),
        "clocks": sampler.summary(),
    }
    if rank == 0 and not args.no_secondary and not args.kv_quant:
        sec_lines = {}
        for kk in SECONDARY:
            if kk == k:
                continue
            q = wl.config(kk)
            rq = Runner(q, device)
            s, roof_q, _ = measure(rq, max(args.steps // 10, 10), args.warmup, pk)
            v, u = headline(q, s)
            entry = {"workload": WORKLOAD_TEXT[kk], "value": round(v, 1), "unit": u, "ms_per_step": round(s * 1e3, 4),
                     "packed_tokens_per_s": round(q.num_tokens / s, 1), "roofline": roof_q}
            if kk == 4:
                t_flop = causal_flops(q) / (pk["bf16_tflops"] * 1e12)
                t_byte = step_bytes(q) / (pk["hbm_gbs"] * 1e9)
                entry["fraction_of_max_roofline_time"] = round(max(t_flop, t_byte) / s, 4)
            sec_lines[q.name] = entry
            del rq
            torch.cuda.empty_cache()
        for fmt in ("int8", "int4"):
            q = wl.config_kv_quant(MAIN, fmt)
            rq = Runner(q, device)
            s, roof_q, _ = measure(rq, max(args.steps // 10, 10), args.warmup, pk)
            v, u = headline(q, s)
            fp16 = wl.config(MAIN)
            sec_lines[q.name] = {
                "workload": quant_text(MAIN, fmt),
                "value": round(v, 1), "unit": u + " (code bytes)", "ms_per_step": round(s * 1e3, 4),
                "fp16_equivalent_kv_gb_s": round(kv_history_bytes(fp16) / s / 1e9, 1),
                "speedup_vs_fp16_step": round(sec / s, 3) if k == MAIN else None,
                "roofline": roof_q}
            del rq
            torch.cuda.empty_cache()
        # the mixed batch on INT8 caches (its prefill rows on the prefill kernel's code-tile
        # path) and the 256-wide heads of both kernels
        for key in ("int8-mixed", "causal-prefill-hs256", "decode-b64-hs256"):
            q = wl.config_kv_quant(4, "int8") if key == "int8-mixed" else wl.variant(key)
            rq = Runner(q, device)
            s, roof_q, _ = measure(rq, max(args.steps // 10, 10), args.warmup, pk)
            v, u = headline(q, s)
            sec_lines[q.name] = {"workload": quant_text(4, "int8") if key == "int8-mixed" else WORKLOAD_TEXT[key],
                                 "value": round(v, 1), "unit": u, "ms_per_step": round(s * 1e3, 4),
                                 "packed_tokens_per_s": round(q.num_tokens / s, 1), "roofline": roof_q}
            del rq
            torch.cuda.empty_cache()
        line["secondary"] = sec_lines
    if rank == 0 and args.no_cpu_baseline:
        line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    elif rank == 0:
        dt, reps, cores = oracle_baseline(p)
        cv, cu = headline(p, dt)
        line["cpu_baseline"] = {"value": round(cv, 4), "unit": cu, "cores": cores, "kind": "oracle",
                                "sample": "the whole %s workload (cache write + attention), fp64 C oracle, %d runs "
                                          "of %.3f s each" % (p.name, reps, dt)}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def _rank_recipe(k, rank):
    """Rank r > 0 runs its own batch of the same workload recipe (seed shifted by 100 r)."""
    seed = 1000 + k + 100 * rank
    if k == 2:
        past = wl.uniform_int(seed, wl.S_PAST, 64, 512, 4096)
        return dict(name=wl.CONFIG_NAMES[2], seed=seed, dtype="fp16", num_heads=32, kv_num_heads=8, head_size=128,
                    block_size=256, past=past, q_lens=np.ones(64, np.int64), max_blocks_per_sequence=17)
    if k == 3:
        return dict(name=wl.CONFIG_NAMES[3], seed=seed, dtype="bf16", num_heads=32, kv_num_heads=8, head_size=128,
                    block_size=256, past=np.zeros(4, np.int64), q_lens=np.full(4, 2048, np.int64))
    raise ValueError("multi-GPU runs use workload 2 or 3")


def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is the whole workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    p, key = load_workload(args.workload, args.kv_quant)
    for _ in range(args.warmup):
        oracle.paged_attention(p)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_attention(p)
    sec = (time.perf_counter() - t0) / args.steps
    value, unit = headline(p, sec)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[key] if not args.kv_quant else quant_text(key, args.kv_quant),
                   "name": p.name},
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": "the whole %s workload per step (cache write + attention)" % p.name},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--workload", default=str(MAIN), choices=["2", "3", "4", "5", *wl.VARIANTS],
                    help="workload of the headline line (2: the decode batch the metric is quoted on; the "
                         "variants serve profiling runs)")
    ap.add_argument("--kv-quant", choices=["int8", "int4"], default=None,
                    help="the workload with integer KV caches (workloads 2 and 4; profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if args.steps > 50:
            args.steps = 10
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
