"""Benchmark: causal varlen prefill attention throughput on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the whole hot path over one batch of the workload: the
device scheduler plus the attention/cache-write kernel, for every launch the
workload has (long32k: one 32768-token prompt, one launch; chunked_decode: 16
launches of a 512-token chunk packed with 64 decode rows).  Inputs are seeded
synthetic N(0,1) bf16 tensors, resident in HBM before timing; q/k/v of the
default workload (805 MB) exceed the 129 MB L2, so no flush is needed between
steps.  The metric is causal-attention TFLOP/s (4 * head_dim * n_heads per
visible (query, key) pair) -- the masked upper triangle is not counted.

For N > 1 (torchrun, one process per GPU) every rank runs its own replica of
the workload: the units of attention are independent, no collective is on
the data path (weak scaling).  Timing is max over ranks.

The line's roofline fraction divides by the measured burst bf16 peak when the
timed region is shorter than 3 s (the sustained, power-capped figure from 3 s
on); the fractions against the other references are reported beside it.  The
default run (long32k) also carries a "per_config" block: the other measured
configurations (tiny_packed, layer512, varlen16, chunked_decode) and
chunked_decode's two parts alone (chunk512: its 512-token chunk over a
4096-token prefix; decode64: its 64 decode rows), each with its time per step,
TFLOP/s, fraction of the burst peak and of its mixed tensor/HBM roofline.

--impl reference times the fp64 CPU oracle on this host's cores on a bounded
sample of the same workload (the baseline this library is compared with).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal varlen prefill attention TFLOP/s and tokens/s; % of GB300 BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129e6  # GB300 L2


# --------------------------------------------------------------------- utils --

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha256() -> str:
    """Hash of the attention kernel's code (ties stored ncu counters to a kernel
    version): its sources with comments and blank lines removed, so that an
    edit of a comment does not orphan the counters of an unchanged kernel."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("attn_fwd.cu", "ptx.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "prefill_phase_attention_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)      # block comments
        src = re.sub(r"//[^\n]*", "", src)                    # line comments (no '//' in the strings here)
        lines = [ln.rstrip() for ln in src.splitlines()]
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
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
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_step_per_rank: float, ms_total_max: float, steps: int, ws: int) -> float:
    """Whole-job TFLOP/s: every rank processed its own copy of the step's units."""
    return ws * flops_per_step_per_rank * steps / (ms_total_max * 1e-3) / 1e12


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ oracle timing --

def oracle_sample_rows(wl, step, target_rows: int, seed: int):
    """A bounded sample of query rows (t*H + h) spread uniformly over tokens and heads."""
    rng = np.random.default_rng(seed)
    T = step.total_q
    n = min(target_rows, T * wl.n_heads)
    return np.sort(rng.choice(T * wl.n_heads, size=n, replace=False)).astype(np.int64)


def row_flops(wl, step, rows, window=0):
    """Causal FLOPs of the selected rows (4 * d per visible key)."""
    cu = np.array(step.cu_seqlens_q())
    off = np.array(step.cache_offsets)
    t = rows // wl.n_heads
    b = np.searchsorted(cu, t, side="right") - 1
    i = t - cu[b]
    n_b = cu[b + 1] - cu[b]
    vis = off[b] + (i + 1 if wl.causal else n_b)
    if window > 0:
        vis = np.minimum(vis, window)
    return int(4 * wl.head_dim * vis.sum())


def time_oracle(wl, inputs, rows, threads, window=0, rope=0.0):
    import oracle
    from prefill_phase_attention_gb300 import workloads as W
    cache_k, cache_v, steps = inputs
    inp = steps[-1]
    ck, cv = W.bf16_bits(cache_k), W.bf16_bits(cache_v)
    t0 = time.perf_counter()
    oracle.prefill_attention(W.bf16_bits(inp["q"]), W.bf16_bits(inp["k"]), W.bf16_bits(inp["v"]),
                             inp["cu_seqlens_q"].numpy(), inp["cu_seqlens_k"].numpy(),
                             inp["cache_offsets"].numpy(), ck, cv, n_heads=wl.n_heads,
                             n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim, max_cache_len=wl.max_cache_len,
                             scale=wl.scale, causal=wl.causal, window=window, rope_theta=rope, rows=rows,
                             want_cache=False,
                             threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(wl, inputs, budget_s: float = 15.0, window: int = 0, rope: float = 0.0):
    """The oracle on this host's cores over a sample sized to about `budget_s` seconds."""
    import oracle
    oracle.build()
    cores = host_cores()
    step = wl.steps[-1]
    time_oracle(wl, inputs, oracle_sample_rows(wl, step, 64, seed=10), cores, window, rope)  # threads, page faults
    cal = oracle_sample_rows(wl, step, 512, seed=11)
    dt = time_oracle(wl, inputs, cal, cores, window, rope)
    rate = row_flops(wl, step, cal, window) / max(dt, 1e-6)  # FLOP/s of the oracle on this host
    per_row = row_flops(wl, step, cal, window) / cal.size
    n = int(rate * budget_s / max(per_row, 1.0))
    rows = oracle_sample_rows(wl, step, max(512, n), seed=12)
    dt = time_oracle(wl, inputs, rows, cores, window, rope)
    fl = row_flops(wl, step, rows, window)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows.size} query rows (token, head) drawn uniformly from {wl.name} "
                      f"(launch {len(wl.steps) - 1}), {fl / 1e9:.1f} GFLOP causal, {dt:.1f} s, fp64 C + OpenMP",
            "seconds": round(dt, 2)}


# ----------------------------------------------------------------- our arm --

DATASHEET_BF16_TFLOPS = 2250.0  # GB300 dense bf16, NVIDIA's figure without 2:4 sparsity
SUSTAINED_AFTER_S = 3.0         # timed regions at least this long are compared with the sustained peak


class Runner:
    """A workload's inputs resident on the device and the call that runs one step."""

    def __init__(self, wl, args, binding, W):
        import torch
        self.wl, self.args, self.binding = wl, args, binding
        self.inputs = W.make_inputs(wl, sentinel=False)
        cache_k, cache_v, steps = self.inputs
        self.table_d = self.sk_d = self.sv_d = None
        if args.kv_quant and args.paged:
            # int8 codes + fp32 row scales in block pools
            table, codes_k, scales_k, codes_v, scales_v = W.make_paged_q8_cache(
                wl, args.paged, torch.Generator().manual_seed(wl.seed), sentinel=False)
            self.ck, self.sk_d, self.cv, self.sv_d = codes_k.cuda(), scales_k.cuda(), codes_v.cuda(), scales_v.cuda()
            self.table_d = table.cuda()
        elif args.kv_quant:
            # the same workload over an int8 cache (codes + fp32 row scales)
            codes_k, scales_k, codes_v, scales_v = W.make_q8_cache(wl, torch.Generator().manual_seed(wl.seed),
                                                                   sentinel=False)
            self.ck, self.sk_d, self.cv, self.sv_d = codes_k.cuda(), scales_k.cuda(), codes_v.cuda(), scales_v.cuda()
        elif args.paged:
            # the same workload over a paged cache: a block pool + per-sequence block table
            table, pool_k, pool_v = W.make_paged_cache(wl, args.paged, torch.Generator().manual_seed(wl.seed),
                                                       sentinel=False)
            self.ck, self.cv, self.table_d = pool_k.cuda(), pool_v.cuda(), table.cuda()
        else:
            self.ck, self.cv = cache_k.cuda(), cache_v.cuda()
        self.dev = [{k: v.cuda() for k, v in s.items()} for s in steps]
        self.outs = [torch.empty_like(d["q"]) for d in self.dev]
        self.lses = [torch.empty(d["q"].shape[0], wl.n_heads, device="cuda", dtype=torch.float32) for d in self.dev]
        self.schedules = set()  # the work schedule each call of a step ran (pa_options.schedule)

    def call(self, d, o, l):
        a, b = self.args, self.binding
        if a.window or a.paged or a.rope or a.kv_quant:
            b.prefill_attn_varlen_ex(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], self.ck, self.cv,
                                     d["cache_offsets"], o, l, scale=self.wl.scale, causal=self.wl.causal,
                                     window=a.window, block_table=self.table_d, rope_theta=a.rope,
                                     cache_k_scale=self.sk_d, cache_v_scale=self.sv_d)
        else:
            b.prefill_attn_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], self.ck, self.cv,
                                  d["cache_offsets"], o, l, scale=self.wl.scale, causal=self.wl.causal)

    def step(self):
        for d, o, l in zip(self.dev, self.outs, self.lses):
            self.call(d, o, l)

    def warm(self, warmup):
        import torch
        for d, o, l in zip(self.dev, self.outs, self.lses):
            self.call(d, o, l)
            self.schedules.add(self.binding.prefill_attn_last_schedule())
        for _ in range(warmup - 1):
            self.step()
        torch.cuda.synchronize()
        if self.binding.prefill_attn_device_status() != 0:
            raise RuntimeError(f"device error word set during warm-up of {self.wl.name}")

    def working_set_bytes(self):
        wl = self.wl
        return wl.tokens() * (wl.n_heads + 2 * wl.n_kv_heads) * wl.head_dim * 2

    def schedule(self):
        s = sorted(self.schedules)
        return s[0] if len(s) == 1 else s


def measure(runner, steps, ws=1, local=0, sampler=None):
    """K timed steps with CUDA events on the launching stream.  A working set
    larger than L2 runs back to back (the region between the first and the last
    event); a smaller one is timed cold: a 256 MB buffer is written before
    every step, outside the step's span, and the spans are summed."""
    import torch
    stream = torch.cuda.current_stream()
    flush = None
    if runner.working_set_bytes() <= L2_BYTES:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    hot_ms_step = None
    if flush is not None:  # the same steps back to back with a warm L2, for reference
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            runner.step()
        e1.record(stream)
        torch.cuda.synchronize()
        hot_ms_step = e0.elapsed_time(e1) / steps
    n_launch = len(runner.dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps * n_launch)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)
    launches = 0
    barrier(ws)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    e_start.record(stream)
    k = 0
    for si in range(steps):
        if flush is not None:
            flush.fill_(si & 0xFF)  # evict L2 (not inside the step's timed span)
        step_ev[si][0].record(stream)
        for d, o, l in zip(runner.dev, runner.outs, runner.lses):
            ev[k][0].record(stream)
            runner.call(d, o, l)
            ev[k][1].record(stream)
            launches += runner.binding.prefill_attn_last_launch_count()
            k += 1
        step_ev[si][1].record(stream)
    e_end.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(ws)
    clocks = sampler.stop() if sampler is not None else None
    ms_total = sum(a.elapsed_time(b) for a, b in step_ev) if flush is not None else e_start.elapsed_time(e_end)
    ms_total = max_over_ranks(ms_total, ws, device=torch.device("cuda", local))
    if runner.binding.prefill_attn_device_status() != 0:
        raise RuntimeError(f"device error word set during the timed region of {runner.wl.name}")
    per_call_ms = [a.elapsed_time(b) for a, b in ev]
    return {"ms_total": ms_total, "ms_step": ms_total / steps, "per_call_ms": per_call_ms, "launches": launches,
            "cold_l2": flush is not None, "hot_ms_step": hot_ms_step, "clocks": clocks,
            "region_s": ms_total * 1e-3 if flush is not None else t_wall}


def graph_ms_step(runner, steps):
    """The step captured once into a CUDA graph (on a stream of its own, after an
    uncaptured step sized that stream's workspace) and replayed `steps` times
    back to back: the step's device time with no host time between launches
    (warm L2), as a serving loop that replays captured steps sees it."""
    import torch
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        runner.step()
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        runner.step()
    for _ in range(10):  # the first replays of a new graph run slower
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(steps):
            g.replay()
        e1.record(st)
    torch.cuda.synchronize()
    if runner.binding.prefill_attn_device_status() != 0:
        raise RuntimeError(f"device error word set during the graph replays of {runner.wl.name}")
    del g
    return e0.elapsed_time(e1) / steps


def algorithmic_bytes(wl, kv_quant=False):
    """q, k, v read; out, lse and the new cache rows written; the cached prefix read once."""
    kv_row = wl.n_kv_heads * wl.head_dim * (1 if kv_quant else 2) + (4 * wl.n_kv_heads if kv_quant else 0)
    return sum(st.total_q * (2 * wl.n_heads + 2 * wl.n_kv_heads) * wl.head_dim * 2 + 4 * st.total_q * wl.n_heads
               + 2 * st.total_q * kv_row + 2 * kv_row * sum(st.cache_offsets) for st in wl.steps)


def peak_for(region_s, peaks):
    """The measured bf16 peak that applies to a timed region: the burst figure
    unless the region runs for seconds (then the power-capped sustained one)."""
    if region_s >= SUSTAINED_AFTER_S:
        return float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])), \
            "bf16_tflops_sustained"
    return float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])), "bf16_tflops"


def mixed_roofline(wl, ms_step, tensor_peak, hbm_peak, kv_quant=False):
    """A step bounded by max(FLOPs / tensor peak, algorithmic bytes / HBM copy bandwidth)."""
    flops = wl.flops()
    byt = algorithmic_bytes(wl, kv_quant)
    t_tensor = flops / (tensor_peak * 1e12) * 1e3
    t_hbm = byt / (hbm_peak * 1e9) * 1e3
    return {"flops_per_step": flops, "bytes_per_step": int(byt), "t_tensor_ms": round(t_tensor, 4),
            "t_hbm_ms": round(t_hbm, 4), "bound": "tensor" if t_tensor >= t_hbm else "hbm",
            "frac": round(max(t_tensor, t_hbm) / ms_step, 4)}


# The configurations the library is measured on besides the headline one, and
# chunked_decode's two parts alone (its 512-token chunk over a 4096-token
# prefix, and its 64 decode rows).
PER_CONFIG = ["tiny_packed", "layer512", "varlen16", "chunked_decode", "chunk512", "decode64"]


def per_config_lines(args, binding, W, peaks, steps):
    import torch
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    lines = {}
    for name in PER_CONFIG:
        wl = W.get(name)
        r = Runner(wl, args, binding, W)
        r.warm(3)
        n = steps if len(wl.steps) == 1 else max(3, steps // 4)
        m = measure(r, n)
        ms = m["ms_step"]
        tflops = wl.flops() / (ms * 1e-3) / 1e12
        byt = algorithmic_bytes(wl)
        lines[name] = {
            "ms_per_step": round(ms, 5), "tflops": round(tflops, 2),
            "tokens_per_s": round(wl.tokens() / (ms * 1e-3), 1), "launches_per_step": len(wl.steps),
            "frac_of_burst_bf16": round(tflops / burst, 4),
            "algorithmic_gbs": round(byt / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm_copy": round(byt / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "roofline_mixed": mixed_roofline(wl, ms, burst, hbm_peak),
            "schedule": r.schedule(), "steps": n,
            "l2": "cold (256 MB written before every step)" if m["cold_l2"] else "inputs larger than L2",
            "value_hot_l2": None if m["hot_ms_step"] is None else
            round(wl.flops() / (m["hot_ms_step"] * 1e-3) / 1e12, 2)}
        # launch-bound configurations: the same step replayed from a CUDA graph
        g_ms = graph_ms_step(r, n)
        lines[name]["value_graph_hot_l2"] = round(wl.flops() / (g_ms * 1e-3) / 1e12, 2)
        lines[name]["ms_per_step_graph_hot_l2"] = round(g_ms, 5)
        del r
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return lines


def run_ours(args, ws, rank, local):
    import torch
    from prefill_phase_attention_gb300 import binding, build
    from prefill_phase_attention_gb300 import workloads as W

    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    binding.load()
    wl = W.get(args.workload)
    runner = Runner(wl, args, binding, W)
    runner.warm(args.warmup)
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    m = measure(runner, args.steps, ws, local, sampler)
    clocks = m["clocks"]
    ms_total, ms_step, per_call_ms = m["ms_total"], m["ms_step"], m["per_call_ms"]
    n_launch = len(runner.dev)
    flops_step = wl.flops(args.window)
    value = weak_scaling_value(flops_step, ms_total, args.steps, ws)
    tokens_s = ws * wl.tokens() / (ms_step * 1e-3)

    peaks, peak_src = load_peaks()
    peak, peak_key = peak_for(m["region_s"], peaks)
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    # roofline of the dominant kernel: algorithmic causal FLOPs per call / mean call time
    per_launch = []
    for li, s in enumerate(wl.steps):
        fl = 4 * wl.head_dim * wl.n_heads * s.visible_pairs(wl.causal, args.window)
        times = per_call_ms[li::n_launch]
        per_launch.append((fl, statistics.mean(times)))
    fl_tot = sum(f for f, _ in per_launch)
    t_tot = sum(t for _, t in per_launch)
    achieved = fl_tot / (t_tot * 1e-3) / 1e12
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    mixed = mixed_roofline(wl, ms_step, peak, hbm_peak, args.kv_quant)
    mixed["peaks"] = f"{peak} TFLOP/s {peak_key}, {hbm_peak} GB/s copy ({peak_src})"
    traffic = None
    variant = (f"_window{args.window}" if args.window else "") + (f"_paged{args.paged}" if args.paged else "") \
        + ("_rope" if args.rope else "") + ("_int8kv" if args.kv_quant else "")
    tpath = os.path.join(ROOT, "profiles", f"traffic_{wl.name}{variant}.json")
    if os.path.exists(tpath):
        rec = json.load(open(tpath))
        if rec.get("kernel_sha256") == kernel_sha256():  # counters of this very kernel code only
            traffic = rec.get("bytes_per_launch")

    # end to end through the public API: pinned host inputs -> device -> call -> host result.
    # Every step copies its own inputs in and its own out/lse back; the copies run
    # on two copy streams into a second set of device buffers, so that step s+1's
    # inputs and step s-1's results move while step s computes.
    steps = runner.inputs[2]
    outs, lses, stream = runner.outs, runner.lses, torch.cuda.current_stream()
    h_in = [{kk: vv.pin_memory() for kk, vv in s.items()} for s in steps]
    h_out = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs] for _ in range(2)]
    h_lse = [[torch.empty(l.shape, dtype=l.dtype).pin_memory() for l in lses] for _ in range(2)]
    d_in = [[{kk: torch.empty_like(vv, device="cuda") for kk, vv in s.items()} for s in steps] for _ in range(2)]
    d_out = [outs, [torch.empty_like(o) for o in outs]]
    d_lse = [lses, [torch.empty_like(l) for l in lses]]
    h2d = sum(v.numel() * v.element_size() for s in steps for v in s.values())
    d2h = sum(o.numel() * o.element_size() for o in outs) + sum(l.numel() * l.element_size() for l in lses)
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]    # inputs of buffer set b landed
    ev_comp = [torch.cuda.Event(), torch.cuda.Event()]  # the step using set b computed
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]   # its results are on the host

    def issue_h2d(step, b):
        if step >= 2:
            h2d_stream.wait_event(ev_comp[b])  # set b's previous step has consumed its inputs
        with torch.cuda.stream(h2d_stream):
            for hi, di in zip(h_in, d_in[b]):
                for kk in hi:
                    di[kk].copy_(hi[kk], non_blocking=True)
            ev_in[b].record(h2d_stream)

    def e2e_run(n):
        issue_h2d(0, 0)
        for step in range(n):
            b = step & 1
            stream.wait_event(ev_in[b])
            if step >= 2:
                stream.wait_event(ev_out[b])  # set b's previous results have been copied out
            for di, o, l in zip(d_in[b], d_out[b], d_lse[b]):
                runner.call(di, o, l)
            ev_comp[b].record(stream)
            if step + 1 < n:
                issue_h2d(step + 1, b ^ 1)
            d2h_stream.wait_event(ev_comp[b])
            with torch.cuda.stream(d2h_stream):
                for o, l, ho, hl in zip(d_out[b], d_lse[b], h_out[b], h_lse[b]):
                    ho.copy_(o, non_blocking=True)
                    hl.copy_(l, non_blocking=True)
                ev_out[b].record(d2h_stream)
        torch.cuda.synchronize()

    e2e_steps = max(3, min(args.steps, 20))
    e2e_run(2)
    barrier(ws)
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    e2e_s = max_over_ranks(time.perf_counter() - t0, ws, device=torch.device("cuda", local))
    e2e_val = ws * flops_step * e2e_steps / e2e_s / 1e12

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": round(tokens_s, 1),
        "pct_of_bf16_peak": round(100 * value / ws / peak, 2),
        "pct_of_bf16_peak_by_reference": {
            "measured_burst": round(100 * value / ws / burst, 2),
            "measured_sustained": round(100 * value / ws / sustained, 2),
            "datasheet_dense": round(100 * value / ws / DATASHEET_BF16_TFLOPS, 2),
            "note": f"measured peaks from MEASURED_PEAKS.json ({peak_src}): cuBLAS bf16 GEMM, burst {burst} and "
                    f"sustained {sustained} TFLOP/s; datasheet: GB300 dense bf16 {DATASHEET_BF16_TFLOPS} TFLOP/s"},
        "config": workload_config(args, wl),
        "run": {"launches_per_step": n_launch, "schedule": runner.schedule(),
                "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                "l2": "inputs larger than L2 (no flush)" if not m["cold_l2"] else
                      "inputs smaller than L2: a 256 MB buffer is written before every timed step (cold L2); "
                      "value_hot_l2 is the same steps back to back",
                "timed_region_s": round(m["region_s"], 4)},
        "roofline_mixed": mixed,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} {peak_key} (timed region {m['region_s']:.3f} s; the sustained "
                                    f"figure applies from {SUSTAINED_AFTER_S:g} s on)",
                     "frac_of_datasheet": round(achieved / DATASHEET_BF16_TFLOPS, 4),
                     "timed": "per prefill_attn_varlen call (scheduler + attention kernel), CUDA events on "
                              "the launching stream"},
        "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                "note": "every step: pinned host q/k/v/metadata -> device, the call, out+lse -> pinned host "
                        "(wall clock over the steps); copies on two copy streams with a second buffer set, "
                        "overlapping the neighbouring steps' compute; KV cache stays device-resident"},
        "gpu_launches": m["launches"],
        "value_hot_l2": None if m["hot_ms_step"] is None else
        round(flops_step / (m["hot_ms_step"] * 1e-3) / 1e12 * ws, 2),
        "clocks": clocks,
    }
    default_run = not (args.window or args.paged or args.rope or args.kv_quant) and args.workload == "long32k"
    if rank == 0 and ws == 1 and not args.no_per_config and default_run:
        del h_in, h_out, h_lse, d_in, d_out, d_lse
        result["per_config"] = per_config_lines(args, binding, W, peaks, max(10, min(args.steps, 50)))
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, runner.inputs, budget_s=args.cpu_budget, window=args.window,
                                              rope=args.rope)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def workload_config(args, wl):
    """The workload part of the JSON line's config (the same in both arms)."""
    return {"workload": wl.name + (f"+window{args.window}" if args.window else "")
            + (f"+paged{args.paged}" if args.paged else "") + (f"+rope{args.rope:g}" if args.rope else "")
            + ("+int8kv" if args.kv_quant else ""),
            "window": args.window, "num_seqs": wl.num_seqs,
            "kv_cache": (f"paged, {args.paged}-token blocks" if args.paged else "contiguous per sequence")
            + (", int8 codes + fp32 row scales" if args.kv_quant else ", bf16"),
            "rope_theta": args.rope,
            "tokens_per_step": wl.tokens(), "n_heads": wl.n_heads, "n_kv_heads": wl.n_kv_heads,
            "head_dim": wl.head_dim, "causal": wl.causal, "causal_flops_per_step": wl.flops(args.window)}


# ----------------------------------------------------------- reference arm --

def run_reference(args, ws, rank):
    if rank != 0:
        return
    from prefill_phase_attention_gb300 import workloads as W
    import oracle
    oracle.build()
    wl = W.get(args.workload)
    inputs = W.make_inputs(wl, sentinel=False)
    step = wl.steps[-1]
    cores = host_cores()
    rows = oracle_sample_rows(wl, step, args.ref_rows, seed=13)
    fl = row_flops(wl, step, rows, args.window)
    for _ in range(args.warmup):
        time_oracle(wl, inputs, rows, cores, args.window, args.rope)
    total = 0.0
    for _ in range(args.steps):
        total += time_oracle(wl, inputs, rows, cores, args.window, args.rope)
    value = fl * args.steps / total / 1e12
    sample = (f"{rows.size} query rows (token, head) drawn uniformly from {wl.name} per step, "
              f"{fl / 1e9:.2f} GFLOP causal per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, wl),
        "run": {"parallelism": "host cores", "launches_per_step": len(wl.steps)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long32k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--window", type=int, default=0, help="sliding window (0: none; the bench line counts only "
                                                             "the visible pairs)")
    ap.add_argument("--paged", type=int, default=0, help="block size of a paged KV cache (0: contiguous cache)")
    ap.add_argument("--rope", type=float, default=0.0, help="rotary embedding base (0: none)")
    ap.add_argument("--kv-quant", action="store_true", help="int8 KV cache with per-token fp32 scales")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-config block of the default run")
    ap.add_argument("--cpu-budget", type=float, default=25.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-rows", type=int, default=128, help="oracle rows per reference step")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps, reported as run
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
