#!/usr/bin/env python
"""Benchmark of the low-bit KV-cache decode hot path on GB300.

A step is one decode step of one layer: append one new token for every
(batch, kv-head) stream (kvq_append), then decode attention for every query
head over the whole cache (kvq_decode_attn: split-T partial kernel + combine).
The default workload is the long-context cache: B=1, H=32/8, D=128,
T=2^20, INT4 with 1% outliers, RoPE theta 5e5, 32 layers resident in HBM
(about 41 GB), one layer per step in rotation. After the headline the same
run measures the other workloads (7B MHA, 8B GQA, INT3, INT2 decode and the
INT3 / INT2 / INT4 prefill appends) and reports them under "configs" in the
same JSON line. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--mode decode|prefill|paged|levels] [--impl kvq|reference]
                  [--configs all|none]

--impl reference times the CPU oracle (the plain C++ reference) on the host
cores: each step is one oracle decode step on a bounded sample of the same
workload (all streams when there are few, a slice of the cached tokens),
sized so the whole run ends within a few minutes; ms_per_step is that
sample step, value the metric of the full step by linear extrapolation.
--mode prefill times one kvq_append of the workload's whole context (the
aggressive-bits prefill run) instead of decode steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import kvq_inputs as ki  # noqa: E402

L2_BYTES = 129 * 2 ** 20
# Sources of the decode kernels: a roofline.traffic figure read from profiles/
# counts only if it was captured on these exact files.
DECODE_SOURCES = {
    128: ["kvq_decode_tc.cuh", "kvq_tc_geom.cuh", "kvq_decode_tc_inst.cuh", "kvq_decode_tc_b4.cu",
          "kvq_decode_tc_b3.cu", "kvq_decode_tc_b2.cu", "kvq_decode_tc_b4o.cu", "kvq_decode_tc_b3o.cu",
          "kvq_decode_tc_b2o.cu", "kvq_decode.cuh", "kvq_decode.cu", "kvq_common.cuh"],
    "paged": ["kvq_decode_tc.cuh", "kvq_tc_geom.cuh", "kvq_decode_tc_inst.cuh", "kvq_decode_tc_b4p.cu",
              "kvq_decode_tc_b3p.cu", "kvq_decode_tc_b2p.cu", "kvq_decode_tc_b4op.cu", "kvq_decode_tc_b3op.cu",
              "kvq_decode_tc_b2op.cu", "kvq_decode.cuh", "kvq_decode.cu", "kvq_common.cuh"],
    64: ["kvq_decode.cuh", "kvq_decode.cu", "kvq_decode_inst.cuh", "kvq_common.cuh"],
}
DECODE_KERNEL = {128: "decode_tc_kernel", 64: "decode_partial_kernel"}


# ----------------------------------------------------------------------------- helpers
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def n_out_of(w):
    return 0 if w.outlier_frac == 0 else max(1, int(math.floor(w.outlier_frac * w.D)))


def workload_string(w):
    """The workload as both arms name it in config.workload."""
    return (f"{w.name}: B={w.B} H_q={w.H_q} H_kv={w.H_kv} D={w.D} T={w.T} INT{w.bits} "
            f"key_block={w.key_block} value_group={w.value_group} outliers={w.outlier_frac} "
            f"rope_theta={w.rope_theta} layers_resident={w.layers}")


def decode_alg_bytes(w, T):
    """Algorithmic bytes one decode call must read/write: packed K and V codes,
    fp16 key metadata per block and channel, fp16 value metadata per token and
    group, outlier pairs, the fp16 tail keys, q and out."""
    streams = w.B * w.H_kv
    cb = w.D * w.bits // 8
    ng = w.D // w.value_group
    nout = n_out_of(w)
    nf, tail = divmod(T, w.key_block)
    per_block = 2 * cb * w.key_block + 4 * w.D + 4 * ng * w.key_block + 2 * 4 * nout * w.key_block
    per_tail_tok = 2 * w.D + cb + 4 * ng + 4 * nout
    qo = 2 * w.B * w.H_q * w.D * 2
    return streams * (nf * per_block + tail * per_tail_tok) + qo


def append_alg_bytes(w, n_new):
    """Prefill append: fp16 K and V read, codes + metadata + outliers written."""
    streams = w.B * w.H_kv
    cb = w.D * w.bits // 8
    ng = w.D // w.value_group
    nout = n_out_of(w)
    nb = n_new // w.key_block
    read = 2 * streams * n_new * w.D * 2
    write = streams * (2 * n_new * cb + nb * w.D * 4 + n_new * ng * 4 + 2 * n_new * nout * 4)
    return read + write


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "bit_quantized_kv_append_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_file, sha):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", kernel_file)
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if "=" in line and not line.lstrip().startswith("#"):
            k, v = line.split("=", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha") != sha or "traffic_bytes_per_launch" not in vals:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except ValueError:
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def physical_gpu(local_index):
    """nvidia-smi's id of a CUDA device index (honours CUDA_VISIBLE_DEVICES)."""
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if cvd:
        items = [x.strip() for x in cvd.split(",")]
        if local_index < len(items):
            return items[local_index]
    return str(local_index)


def host_cpu():
    model = platform.processor() or platform.machine()
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    return model


def max_over_ranks(values, device):
    """Element-wise max of a list of floats over all ranks (identity at world 1).
    Replicas run independently; the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def replica_throughput(units_per_rank, world, ms):
    """Whole-job units/s of `world` independent replicas that each processed
    units_per_rank units in (at most) ms milliseconds."""
    return world * units_per_rank / (ms * 1e-3)


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_sample(w, n_streams, n_tok):
    """A bounded sample for the oracle: n_streams streams of n_tok cached
    tokens, generated and encoded once. Returns (step, threads): step() runs
    and times (wall clock) one decode step of the oracle on all host threads:
    encode the new token, dequantize the cache, float64 attention of the
    stream's G heads."""
    from oracle import oracle_cpp as oc

    streams = [(s // w.H_kv % w.B, s % w.H_kv) for s in range(n_streams)]
    K, V = ki.streams_np(w, streams, n_tok + 1)
    enc = oc.encode(K[:, :n_tok], V[:, :n_tok], w.bits, w.key_block, w.value_group, n_out_of(w))
    q = ki.queries_np(w, 0, 0)
    qs = np.stack([q[b, h * w.G:(h + 1) * w.G] for (b, h) in streams])
    threads = oc.default_threads()
    k_new, v_new = np.ascontiguousarray(K[:, n_tok:]), np.ascontiguousarray(V[:, n_tok:])

    def step():
        t0 = time.perf_counter()
        oc.encode(k_new, v_new, w.bits, w.key_block, w.value_group, n_out_of(w), threads)
        Kh, Vh = oc.dequant(enc, n_tok, w.D, w.bits, w.key_block, w.value_group, n_out_of(w), threads)
        oc.attention(Kh, Vh, qs, n_tok, w.rope_theta, 1.0 / math.sqrt(w.D), 0.0, threads)
        return time.perf_counter() - t0

    return step, threads


def oracle_step_seconds(w, n_streams, n_tok, reps=1):
    """Median wall time of `reps` oracle decode steps on one bounded sample."""
    step, threads = oracle_sample(w, n_streams, n_tok)
    return statistics.median(step() for _ in range(reps)), threads


def cpu_baseline_prefill(w, budget_s=15.0):
    """Oracle encode (the quantizer) on a bounded sample of the prefill:
    one stream per host thread, a slice of the new tokens, extrapolated."""
    from oracle import oracle_cpp as oc
    threads = oc.default_threads()
    n_streams = min(threads, w.B * w.H_kv)
    streams = [(s // w.H_kv % w.B, s % w.H_kv) for s in range(n_streams)]
    n_tok = min(w.T, 4096)
    K, V = ki.streams_np(w, streams, n_tok)
    t0 = time.perf_counter()
    oc.encode(K, V, w.bits, w.key_block, w.value_group, n_out_of(w), threads)
    t = time.perf_counter() - t0
    if t < budget_s / 4 and n_tok < w.T:
        n_tok = min(w.T, int(n_tok * budget_s / 2 / max(t, 1e-3)) // w.key_block * w.key_block)
        K, V = ki.streams_np(w, streams, n_tok)
        t0 = time.perf_counter()
        oc.encode(K, V, w.bits, w.key_block, w.value_group, n_out_of(w), threads)
        t = time.perf_counter() - t0
    return {
        "value": n_streams * n_tok / t, "unit": "kv-tokens/s", "cores": threads, "kind": "oracle",
        "sample": (f"{n_streams} of {w.B * w.H_kv} (b,h_kv) streams x {n_tok} of {w.T} new tokens, "
                   f"oracle encode (outliers, scales, codes, packing), {t:.2f} s wall; host {host_cpu()}"),
    }


def cpu_baseline(w, budget_s=15.0):
    """Oracle on a bounded sample: one stream per host thread, the full T each,
    extrapolated to all B*H_kv streams."""
    from oracle import oracle_cpp as oc
    threads = oc.default_threads()
    n_streams = min(threads, w.B * w.H_kv)
    n_tok = w.T
    t_probe, _ = oracle_step_seconds(w, 1, min(n_tok, 4096))
    est = t_probe * (n_tok / min(n_tok, 4096)) * math.ceil(n_streams / threads)
    if est > budget_s:
        n_tok = max(w.key_block, int(n_tok * budget_s / est) // w.key_block * w.key_block)
    # the sample is generated and encoded once (host numpy + oracle): keep it
    # to about 2^21 cached token-heads so the setup stays a few seconds
    n_tok = max(w.key_block, min(n_tok, (1 << 21) // n_streams // w.key_block * w.key_block))
    t, threads = oracle_step_seconds(w, n_streams, n_tok)
    # repeat a short sample until it holds about budget_s of host work; median per repetition
    reps = max(1, min(64, int(budget_s / max(t, 1e-3))))
    if reps > 1:
        t, threads = oracle_step_seconds(w, n_streams, n_tok, reps)
    full = t * (w.T / n_tok) * (w.B * w.H_kv / n_streams)
    return {
        "value": w.B / full, "unit": "tokens/s", "cores": threads, "kind": "oracle",
        "sample": (f"{n_streams} of {w.B * w.H_kv} (b,h_kv) streams x {n_tok} of {w.T} cached tokens, "
                   f"one decode step (encode new token, dequantize, float64 attention), "
                   f"{reps} repetitions, median {t:.3f} s wall each, extrapolated linearly to the full step; "
                   f"host {host_cpu()}"),
    }


# ----------------------------------------------------------------------------- GPU runs
def build_cache(w, T, T_max, device, layer=0, rope_table=None, precise=False):
    import bit_quantized_kv_append_gb300 as kvq
    cache = kvq.QuantizedKVCache(w.B, w.H_kv, w.D, T_max, w.bits, w.key_block, w.value_group,
                                 w.outlier_frac, H_q=w.H_q, rope_theta=w.rope_theta, device=device,
                                 rope_table=rope_table, precise=precise)
    chunk = max(w.key_block, (1 << 26) // max(1, w.B * w.H_kv * w.D) // w.key_block * w.key_block)
    t = 0
    while t < T:
        n = min(chunk, T - t)
        K, V = ki.kv_torch(w, layer, t, n, device)
        cache.append(K, V)
        t += n
    return cache


def run_decode(args, w, rank, world, device):
    import torch
    import torch.distributed as dist

    T = w.T
    T_max = T + w.key_block
    n_layers = w.layers
    precise = getattr(args, "precise", False)
    cache0 = build_cache(w, T, T_max, device, precise=precise)
    caches = [cache0] + [build_cache(w, T, T_max, device, layer=l, rope_table=cache0.rope, precise=precise)
                         for l in range(1, n_layers)]
    k1, v1 = ki.kv_torch(w, 0, T, 1, device)
    q = ki.queries_torch(w, 0, 1, device)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        c = caches[i % n_layers]
        c.reset(T)
        c.append(k1, v1)
        if ev is not None:
            ev[0].record(stream)
        c.decode(q, out=out)
        if ev is not None:
            ev[1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(physical_gpu(torch.cuda.current_device()))
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = t_start.elapsed_time(t_end)
    dec_ms = [a.elapsed_time(b) for a, b in evs]

    # end to end through the public API from pinned host buffers
    kh, vh, qh = k1.cpu().pin_memory(), v1.cpu().pin_memory(), q.cpu().pin_memory()
    oh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    kd, vd, qd = torch.empty_like(k1), torch.empty_like(v1), torch.empty_like(q)

    def e2e_step(i):
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        qd.copy_(qh, non_blocking=True)
        c = caches[i % n_layers]
        c.reset(T)
        c.decode_step(kd, vd, qd, out=out)          # kvq_decode_step: append + attention, one call
        oh.copy_(out, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_end)

    ms, e2e_ms, dec_mean = max_over_ranks([ms, e2e_ms, statistics.mean(dec_ms)], device)
    bytes_step_in = (k1.numel() + v1.numel() + q.numel()) * 2
    bytes_step_out = out.numel() * 2
    alg = decode_alg_bytes(w, T + 1)
    peak, peak_kind = measured_peaks()
    achieved = alg / (dec_mean * 1e-3) / 1e9
    sha = source_sha(DECODE_SOURCES[w.D])
    kname = DECODE_KERNEL[w.D]
    line = {
        "metric": "decode-attn tokens/s (one layer; B query tokens per step)",
        "value": replica_throughput(w.B * args.steps, world, ms),
        "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"u{w.bits}/f16/f32", "data": "synthetic",
        "config": {
            "workload": workload_string(w),
            "step": "kvq_append of 1 token per stream + kvq_decode_attn over T+1 tokens"
                    + (" (KVQ_FLAG_PRECISE_SCORES)" if precise else ""),
            "l2": f"inputs larger than L2 (cache {caches[0].layout.cache_bytes / 1e9:.2f} GB per layer > 129 MB); no flush",
            "parallelism": f"replicas x{world}",
            "kv_tokens_per_s": replica_throughput(w.B * (T + 1) * args.steps, world, ms),
            "model_level_tokens_per_s_32_layers": replica_throughput(w.B * args.steps, world, ms) / 32,
            "decode_call_ms": dec_mean,
        },
        "e2e": {"value": replica_throughput(w.B * args.steps, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": bytes_step_in, "d2h_bytes_per_step": bytes_step_out,
                "call": "kvq_decode_step from pinned host buffers"},
        "gpu_launches": 3 * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "kernel": f"{kname} (+ decode_combine_kernel: one kvq_decode_attn call timed per step)",
                     "alg_bytes_per_launch": alg,
                     "traffic": profile_traffic(f"{kname}_{w.name}.txt", sha),
                     "source_sha": sha},
        "clocks": clk,
    }
    return line


def run_prefill(args, w, rank, world, device):
    import torch
    import torch.distributed as dist
    import bit_quantized_kv_append_gb300 as kvq

    n_new = w.T
    T_max = n_new
    cache = kvq.QuantizedKVCache(w.B, w.H_kv, w.D, T_max, w.bits, w.key_block, w.value_group,
                                 w.outlier_frac, H_q=w.H_q, device=device)
    K, V = ki.kv_torch(w, 0, 0, n_new, device)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        cache.reset(0)
        cache.append(K, V)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(physical_gpu(torch.cuda.current_device()))
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        cache.reset(0)
        evs[i][0].record(stream)
        cache.append(K, V)
        evs[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    # end to end: fp16 K/V copied from pinned host memory each step
    Kh, Vh = K.cpu().pin_memory(), V.cpu().pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        K.copy_(Kh, non_blocking=True)
        V.copy_(Vh, non_blocking=True)
        cache.reset(0)
        cache.append(K, V)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    ms, e2e_ms, call_ms = max_over_ranks([ms, e2e_ms, call_ms], device)
    alg = append_alg_bytes(w, n_new)
    peak, peak_kind = measured_peaks()
    achieved = alg / (call_ms * 1e-3) / 1e9
    sha = source_sha(["kvq_append.cu", "kvq_common.cuh"])
    toks = w.B * w.H_kv * n_new
    return {
        "metric": "append (prefill quantize) kv-tokens/s",
        "value": replica_throughput(toks * args.steps, world, ms), "unit": "kv-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": f"f16/f32->u{w.bits}",
        "data": "synthetic",
        "config": {"workload": f"{w.name} prefill: B={w.B} H_kv={w.H_kv} D={w.D} n_new={n_new} INT{w.bits} "
                               f"key_block={w.key_block} value_group={w.value_group} outliers={w.outlier_frac}",
                   "l2": f"inputs larger than L2 ({2 * toks * w.D * 2 / 1e9:.2f} GB fp16 in); no flush",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": replica_throughput(toks * args.steps, world, e2e_ms), "unit": "kv-tokens/s",
                "h2d_bytes_per_step": 2 * toks * w.D * 2, "d2h_bytes_per_step": 0},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind, "kernel": "append_kernel", "alg_bytes_per_launch": alg,
                     "traffic": profile_traffic(f"append_{w.name}.txt", sha), "source_sha": sha},
        "clocks": clk,
    }


def paged_lengths(w):
    """Ragged prefill lengths of the paged workload: T (B - b) / B tokens for
    sequence b, rounded down to whole key blocks (at least one block)."""
    return [max(w.key_block, w.T * (w.B - b) // w.B // w.key_block * w.key_block) for b in range(w.B)]


def run_paged(args, w, rank, world, device):
    """Decode step of a paged, ragged batch: every sequence appends one token
    at its own position (kvq_paged_append) and attends over all of its tokens
    (kvq_paged_decode_attn); the sequences' key blocks sit in one pool in a
    seeded random order. The sequences grow by one token per step."""
    import numpy as np
    import torch
    import torch.distributed as dist
    import bit_quantized_kv_append_gb300 as kvq

    Bk = w.key_block
    lens = paged_lengths(w)
    grow = args.warmup + args.steps + 2
    T_max = (max(lens) + grow + Bk - 1) // Bk * Bk
    per_seq = [(L + grow + Bk - 1) // Bk for L in lens]
    n_blocks = sum(per_seq) + 8
    cache = kvq.PagedKVCache(w.B, w.H_kv, w.D, T_max, n_blocks, w.bits, Bk, w.value_group, w.outlier_frac,
                             H_q=w.H_q, rope_theta=w.rope_theta, device=device)
    rng = np.random.default_rng(1000 + w.seed)
    perm = rng.permutation(n_blocks)
    table = np.zeros((w.B, T_max // Bk), np.int32)
    k = 0
    for b, nb in enumerate(per_seq):
        table[b, :nb] = perm[k:k + nb]
        k += nb
    cache.block_table.copy_(torch.from_numpy(table))
    chunk = 1 << 15
    for t0 in range(0, max(lens), chunk):
        n = min(chunk, max(lens) - t0)
        K, V = ki.kv_torch(w, 0, t0, n, device)
        for b, L in enumerate(lens):
            if t0 < L:
                m = min(n, L - t0)
                cache.append_seq(b, K[b:b + 1, :, :m].contiguous(), V[b:b + 1, :, :m].contiguous())
        del K, V
    k1, v1 = ki.kv_torch(w, 0, max(lens), 1, device)     # the step's new token of every sequence
    q = ki.queries_torch(w, 0, 1, device)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        cache.append(k1, v1)
        if ev is not None:
            ev[0].record(stream)
        cache.decode(q, out=out)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    lens_t0 = list(cache.lengths)
    clocks = ClockSampler(physical_gpu(torch.cuda.current_device()))
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    dec_ms = [a.elapsed_time(b) for a, b in evs]
    ms, dec_mean = max_over_ranks([ms, statistics.mean(dec_ms)], device)
    # algorithmic bytes of the average decode call (lengths after each step's append)
    one = w.replace(B=1)
    alg = statistics.mean(sum(decode_alg_bytes(one, L + 1 + i) for L in lens_t0) for i in range(args.steps))
    peak, peak_kind = measured_peaks()
    achieved = alg / (dec_mean * 1e-3) / 1e9
    sha = source_sha(DECODE_SOURCES["paged"])
    return {
        "metric": "decode-attn tokens/s (one layer; B query tokens per step), paged ragged batch",
        "value": replica_throughput(w.B * args.steps, world, ms), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"u{w.bits}/f16/f32", "data": "synthetic",
        "config": {
            "workload": (f"{w.name} paged: B={w.B} H_q={w.H_q} H_kv={w.H_kv} D={w.D} lengths={lens_t0} (+1 per "
                         f"step) INT{w.bits} key_block={Bk} value_group={w.value_group} outliers={w.outlier_frac} "
                         f"rope_theta={w.rope_theta} pool={n_blocks} blocks, shuffled block table"),
            "step": "kvq_paged_append of 1 token per sequence + kvq_paged_decode_attn",
            "l2": f"inputs larger than L2 (pools {cache.layout.cache_bytes / 1e9:.2f} GB > 129 MB); no flush",
            "parallelism": f"replicas x{world}",
            "decode_call_ms": dec_mean,
        },
        "gpu_launches": 4 * args.steps,      # append + length advance, decode + combine
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind,
                     "kernel": "decode_tc_kernel paged (+ decode_combine_kernel: one kvq_paged_decode_attn call)",
                     "alg_bytes_per_launch": alg,
                     "traffic": profile_traffic(f"decode_tc_kernel_{w.name}_paged.txt", sha), "source_sha": sha},
        "clocks": clk,
    }


def run_levels(args, w, rank, world, device):
    """Non-uniform codes: a level table fitted (kvq_fit_levels) to the
    normalized values of another layer's groups; the cache is filled with
    kvq_append_levels and each step times one kvq_decode_attn_levels call over
    T tokens (the tensor-core kernel in its level-table mode at head_dim 128,
    the CUDA-core kernel at head_dim 64)."""
    import numpy as np
    import torch
    import torch.distributed as dist
    import bit_quantized_kv_append_gb300 as kvq

    T = w.T
    sha = source_sha(DECODE_SOURCES[128] + ["kvq_decode_tc_b2lv.cu", "kvq_decode_tc_b3lv.cu", "kvq_decode_tc_b4lv.cu",
                                            "kvq_decode_tc_b8lv.cu"])
    Kc, Vc = ki.streams_np(w, [(0, 0)], 1024, layer=9)
    x = np.concatenate([Kc.reshape(-1, w.value_group), Vc.reshape(-1, w.value_group)]).astype(np.float64)
    span = x.max(axis=1, keepdims=True) - x.min(axis=1, keepdims=True)
    levels = kvq.fit_levels(((x - x.min(axis=1, keepdims=True)) / np.where(span > 0, span, 1.0)).ravel(), w.bits, 60)
    cache = kvq.QuantizedKVCache(w.B, w.H_kv, w.D, T + w.key_block, w.bits, w.key_block, w.value_group,
                                 w.outlier_frac, H_q=w.H_q, rope_theta=w.rope_theta, device=device)
    stream = torch.cuda.current_stream()
    chunk = 1 << 15
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for t0 in range(0, T, chunk):
        K, V = ki.kv_torch(w, 0, t0, min(chunk, T - t0), device)
        cache.append_levels(K, V, levels)
    a1.record(stream)
    q = ki.queries_torch(w, 0, 1, device)
    out = torch.empty_like(q)
    for _ in range(args.warmup):
        cache.decode_levels(q, levels, out=out)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(physical_gpu(torch.cuda.current_device()))
    clocks.start()
    time.sleep(0.3)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        cache.decode_levels(q, levels, out=out)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    (ms,) = max_over_ranks([ms], device)
    dec_ms = ms / args.steps
    alg = decode_alg_bytes(w, T)
    peak, peak_kind = measured_peaks()
    achieved = alg / (dec_ms * 1e-3) / 1e9
    return {
        "metric": "decode-attn tokens/s (one layer; B query tokens per step), non-uniform codes",
        "value": replica_throughput(w.B * args.steps, world, ms), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dec_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"u{w.bits}/f16/f32", "data": "synthetic",
        "config": {
            "workload": (f"{w.name} with a {1 << w.bits}-level table: B={w.B} H_q={w.H_q} H_kv={w.H_kv} D={w.D} "
                         f"T={T} INT{w.bits} key_block={w.key_block} value_group={w.value_group} "
                         f"outliers={w.outlier_frac} rope_theta={w.rope_theta}"),
            "step": "kvq_decode_attn_levels over T tokens",
            "append_ms_whole_context_with_input_generation": a0.elapsed_time(a1),
            "l2": f"inputs larger than L2 (cache {cache.layout.cache_bytes / 1e9:.2f} GB > 129 MB); no flush",
            "parallelism": f"replicas x{world}",
        },
        "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind,
                     "kernel": ("decode_tc_kernel, level-table mode (+ decode_combine_kernel)" if w.D == 128
                                else "decode_levels_kernel + combine (CUDA cores)"),
                     "alg_bytes_per_launch": alg,
                     "traffic": profile_traffic(f"decode_tc_kernel_{w.name}_levels.txt", sha) if w.D == 128 else None,
                     "source_sha": sha},
        "clocks": clk,
    }


def reference_sample_size(w, n_steps, budget_s=80.0):
    """Streams and cached tokens of the reference arm's per-step sample: every
    stream when they fit twice the host threads (else one per thread), and
    the largest whole number of key blocks for which n_steps oracle steps
    plus the sample's one-time generation and encoding (measured at about
    seven steps) stay within budget_s of host time."""
    from oracle import oracle_cpp as oc
    threads = oc.default_threads()
    streams = w.B * w.H_kv
    n_streams = streams if streams <= 2 * threads else threads
    probe_tok = min(w.T, 4096)
    t_probe, _ = oracle_step_seconds(w, n_streams, probe_tok, reps=2)
    per_tok = t_probe / probe_tok
    n_tok = int(budget_s / ((n_steps + 8) * max(per_tok, 1e-12)))
    n_tok = max(w.key_block, min(w.T, n_tok // w.key_block * w.key_block))
    return n_streams, n_tok


def run_reference(args, w):
    """The CPU oracle as the reference arm. Each step is one oracle decode step
    (encode the new token, dequantize, float64 attention) on a bounded sample of
    the workload; ms_per_step is that step's wall time, value the metric of the
    full step (all streams, all T tokens) by linear extrapolation."""
    from oracle import oracle_cpp as oc
    oc.build()
    n_streams, n_tok = reference_sample_size(w, args.steps + args.warmup)
    step, threads = oracle_sample(w, n_streams, n_tok)
    times = []
    for i in range(args.warmup + args.steps):
        t = step()
        if i >= args.warmup:
            times.append(t)
    step_s = statistics.mean(times)
    factor = (w.T / n_tok) * (w.B * w.H_kv / n_streams)
    value = w.B / (step_s * factor)
    sample = (f"per step {n_streams} of {w.B * w.H_kv} (b,h_kv) streams x {n_tok} of {w.T} cached tokens "
              f"(encode new token, dequantize, float64 attention) on {threads} host threads; value "
              f"extrapolated linearly to the full step (x{factor:.3g}); host {host_cpu()}")
    return {
        "impl": "reference", "metric": "decode-attn tokens/s (one layer; B query tokens per step)",
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_string(w),
                   "step": "one oracle decode step on the bounded sample below (ms_per_step); "
                           "value = B / (ms_per_step x extrapolation factor)",
                   "full_step_ms_extrapolated": step_s * factor * 1e3},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


SUITE = [("decode", "mha7b"), ("decode", "gqa8b"), ("decode", "int3"), ("decode", "int2"),
         ("prefill", "int3"), ("prefill", "int2"), ("prefill", "gqa8b")]


def run_config_suite(args, rank, world, device):
    """The other workloads, measured after the headline in the same run (up to
    20 timed steps each, at least 3 warm-up steps); their figures go into the
    headline's JSON line under "configs"."""
    import argparse as _ap
    import torch
    sub = _ap.Namespace(**vars(args))
    sub.steps = max(1, min(args.steps, 20))
    sub.warmup = max(3, min(args.warmup, 5))
    out = {}
    for mode, name in SUITE:
        w = ki.WORKLOADS[name]
        line = (run_decode if mode == "decode" else run_prefill)(sub, w, rank, world, device)
        torch.cuda.empty_cache()
        rf = line["roofline"]
        entry = {"metric": line["metric"], "value": line["value"], "unit": line["unit"],
                 "ms_per_step": line["ms_per_step"], "steps": sub.steps, "warmup": sub.warmup,
                 "workload": line["config"]["workload"],
                 "roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac", "kernel",
                                                 "alg_bytes_per_launch", "traffic")},
                 "e2e": line["e2e"]["value"], "clocks": line["clocks"]}
        if "decode_call_ms" in line["config"]:
            entry["decode_call_ms"] = line["config"]["decode_call_ms"]
        out[f"{mode}:{name}"] = entry
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default="long1m", choices=list(ki.WORKLOADS))
    ap.add_argument("--configs", default="all", choices=["all", "none"],
                    help="after a default decode run, also measure the other workloads")
    ap.add_argument("--mode", default="decode", choices=["decode", "prefill", "paged", "levels"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--precise", action="store_true",
                    help="decode with KVQ_FLAG_PRECISE_SCORES (fp32 keys, hi + lo operands)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = ki.WORKLOADS[args.workload]
    rank, local_rank, world = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return

    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from bit_quantized_kv_append_gb300 import build as kbuild
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0:
        kbuild.build()
    if world > 1:
        dist.barrier()
    device = torch.device("cuda", local_rank if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    line = {"prefill": run_prefill, "paged": run_paged, "decode": run_decode,
            "levels": run_levels}[args.mode](args, w, rank, world, device)
    torch.cuda.empty_cache()
    if args.configs == "all" and args.mode == "decode" and args.workload == "long1m":
        line["configs"] = run_config_suite(args, rank, world, device)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_prefill(w) if args.mode == "prefill" else cpu_baseline(w)
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
