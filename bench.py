#!/usr/bin/env python
"""Throughput of the chunked gated delta rule forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--algo auto|simt|tc]

A step is one full forward (WY build, recompute_w_u, chunk_fwd_h, chunk_fwd_o)
over one batch of the named synthetic workload, through the C ABI, with the
inputs resident in HBM; the L2 is flushed (a 512 MiB write) before every timed
step. The metric is tokens/s (B*T per step). Under torchrun each rank runs its
own copy of the workload on its own GPU (weak scaling, no collective on the
data path); the time is the max over ranks. Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on the host cores instead (rank 0
only), each step a bounded sample of the workload's (b, h) sequences.

The line also carries "decode": the recurrent decode step timed on its own
workload (256 sequences x 16 heads, one token, K = V = 128, bf16) against the
HBM roofline of reading and writing the fp32 state once (--no-decode skips it);
"frontend": the same step on raw inputs with the chunk-local cumsum of g
and the q/k L2 norm done in the kernels (--no-frontend skips it); and
"output_norm": the same step with the gated RMSNorm output stage, and
"output_norm_headline": the stage on the headline workload, each with its ratio
to the plain step (--no-output-norm skips both); "per_channel": the chunked
step and the decode step with per-channel (KDA) decay (--no-per-channel skips
it). "pipeline_roofline.design_traffic" is the DRAM bytes the step's kernels
move (the committed ncu records, where current), beside the compulsory bytes.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import torch  # noqa: E402

from gated_delta_rule_35_gb300.inputs import (BENCH_WORKLOAD, DECODE_WORKLOADS, FEATURE_WORKLOAD,  # noqa: E402
                                              WORKLOADS,
                                              make_inputs, make_workload, to_f64)

DECODE_WORKLOAD = "bf16_b256_h16_t1_k128_v128_decode"

METRIC = "GDN chunked-fwd tokens/s on 1 GB300; % of roofline; vs CPU oracle"
CHUNK = 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
SMS, FP32_LANES = 152, 128          # GB300: SMs, fp32 FMA lanes per SM
DSIZE = {"f32": 4, "bf16": 2}


# --------------------------------------------------------------------------- cost model
def flops_per_token_head(K, V, C=CHUNK):
    """Algorithmic flops per token-head (triangular halves counted once):
    Gram (C-1)K, w/u (C+1)(K+V), q k^T (C+1)K, P v_new (C+1)V, state terms
    6KV (w@h, k^T@v_gated, q@h), triangular inverse ~C^2/3."""
    return (C - 1) * K + (C + 1) * (K + V) + (C + 1) * K + (C + 1) * V + 6 * K * V + C * C / 3


def bytes_per_token_head(K, V, d):
    """Compulsory HBM bytes per token-head: read q, k, v, g, beta; write o."""
    return d * (2 * K + 2 * V) + 8


# Per kernel: (bound, algorithmic bytes per token-head, flops per token-head) as
# functions of (K, V, element size). The SIMT kernels keep fp32 intermediates.
def _simt_prepare(K, V, d):
    return d * (K + V) + 8 + 4 * (CHUNK + K + V), (CHUNK - 1) * K + CHUNK * CHUNK / 3 + (CHUNK + 1) * (K + V)


def _simt_h(K, V, d):
    return 4 * (K + V) + d * K + 4 + 4 * K * V / CHUNK + 4 * V, 4 * K * V


def _simt_o(K, V, d):
    return 2 * d * K + 4 + 4 * K * V / CHUNK + 4 * V + d * V, 2 * K * V + (CHUNK + 1) * (K + V)


def _fused(K, V, d):
    return bytes_per_token_head(K, V, d), flops_per_token_head(K, V)


KERNEL_MODEL = {
    "gdn_fused_tc_kernel": ("hbm", _fused),
    "gdn_wide_tc_kernel": ("hbm", _fused),
    "wy_prepare_kernel": ("alu", _simt_prepare),
    "chunk_h_kernel": ("alu", _simt_h),
    "chunk_o_kernel": ("alu", _simt_o),
}
KERNEL_SOURCE = {
    "gdn_fused_tc_kernel": "gated_delta_rule_35_gb300/csrc/gdn_tc.cu",
    "gdn_wide_tc_kernel": "gated_delta_rule_35_gb300/csrc/gdn_tc_wide.cu",
    "gdn_wy_tc_kernel": "gated_delta_rule_35_gb300/csrc/gdn_tc_wy.cu",
    "gdn_decode_step_kernel": "gated_delta_rule_35_gb300/csrc/gdn_decode.cu",
    "wy_prepare_kernel": "gated_delta_rule_35_gb300/csrc/gdn_simt.cu",
    "chunk_h_kernel": "gated_delta_rule_35_gb300/csrc/gdn_simt.cu",
    "chunk_o_kernel": "gated_delta_rule_35_gb300/csrc/gdn_simt.cu",
}


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        d["_source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["_source"] = "fallback"
    return d


def source_sha(rel_path):
    return hashlib.sha256((ROOT / rel_path).read_bytes()).hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's source changed since the counters were taken (for a split
    forward, "a+b", the sum of both records, or None)."""
    if "+" in kernel:
        parts = [ncu_traffic(k, workload) for k in kernel.split("+")]
        return None if any(p is None for p in parts) else sum(parts)
    f = ROOT / "profiles" / "dram_traffic.json"
    if not f.exists():
        return None
    recs = json.loads(f.read_text()).get(kernel)
    # one record, or a list of them (one per workload)
    recs = recs if isinstance(recs, list) else [recs] if recs else []
    rec = next((r for r in recs if r.get("workload") == workload), None)
    if rec is None:
        return None
    src = KERNEL_SOURCE.get(kernel)
    if not src or rec.get("source_sha") != source_sha(src):
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and clock-event reasons seen while the timed steps run.

    A host thread reads them through NVML (libnvidia-ml, read-only queries)
    about every millisecond, so that even a timed region of a few milliseconds
    gets samples; without NVML it polls nvidia-smi every 100 ms instead. Only
    samples taken between mark_start() and mark_end() are reported; when the
    region is shorter than the sampling period the nearest sample stands in and
    "window" says so."""
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    # nvmlClocksEventReason* bit values from the public NVML header
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, device, period_s=0.001):
        import threading
        self.samples = []          # (perf_counter, sm_mhz, set of reasons)
        self.max_mhz = None
        self.source = None
        self.t0 = self.t1 = None
        self._halt = threading.Event()
        self._period = period_s
        self._thread = None
        uuid = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        if self._open_nvml(uuid):
            self.source = "nvml"
            self._thread = threading.Thread(target=self._run_nvml, daemon=True)
        else:
            self.source = "nvidia-smi"
            self._thread = threading.Thread(target=self._run_smi, args=(uuid,), daemon=True)
        self._thread.start()

    def _open_nvml(self, uuid):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            if uuid is None or lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                return False
            self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            self._lib, self._h = lib, h
            return True
        except Exception:
            return False

    def _run_nvml(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._halt.is_set():
            if (self._lib.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0 and
                    self._reasons_fn(self._h, ctypes.byref(rs)) == 0):
                names = {n for n, bit in self.BITS.items() if rs.value & bit}
                self.samples.append((time.perf_counter(), float(clk.value), names))
            time.sleep(self._period)

    def _run_smi(self, uuid):
        try:
            proc = subprocess.Popen(["nvidia-smi", f"--id={uuid}" if uuid else "--id=0",
                                     f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                                     "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                    text=True)
        except Exception:
            return
        while not self._halt.is_set():
            line = proc.stdout.readline()
            if not line:
                break
            parts = [x.strip() for x in line.split(",")]
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except (ValueError, IndexError):
                continue
            self.max_mhz = mx
            names = {n for n, v in zip(self.NAMES, parts[2:6]) if v.lower() == "active"}
            self.samples.append((time.perf_counter(), sm, names))
        proc.terminate()

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        self._halt.set()
        self._thread.join(timeout=5)
        if self.source == "nvml":
            try:
                self._lib.nvmlShutdown()
            except Exception:
                pass
        inside = [s for s in self.samples if self.t0 is not None and self.t0 <= s[0] <= self.t1]
        window = "timed region"
        if not inside and self.samples and self.t0 is not None:
            mid = 0.5 * (self.t0 + self.t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))]
            window = "nearest sample to a timed region shorter than the sampling period"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": self.source}
        reasons = set().union(*(s[2] for s in inside))
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "sm_min_mhz": min(s[1] for s in inside), "reasons": sorted(reasons),
                "samples": len(inside), "source": self.source, "window": window}


# --------------------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- CPU oracle
def oracle_sample(x, n_seq):
    """fp64 views of the first n_seq (b, h) sequences, each as a [1,T,1,*] problem batch."""
    B, T, H = x["g"].shape
    seqs = [(s // H, s % H) for s in range(min(n_seq, B * H))]
    out = []
    for b, h in seqs:
        sub = {n: to_f64(x[n][b:b + 1, :, h:h + 1].contiguous()) for n in ("q", "k", "v", "g", "beta")}
        sub["h0"] = None if x["h0"] is None else to_f64(x["h0"][b:b + 1, h:h + 1].contiguous())
        out.append(sub)
    return out


def run_oracle_sample(samples, threads):
    """Runs the oracle over the sampled sequences as one batch (stacked over H)."""
    import numpy as np

    from oracle import recurrence
    cat = lambda n: np.concatenate([s[n] for s in samples], axis=2)
    h0 = None if samples[0]["h0"] is None else np.concatenate([s["h0"] for s in samples], axis=1)
    t = time.perf_counter()
    recurrence.forward(cat("q"), cat("k"), cat("v"), cat("g"), cat("beta"), 1.0, h0, nthreads=threads)
    return time.perf_counter() - t


def cpu_baseline(x, w, budget_s):
    """The oracle on a bounded sample of the workload, on all host cores."""
    threads = os.cpu_count() or 1
    n_total = w.B * w.H
    n = min(n_total, max(1, threads))
    dt = run_oracle_sample(oracle_sample(x, n), threads)
    # grow the sample (up to the whole workload) to fill about budget_s seconds
    per_seq = dt / n
    n2 = int(min(n_total, max(n, budget_s / max(per_seq, 1e-9))))
    if n2 > n:
        n = n2
        dt = run_oracle_sample(oracle_sample(x, n), threads)
    # a sample shorter than the budget is repeated, the rate is the mean
    samples, reps = oracle_sample(x, n), 1
    while dt < budget_s and reps < 100:
        dt += run_oracle_sample(samples, threads)
        reps += 1
    tokens = reps * n * w.T / w.H     # B*T-equivalent tokens of the sample
    return {"value": tokens / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {n_total} (b,h) sequences of {w.name}, full T={w.T}, run {reps}x, "
                      f"fp64 token recurrence, {dt:.2f} s; tokens = sequences*T/H"}


# --------------------------------------------------------------------------- arms
def bench_reference(args, w, world, rank):
    if rank != 0:
        return
    x = make_workload(w)
    threads = os.cpu_count() or 1
    n_seq = min(w.B * w.H, max(1, threads))
    samples = oracle_sample(x, n_seq)
    for _ in range(args.warmup):
        run_oracle_sample(samples, threads)
    total = 0.0
    for _ in range(args.steps):
        total += run_oracle_sample(samples, threads)
    tokens = n_seq * w.T / w.H
    value = tokens * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {n_seq} of {w.B * w.H} (b,h) sequences of {w.name}, "
                                   f"full T={w.T}; tokens = sequences*T/H"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, args):
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V, "chunk": CHUNK,
            "io_dtype": w.dtype, "algo": args.algo, "l2": "flushed before every timed step (512 MiB write)",
            "parallelism": f"replica x{args.gpus}" if args.gpus > 1 else "single GPU"}


def bench_frontend(args, w, world, dev, flush):
    """The same workload with the input front-end in the kernels: q and k as
    drawn (unnormalised), g the raw per-token log decays, flags RAW_G and
    QK_L2NORM, scale K^-0.5. Timed like the main step (L2 flushed before each
    step, CUDA events on the launching stream)."""
    from gated_delta_rule_35_gb300 import chunk_fwd, native

    x = make_inputs(w.B, w.T, w.H, w.K, w.V, dtype=w.dtype, seed=w.seed, h0_std=w.h0_std,
                    g_mean=w.g_mean, g_div=w.g_div, beta_mean=w.beta_mean, raw=True)
    d = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    flags = native.flags_of(True, True)
    p = native.problem(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, args.algo, flags)
    ws = torch.empty(native.workspace_bytes(p), dtype=torch.uint8, device=dev)
    o = torch.empty((w.B, w.T, w.H, w.V), dtype=d["q"].dtype, device=dev)
    hf = torch.empty((w.B, w.H, w.K, w.V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    n = max(10, min(args.steps, 100))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]

    def step():
        chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.K ** -0.5, d["h0"], algo=args.algo,
                  workspace=ws, out=o, final_state=hf, stream=stream, raw_g=True, qk_l2norm=True)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    t = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / n / 1e3, world, dev)
    return {"workload": w.name + "_raw", "flags": ["RAW_G", "QK_L2NORM"], "steps_timed": n,
            "ms_per_step": 1e3 * t, "tokens_per_s": w.B * w.T * world / t,
            "kernels": native.launches(p), "gpu_launches": len(native.launches(p)) * n,
            "inputs": "q, k unnormalised N(0,1); g per-token log decays; scale K^-0.5"}


def bench_output_norm(args, w, world, dev, flush, d):
    """The same step with the gated RMSNorm output stage (gate and norm weight
    read, o normalised before its rounding; the tensor-core path runs each
    head's V tiles as a cluster). Timed like the main step."""
    from gated_delta_rule_35_gb300 import chunk_fwd, native
    from gated_delta_rule_35_gb300.inputs import make_output_norm

    gate, weight = make_output_norm(w.B, w.T, w.H, w.V, dtype=w.dtype, seed=w.seed)
    gate, weight = gate.to(dev), weight.to(dev)
    p = native.problem(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, args.algo)
    ws = torch.empty(native.workspace_bytes(p), dtype=torch.uint8, device=dev)
    o = torch.empty((w.B, w.T, w.H, w.V), dtype=d["q"].dtype, device=dev)
    hf = torch.empty((w.B, w.H, w.K, w.V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    n = max(10, min(args.steps, 100))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]

    def step():
        chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo=args.algo,
                  workspace=ws, out=o, final_state=hf, stream=stream, gate=gate,
                  norm_weight=weight, norm_eps=1e-6)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    t = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / n / 1e3, world, dev)
    kernels = native.launches(p)   # the plain call's kernels, the stage inside them
    return {"workload": w.name + "_gated_rmsnorm", "steps_timed": n, "ms_per_step": 1e3 * t,
            "tokens_per_s": w.B * w.T * world / t, "kernels": kernels,
            "gpu_launches": len(kernels) * n,
            "extra_bytes_per_token_head": 2 * w.V,
            "inputs": "gate N(0,1) in the I/O dtype, norm weight 1 + 0.1 N(0,1), eps 1e-6"}


def bench_per_channel(args, w, world, dev, flush):
    """Per-channel (KDA) decay: the chunked step on the same shape (one decay per
    key channel; 'auto' runs bf16 on the tensor-core form, the CUDA-core
    pipeline timed beside it) and the decode step on the decode workload with a
    per-channel gamma [B,T,H,K]."""
    from gated_delta_rule_35_gb300 import chunk_fwd, decode_step, native

    x = make_inputs(w.B, w.T, w.H, w.K, w.V, dtype=w.dtype, seed=w.seed, h0_std=w.h0_std,
                    per_channel=True)
    d = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    flags = native.flags_of(per_channel=True)
    p = native.problem(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, "auto", flags)
    ws = torch.empty(native.workspace_bytes(p), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn, n, flush_each):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for _ in range(args.warmup):
            if flush_each:
                flush.zero_()
            fn()
        torch.cuda.synchronize(dev)
        for a, b in evs:
            if flush_each:
                flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / n / 1e3, world, dev)

    t_chunk = timed(lambda: chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"],
                                      workspace=ws, stream=stream, per_channel_decay=True),
                    max(5, min(args.steps, 20)), True)
    t_simt = timed(lambda: chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo="simt",
                                     workspace=ws, stream=stream, per_channel_decay=True),
                   5, True)
    # algorithmic bytes: q, k, v in, o out, g (fp32 per channel) and beta in,
    # h0 in and h_final out
    es_c = DSIZE[w.dtype]
    chunk_bytes = (w.B * w.T * w.H * ((2 * w.K + 2 * w.V) * es_c + 4 * w.K + 4)
                   + w.B * w.H * w.K * w.V * 4 * (2 if w.h0_std else 1))
    wd = DECODE_WORKLOADS[DECODE_WORKLOAD]
    y = make_inputs(wd.B, wd.T, wd.H, wd.K, wd.V, dtype=wd.dtype, seed=wd.seed, h0_std=wd.h0_std,
                    chunk=1, per_channel=True)
    dy = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in y.items()}
    o = torch.empty((wd.B, wd.T, wd.H, wd.V), dtype=dy["q"].dtype, device=dev)
    t_dec = timed(lambda: decode_step(dy["q"], dy["k"], dy["v"], dy["g"], dy["beta"], dy["h0"],
                                      1.0, out=o, stream=stream, per_channel_decay=True),
                  max(10, min(args.steps, 100)), False)
    heads = wd.B * wd.H
    es = DSIZE[wd.dtype]
    nbytes = heads * wd.K * wd.V * 8 + heads * wd.T * ((2 * wd.K + 2 * wd.V) * es + 4 * wd.K + 4)
    peaks = load_peaks()
    return {"chunked": {"workload": w.name + "_per_channel", "ms_per_step": 1e3 * t_chunk,
                        "tokens_per_s": w.B * w.T * world / t_chunk, "kernels": native.launches(p),
                        "cuda_core_ms_per_step": 1e3 * t_simt,
                        "algorithmic_bytes_per_step": chunk_bytes,
                        "pipeline_roofline": {"bound": "hbm", "achieved": chunk_bytes / t_chunk / 1e9,
                                              "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                              "frac": chunk_bytes / t_chunk / 1e9 / peaks["hbm_gbs"]}},
            "decode": {"workload": wd.name + "_per_channel", "ms_per_call": 1e3 * t_dec,
                       "algorithmic_bytes_per_call": nbytes,
                       "roofline": {"bound": "hbm", "achieved": nbytes / t_dec / 1e9,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": nbytes / t_dec / 1e9 / peaks["hbm_gbs"]}}}


def bench_decode(args, world, dev):
    """The decode step on its own workload: one token for each of B*H heads, the
    state [B,H,K,V] fp32 read and written in place once per call. The state
    (537 MB) is larger than L2, so no flush is needed between calls."""
    from gated_delta_rule_35_gb300 import decode_step, native

    w = DECODE_WORKLOADS[DECODE_WORKLOAD]
    x = make_workload(w)
    d = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    state = d.pop("h0")
    o = torch.empty((w.B, w.T, w.H, w.V), dtype=d["q"].dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    kernels = native.decode_launches(native.problem(w.B, w.T, w.H, w.K, w.V, d["q"].dtype))
    n = max(10, min(args.steps, 100))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]

    def call():
        decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, 1.0, out=o, stream=stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    for a, b in evs:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize(dev)
    t = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / n / 1e3, world, dev)
    es = DSIZE[w.dtype]
    heads = w.B * w.H
    nbytes = heads * w.K * w.V * 4 * 2 + heads * w.T * ((2 * w.K + 2 * w.V) * es + 8)
    peaks = load_peaks()
    achieved = nbytes / t / 1e9
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V,
            "calls_timed": n, "ms_per_call": 1e3 * t, "tokens_per_s": w.B * w.T * world / t,
            "kernels": kernels, "gpu_launches": len(kernels) * n,
            "l2": "not flushed: the 537 MB state exceeds L2",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": ncu_traffic(kernels[0], w.name) if kernels else None,
                         "algorithmic_bytes_per_call": nbytes, "peak_source": peaks["_source"]}}


def step_stats(ms):
    """Median, mean and the 10th / 90th percentiles of per-step times (ms)."""
    xs = sorted(ms)
    pick = lambda f: xs[min(len(xs) - 1, max(0, int(round(f * (len(xs) - 1)))))]
    return {"steps": len(xs), "median_ms": statistics.median(xs), "mean_ms": statistics.fmean(xs),
            "p10_ms": pick(0.1), "p90_ms": pick(0.9), "min_ms": xs[0], "max_ms": xs[-1]}


def pipeline_roofline(w, t_step_s, peaks, has_h0, kernels=None):
    """The whole step against max(flops / bf16 peak, compulsory bytes / HBM).
    With the step's kernels: the DRAM bytes the design actually moves per step
    (the committed ncu records of every kernel, when all are current), against
    the compulsory bytes and as a rate against HBM."""
    units = w.B * w.T * w.H
    hbytes = (2 if has_h0 else 1) * w.B * w.H * w.K * w.V * 4
    F = flops_per_token_head(w.K, w.V) * units
    Bt = bytes_per_token_head(w.K, w.V, DSIZE[w.dtype]) * units + hbytes
    t_f, t_b = F / (peaks["bf16_tflops"] * 1e12), Bt / (peaks["hbm_gbs"] * 1e9)
    t_roof = max(t_f, t_b)
    out = {"t_roof_us": 1e6 * t_roof, "t_meas_us": 1e6 * t_step_s, "frac": t_roof / t_step_s,
           "flops": F, "bytes": Bt, "bound": "hbm" if t_b >= t_f else "tensor",
           "peak_source": peaks["_source"]}
    if kernels:
        parts = [ncu_traffic(k, w.name) for k in kernels]
        moved = None if any(x is None for x in parts) else sum(parts)
        out["design_traffic"] = moved
        out["design_traffic_over_compulsory"] = None if moved is None else moved / Bt
        out["design_traffic_frac_of_hbm"] = None if moved is None else moved / t_step_s / 1e9 / peaks["hbm_gbs"]
    return out


PAIR_TIMING = ("the 64-column grid runs beside the wide grid's last wave, which a marker between them "
               "would serialise: the pair's time is the unmarked steps' time minus the other kernels' marked time")


def dominant(kernels, per_kernel, steps_total=None):
    """The kernel that takes most of the step, and its time. When the forward
    work is split (whole waves on the wide kernel, the remaining heads on the
    64-column kernel right behind it) the two count as one launch over all
    token-heads. With steps_total (the same steps timed without markers) that
    launch's time is the steps' time minus the other kernels' (PAIR_TIMING),
    when that is the smaller."""
    names, times = list(kernels), list(per_kernel)
    if "gdn_wide_tc_kernel" in names and "gdn_fused_tc_kernel" in names:
        i, j = names.index("gdn_wide_tc_kernel"), names.index("gdn_fused_tc_kernel")
        merged = times[i] + times[j]
        if steps_total is not None:
            rest = sum(t for k, t in enumerate(times) if k not in (i, j))
            merged = min(merged, steps_total - rest)
        names = [n for k, n in enumerate(names) if k not in (i, j)] + ["gdn_wide_tc_kernel+gdn_fused_tc_kernel"]
        times = [t for k, t in enumerate(times) if k not in (i, j)] + [merged]
    k = max(range(len(names)), key=lambda q: times[q])
    return names[k], times[k]


def kernel_roofline(name, w, t_launch_s, peaks, has_h0):
    """The dominant kernel against its bound: compulsory bytes of the launch
    (per token-head, plus the fp32 states it reads and writes) over its time."""
    units = w.B * w.T * w.H
    bound, model = KERNEL_MODEL.get(name, ("hbm", _fused))
    bpt, fpt = model(w.K, w.V, DSIZE[w.dtype])
    state_bytes = ((2 if has_h0 else 1) * w.B * w.H * w.K * w.V * 4) if bound == "hbm" else 0
    if bound == "hbm":
        achieved, peak, unit = (bpt * units + state_bytes) / t_launch_s / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "tensor":
        achieved, peak, unit = fpt * units / t_launch_s / 1e12, peaks["bf16_tflops_sustained"], "TFLOP/s"
    else:   # fp32 FMA pipe: SMs x lanes x 2 flop x max SM clock
        peak = SMS * FP32_LANES * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        achieved, unit = fpt * units / t_launch_s / 1e12, "TFLOP/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": ncu_traffic(name, w.name), "kernel": name,
            "kernel_ms": 1e3 * t_launch_s, "peak_source": peaks["_source"],
            "algorithmic_per_token_head": {"bytes": bpt, "flops": fpt},
            "algorithmic_state_bytes": state_bytes}


def time_steps(args, w, dev, flush, steps, warmup, per_kernel=True, d=None):
    """Device times of `steps` full forwards of workload w (L2 flushed before
    each): per-step times from events at the ends of each step only, then
    (per_kernel) the same steps with a marker after every kernel."""
    from gated_delta_rule_35_gb300 import chunk_fwd, native

    if d is None:
        x = make_workload(w)
        d = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    p = native.problem(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, args.algo)
    kernels = native.launches(p)
    nk = len(kernels)
    ws = torch.empty(native.workspace_bytes(p), dtype=torch.uint8, device=dev)
    o = torch.empty((w.B, w.T, w.H, w.V), dtype=d["q"].dtype, device=dev)
    hf = torch.empty((w.B, w.H, w.K, w.V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["h0"], algo=args.algo,
                  workspace=ws, out=o, final_state=hf, stream=stream,
                  events=None if evs is None else [e.cuda_event for e in evs])

    bounds = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    return {"d": d, "kernels": kernels, "step": step, "bounds": bounds, "stream": stream,
            "flush": flush, "nk": nk, "per_kernel": per_kernel}


def run_timed(t, dev, clocks=None):
    """Runs the prepared steps; returns (per-step ms list, per-kernel ms sums, wall s)."""
    stream, flush, step, bounds, nk = t["stream"], t["flush"], t["step"], t["bounds"], t["nk"]
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.mark_start()
    wall0 = time.perf_counter()
    for a, b in bounds:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if clocks is not None:
        clocks.mark_end()
    step_ms = [a.elapsed_time(b) for a, b in bounds]
    per_kernel = [0.0] * nk
    if t["per_kernel"]:
        marks = []
        for _ in bounds:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
            for e in evs:
                e.record(stream)      # creates the underlying cudaEvent_t
            flush.zero_()
            step(evs)
            marks.append(evs)
        torch.cuda.synchronize(dev)
        for evs in marks:
            for j in range(nk):
                per_kernel[j] += evs[j].elapsed_time(evs[j + 1])
    return step_ms, per_kernel, wall


def bench_other_workloads(args, main_w, dev, flush, peaks, world):
    """Every other bf16 workload, device-timed like the headline (median of at
    least 50 steps, L2 flushed before each), with its pipeline and kernel
    roofline fractions."""
    out = {}
    for name, w in WORKLOADS.items():
        if name == main_w.name or w.dtype != "bf16":
            continue
        t = time_steps(args, w, dev, flush, max(50, args.steps), args.warmup)
        step_ms, per_kernel, _ = run_timed(t, dev)
        st = step_stats(step_ms)
        t_step = max_over_ranks(st["median_ms"] / 1e3, world, dev)
        kernels, nk = t["kernels"], t["nk"]
        dom_name, dom_t = dominant(kernels, per_kernel, sum(step_ms))
        has_h0 = t["d"]["h0"] is not None
        out[name] = {
            "tokens_per_s": w.B * w.T * world / t_step, "ms_per_step": 1e3 * t_step,
            "timing": st,
            "pipeline_roofline": pipeline_roofline(w, t_step, peaks, has_h0, kernels),
            "roofline": kernel_roofline(dom_name, w, dom_t / len(step_ms) / 1e3, peaks, has_h0),
            "per_kernel_ms": {k: per_kernel[j] / len(step_ms) for j, k in enumerate(kernels)},
            "kernels": kernels, "gpu_launches": nk * len(step_ms),
        }
        del t
        torch.cuda.empty_cache()
    return out


def bench_ours(args, w, world, rank, local):
    from gated_delta_rule_35_gb300 import chunk_fwd_host

    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    x = make_workload(w)
    d = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    peaks = load_peaks()
    t = time_steps(args, w, dev, flush, args.steps, args.warmup, d=d)
    kernels, nk = t["kernels"], t["nk"]
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev)
    time.sleep(0.05)   # let the sampler take its first readings
    step_ms, per_kernel, wall = run_timed(t, dev, clocks)
    clk = clocks.stop()
    barrier(world)
    torch.cuda.synchronize(dev)

    st = step_stats(step_ms)
    # the value: B*T tokens per median step, max over ranks
    t_step = max_over_ranks(st["median_ms"] / 1e3, world, dev)
    tokens_step = w.B * w.T
    value = tokens_step * world / t_step
    has_h0 = d["h0"] is not None

    dom_name, dom_t = dominant(kernels, per_kernel, sum(step_ms))
    roofline = kernel_roofline(dom_name, w, dom_t / args.steps / 1e3, peaks, has_h0)
    roofline["share"] = dom_t / max(sum(per_kernel), 1e-12)
    if "+" in dom_name:
        roofline["kernel_ms_how"] = PAIR_TIMING
    pipeline = pipeline_roofline(w, t_step, peaks, has_h0, kernels)

    # end to end through the public host-tensor API: H2D inputs, forward, D2H o and h_final
    hx = {n: (t_.pin_memory() if isinstance(t_, torch.Tensor) else t_) for n, t_ in x.items()}
    h2d = sum(t_.numel() * t_.element_size() for n, t_ in hx.items() if isinstance(t_, torch.Tensor))
    d2h = w.B * w.T * w.H * w.V * DSIZE[w.dtype] + w.B * w.H * w.K * w.V * 4
    e2e_steps = max(1, min(args.steps, 20))
    # pinned outputs kept across steps, as a serving loop keeps its buffers
    ho = torch.empty((w.B, w.T, w.H, w.V), dtype=d["q"].dtype, pin_memory=True)
    hhf = torch.empty((w.B, w.H, w.K, w.V), dtype=torch.float32, pin_memory=True)
    for _ in range(2):
        chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["g"], hx["beta"], 1.0, hx["h0"], algo=args.algo,
                       device=dev, out=ho, final_state=hhf)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["g"], hx["beta"], 1.0, hx["h0"], algo=args.algo,
                       device=dev, out=ho, final_state=hhf)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e = {"value": tokens_step * e2e_steps * world / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    del hx, ho, hhf, t
    torch.cuda.empty_cache()

    fw = WORKLOADS[FEATURE_WORKLOAD]
    others = None if args.no_other_workloads else bench_other_workloads(args, w, dev, flush, peaks, world)
    dec = None if args.no_decode else bench_decode(args, world, dev)
    fe = None if args.no_frontend else bench_frontend(args, fw, world, dev, flush)
    fd = None
    if not args.no_output_norm or not args.no_per_channel:
        fx = make_workload(fw.name)
        fd = {n: (t_.to(dev) if isinstance(t_, torch.Tensor) else t_) for n, t_ in fx.items()}
    on = None if args.no_output_norm else bench_output_norm(args, fw, world, dev, flush, fd)
    if on is not None and others and fw.name in others:
        on["plain_ms_per_step"] = others[fw.name]["ms_per_step"]
        on["ratio_to_plain"] = on["ms_per_step"] / on["plain_ms_per_step"]
    # the same on the headline workload (its grid takes the 128-column kernel)
    on_head = None
    if not args.no_output_norm:
        on_head = bench_output_norm(args, w, world, dev, flush, d)
        on_head["plain_ms_per_step"] = 1e3 * t_step
        on_head["ratio_to_plain"] = on_head["ms_per_step"] / on_head["plain_ms_per_step"]
    pcd = None if args.no_per_channel else bench_per_channel(args, fw, world, dev, flush)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x, w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16-in/f32-acc" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_of(w, args),
            "timing": dict(st, statistic="value and ms_per_step use the median step"),
            "token_heads_per_s": value * w.H,
            "roofline": roofline, "pipeline_roofline": pipeline,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": nk * args.steps,
            "kernels": kernels,
            "per_kernel_ms": {k: per_kernel[j] / args.steps for j, k in enumerate(kernels)},
            "per_kernel_note": "second pass of the same steps with a marker after every kernel",
            "clocks": clk, "wall_timed_s": wall, "workloads": others,
            "decode": dec, "frontend": fe, "output_norm": on, "output_norm_headline": on_head,
            "per_channel": pcd,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=BENCH_WORKLOAD, choices=list(WORKLOADS))
    ap.add_argument("--algo", default="auto", choices=["auto", "simt", "tc", "tc1"])
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload with this many sequences instead of its own B "
                         "(a slice of the same shape, for profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-step measurement")
    ap.add_argument("--no-frontend", action="store_true",
                    help="skip the in-kernel front-end measurement")
    ap.add_argument("--no-output-norm", action="store_true",
                    help="skip the gated RMSNorm output-stage measurement")
    ap.add_argument("--no-per-channel", action="store_true",
                    help="skip the per-channel (KDA) decay measurements")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the device-timed lines of the other bf16 workloads")
    ap.add_argument("--cpu-seconds", type=float, default=5.0,
                    help="target CPU time of the oracle baseline sample")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = WORKLOADS[args.workload]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}_slice_b{args.batch}")
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        bench_reference(args, w, world, rank)
    else:
        bench_ours(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
