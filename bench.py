#!/usr/bin/env python3
"""Benchmark of the sequential-MTP hot path on GB300.

One step = the whole hot path over one batch of synthetic input:
  * mtp_chain_loss on the mid-size MTP-chain workload (B=8 packed rows of
    T=1024, d=1024, 16x64 heads, SwiGLU ffn 2816, V=32000, D=3 sequential
    depths, Zipf(1.1) tokens, geometric documents of mean length 256): the
    main term plus the masked CE of every depth and the assembled loss;
  * spec_verify on the verification workload (64 requests, gamma=4 drafts,
    V=129280, target/draft rows built with mean overlap ~0.70).

value = MTP-chain tokens per step (sum over depths k of B*(T-k) rows) / the
step's device time (CUDA events on the launching stream, max over ranks,
times the number of ranks).  spec_verify rows/s (R*(gamma+1) rows per call)
is reported beside it.  L2 is flushed (256 MiB written, then read back, so
that no dirty line of the flush is left for the timed kernels to write back)
between timed steps,
outside the events.  `roofline` covers the dominant kernel (the shared-head
GEMM with the fused online-softmax CE epilogue); `cpu_baseline` times the
CPU oracle on a bounded sample of the same workload.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) each rank runs its own batch (weak scaling); the one
exchange is the data-parallel all-reduce of the per-term (sum, count) pairs
before the loss is assembled.
"""
from __future__ import annotations

import argparse
import dataclasses
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

METRIC = "MTP-chain tokens/s (all depths) + spec_verify rows/s, % of roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HEAD_PROFILE = os.path.join(ROOT, "profiles", "head_ce_gemm_mid_bf16.md")
GEMM_SOURCES = [os.path.join(ROOT, "deepseek_sequential_mtp_gb300", "csrc", f)
                for f in ("gemm_tc.cu", "gemm_tc.cuh")]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference", "cpu-one-core"], default="ours",
                    help="cpu-one-core: internal, the single-core oracle timing (run in a child process)")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-max-len", type=int, default=256, help=argparse.SUPPRESS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--draft-steps", type=int, default=30)
    ap.add_argument("--train-steps", type=int, default=5, help="timed training steps (0 = off)")
    ap.add_argument("--c3-steps", type=int, default=4, help="timed calls of the DeepSeek-V3-width section (0 = off)")
    ap.add_argument("--draft-gamma", type=int, default=4, help="steps of the recurrent draft round (<= 1: off)")
    ap.add_argument("--no-draft-fp8", dest="draft_fp8", action="store_false",
                    help="skip the draft step with FP8 block-scaled module weights")
    ap.add_argument("--only-c3", action="store_true",
                    help="run only the DeepSeek-V3-width section (profiling its kernels) and print its record")
    ap.add_argument("--draft-requests", type=int, default=32,
                    help="requests of the draft-step section (32 = the measured workload; fewer for profiling)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(peaks):
    """Dense bf16 peak for kernels timed inside a step of a few milliseconds: the burst figure
    (the SM clock stays at its maximum over such a step; the sustained figure was measured over
    a seconds-long loop at a lower, power-capped clock)."""
    return float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))


def step_roofline(cfg, seg, supervised_rows, verify_bytes, step_ms, peaks):
    """Roofline time of one step: the sum over its kernels of max(FLOPs / tensor peak,
    bytes / HBM bandwidth), counting algorithmic work only (rows with state at each depth,
    supervised rows for the heads, visible (query, key) pairs for attention).  frac = that
    time over the measured step time."""
    import numpy as np
    P = tensor_peak(peaks) * 1e12
    BW = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])) * 1e9
    d, f, V, D = cfg.d, cfg.ffn, cfg.V, cfg.D
    B, T = seg.shape
    t_idx = np.arange(T)
    flops = {"gemm_block": 0.0, "attention": 0.0}
    bytes_ = {"norms_prologue": 0.0, "attention": 0.0}
    for k in range(1, D + 1):
        # state-valid rows: t + k < T, s[t] >= 0, s[t + k] == s[t]; attention pairs: keys
        # from the segment start to t (all state-valid, contiguous segments)
        valid = np.zeros((B, T), dtype=bool)
        valid[:, :T - k] = (seg[:, :T - k] >= 0) & (seg[:, k:] == seg[:, :T - k])
        rows = float(valid.sum())
        start = np.zeros((B, T), dtype=np.int64)
        for b in range(B):
            new = np.r_[True, seg[b, 1:] != seg[b, :-1]]
            start[b] = np.maximum.accumulate(np.where(new, t_idx, 0))
        pairs = float(((t_idx[None, :] - start + 1) * valid).sum())
        flops["gemm_block"] += rows * (4 * d * d + 6 * d * d + 2 * d * d + 4 * d * f + 2 * d * f)
        flops["attention"] += 4.0 * d * pairs
        bytes_["attention"] += rows * (3 * d + d) * 2.0  # read q, k, v; write o (bf16)
        # prologue (gather E row, read h, write c = 8 d bytes) and the two block norms (4 d each)
        bytes_["norms_prologue"] += rows * (8 * d + 2 * 4 * d)
    heads = float(np.sum(supervised_rows))
    flops["head_ce"] = 2.0 * d * V * heads
    bytes_["head_norms"] = 4.0 * d * heads
    bytes_["spec_verify"] = float(verify_bytes)
    terms = {k: v / P * 1e3 for k, v in flops.items() if k not in bytes_}
    terms.update({k: v / BW * 1e3 for k, v in bytes_.items() if k not in flops})
    for k in set(flops) & set(bytes_):  # attention: whichever bound is larger
        terms[k] = max(flops[k] / P, bytes_[k] / BW) * 1e3
    t_ms = sum(terms.values())
    return {"roofline_ms": t_ms, "step_ms": step_ms, "frac": t_ms / step_ms,
            "terms_ms": terms, "tensor_peak_tflops": P / 1e12, "hbm_gbs": BW / 1e9,
            "note": "sum over kernels of max(FLOPs / burst bf16 peak, bytes / HBM bandwidth); "
                    "each term here is bound by one of the two"}


def code_lines(text):
    """The code of a C++/CUDA source: // comments, surrounding blanks and empty lines dropped
    (so a comment edit does not count as a kernel change)."""
    out = []
    for line in text.splitlines():
        i = line.find("//")
        while i >= 0 and line.count('"', 0, i) % 2 == 1:  # a // inside a string literal
            i = line.find("//", i + 2)
        if i >= 0:
            line = line[:i]
        line = line.strip()
        if line:
            out.append(line)
    return "\n".join(out)


def gemm_source_hash():
    """Hash of the GEMM core's code (gemm_tc.cu and .cuh, comments excluded): the key that ties
    the committed ncu capture to the kernel it was taken on."""
    h = hashlib.sha256()
    for p in GEMM_SOURCES:
        with open(p, encoding="utf-8") as fh:
            h.update(code_lines(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """Per-launch DRAM traffic of the head GEMM from the committed ncu summary,
    or None when it is absent or was taken on other kernel sources."""
    try:
        text = open(HEAD_PROFILE).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, _, v = line[2:].partition(":")
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha256") != gemm_source_hash():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------
# nvidia-smi clock sampling during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU oracle baseline (the reference arm and the cpu_baseline leg)
# --------------------------------------------------------------------------
def first_segment_window(seg_row, max_len):
    s = 0
    while s < len(seg_row) and seg_row[s] == -1:
        s += 1
    e = s
    while e < len(seg_row) and seg_row[e] == seg_row[s] and e - s < max_len:
        e += 1
    return s, e


def oracle_sample(cfg, batch, h0, W, b, max_len):
    """Runs the oracle's chain + loss on one whole-segment prefix of packed row
    b; returns (tokens processed, seconds)."""
    import numpy as np
    from oracle import chain as oc
    s0, s1 = first_segment_window(batch["seg"][b], max_len)
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=cfg.D, eps=cfg.eps, rope_base=cfg.rope_base)
    t = time.perf_counter()
    out = oc.chain_forward_loss(batch["tokens"][b:b + 1, s0:s1], batch["seg"][b:b + 1, s0:s1],
                                batch["pos"][b:b + 1, s0:s1], h0[b:b + 1, s0:s1], W, dims,
                                precision="bf16", lam=cfg.lam)
    dt = time.perf_counter() - t
    tokens = int(np.isfinite(out["h"][:, 0, :, 0]).sum())  # state rows over all depths
    return tokens, dt


def cpu_oracle_inputs(cfg, seed):
    from deepseek_sequential_mtp_gb300 import synth
    from oracle import chain as oc
    batch = synth.make_batch(cfg, seed)
    h0 = synth.make_h0(cfg, seed).float().numpy()
    W = oc.weights_to_numpy(synth.make_weights(cfg, seed + 1))
    return batch, h0, W


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def oracle_rate(cfg, seed, seconds, max_len):
    batch, h0, W = cpu_oracle_inputs(cfg, seed)
    tok_total, t_total, n = 0, 0.0, 0
    while t_total < seconds or n == 0:
        tok, dt = oracle_sample(cfg, batch, h0, W, n % cfg.B, max_len)
        tok_total += tok
        t_total += dt
        n += 1
    return tok_total / t_total, n, t_total


def one_core_rate(seconds, max_len):
    """The same oracle sample in a child process pinned to one core with one BLAS/OpenMP
    thread (a fresh process, so the thread pools start with that setting)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "cpu-one-core", "--cpu-seconds", str(seconds),
           "--cpu-max-len", str(max_len)]
    first = sorted(os.sched_getaffinity(0))[0] if hasattr(os, "sched_getaffinity") else None

    def pin():
        if first is not None:
            os.sched_setaffinity(0, {first})

    try:
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600, preexec_fn=pin)
        return json.loads(res.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError) as exc:
        return {"error": f"one-core run failed: {exc}"}


def cpu_baseline(cfg, seed, seconds, max_len=256):
    value, n, t_total = oracle_rate(cfg, seed, seconds, max_len)
    one = one_core_rate(max(2.0, seconds / 2), max_len)
    return {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "cpu_model": cpu_model(),
            "one_core": one,
            "sample": f"{n} whole-segment prefixes (<= {max_len} rows) of the mid workload's packed rows, "
                      f"all {cfg.D} depths + main and depth heads, fp64 numpy with bf16 storage rounding; "
                      f"{t_total:.1f} s on all cores (numpy's threaded BLAS); one_core: the same sample "
                      f"in a process pinned to one core with one BLAS thread"}


def run_one_core(args):
    from deepseek_sequential_mtp_gb300 import synth
    value, n, t_total = oracle_rate(synth.MID_BF16, 1, args.cpu_seconds, args.cpu_max_len)
    print(json.dumps({"value": value, "unit": UNIT, "cores": 1, "samples": n, "seconds": t_total}), flush=True)


# --------------------------------------------------------------------------
# Reference arm: the CPU oracle, timed on the host cores
# --------------------------------------------------------------------------
def run_reference(args):
    from deepseek_sequential_mtp_gb300 import synth
    rank, _, world = dist_env()
    if rank != 0:
        return
    cfg = synth.MID_BF16
    batch, h0, W = cpu_oracle_inputs(cfg, 1)
    per_step_rows = 32  # bounded sample per step so K + W steps end within minutes
    for i in range(args.warmup):
        oracle_sample(cfg, batch, h0, W, i % cfg.B, per_step_rows)
    tok_total, t_total = 0, 0.0
    for i in range(args.steps):
        tok, dt = oracle_sample(cfg, batch, h0, W, i % cfg.B, per_step_rows)
        tok_total += tok
        t_total += dt
    value = tok_total / t_total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"per step one whole-segment prefix (<= {per_step_rows} rows) of a packed "
                                       f"row of the mid workload, all depths + heads, fp64 numpy"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config():
    return {"workload": "mtp_chain mid_bf16_D3 (B=8, T=1024, d=1024, 16x64 heads, SwiGLU ffn=2816, V=32000, "
                        "D=3, Zipf(1.1) tokens, geometric docs mean 256, lambda=0.3, main+3 depth CE) + "
                        "spec_verify (R=64, gamma=4, V=129280, alpha~0.70)",
            "global_batch": 8, "seq_len": 1024, "parallelism": "dp (independent packed rows per rank)",
            "l2": "flushed between timed steps (256 MiB written then read, outside the step events)"}


class L2Flush:
    """Evicts L2 (126 MB on GB300) between timed calls: writes a 256 MiB
    buffer, then reads it back so the cache ends up holding clean lines of the
    flush buffer rather than dirty ones the next kernel would have to write
    back."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(256 * 1024 * 1024 // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        import torch
        self.buf.zero_()
        torch.sum(self.buf, dim=0, out=self.sink)


# --------------------------------------------------------------------------
# Our arm
# --------------------------------------------------------------------------
def run_ours(args):
    import numpy as np
    import torch

    from deepseek_sequential_mtp_gb300 import build as mtp_build
    from deepseek_sequential_mtp_gb300 import dp, lib, synth

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    mtp_build.build()
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    if args.only_c3:
        res = measure_dsv3(args, dev, rank, load_peaks()[0])
        if rank == 0:
            print(json.dumps({"dsv3_width": res}), flush=True)
        return
    cfg = synth.MID_BF16
    vcfg = synth.VERIFY_C4
    seed = 1 + 1000 * rank

    # inputs resident in HBM
    batch = synth.make_batch(cfg, seed)
    x = {k: torch.from_numpy(v).to(dev) for k, v in batch.items()}
    x["h0"] = synth.make_h0(cfg, seed, device=dev)
    weights = synth.make_weights(cfg, seed + 1, device=dev)
    vin = synth.make_verify_inputs(vcfg, seed, device=dev)
    chain = lib.Chain(cfg, weights, device=dev)
    out = {"sums_counts": torch.empty(2 * (cfg.D + 1), dtype=torch.float64, device=dev),
           "losses": torch.empty(cfg.D + 2, dtype=torch.float32, device=dev)}
    K, W = args.steps, args.warmup
    KB = min(K, 20)  # steps of the per-kernel breakdown pass
    vouts = torch.empty((K + W + KB, 4, vcfg.R), dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    global_losses = torch.empty(cfg.D + 2, dtype=torch.float32, device=dev)

    def step(i):
        chain.loss(x["tokens"], x["seg"], x["pos"], x["h0"], den="fixed", with_main=True, out=out)
        if world > 1:
            dp.allreduce_sums_counts(out["sums_counts"])
            lib.loss_assemble(out["sums_counts"], cfg.D, dp.global_positions(cfg.B, cfg.T), cfg.lam, "fixed",
                              True, losses=global_losses)
        vo = vouts[i]
        lib.spec_verify(vin["p"], vin["q"], vin["draft"], seed=7 + rank, offset=i,
                        out={"accepted": vo[0], "next_token": vo[1], "n_emit": vo[2], "status": vo[3]})

    for i in range(W):
        flush()
        step(i)
    torch.cuda.synchronize()
    lib.check_errors()

    # only the dominant kernel's event timer is armed in the timed loop, and only in a few evenly
    # spaced steps: an event record between two kernels costs ~2 us of stream time and stops the
    # next launch from starting while its predecessor drains (programmatic dependent launch)
    launches_per_step = (("head_ce_gemm", cfg.D + 1), ("gate_up_gemm", cfg.D), ("down_gemm", cfg.D),
                         ("qkv_gemm", cfg.D), ("o_gemm", cfg.D), ("proj_gemm", cfg.D), ("attention", cfg.D),
                         ("spec_verify", 1), ("prologue", cfg.D))
    n_sampled = min(K, 4)
    sampled = {(j * K) // n_sampled: lib.KernelTimer("head_ce_gemm", cfg.D + 1) for j in range(n_sampled)}
    torch.cuda.synchronize()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    clocks = ClockSampler(visible[local_rank] if len(visible) > local_rank and visible[local_rank] else str(local_rank))
    clocks.start()
    launches0 = lib.kernel_launches()
    t_wall0 = time.perf_counter()
    for i in range(K):
        flush()
        if i in sampled:
            sampled[i].arm()
        ev0[i].record()
        step(W + i)
        ev1[i].record()
        if i in sampled:
            lib.KernelTimer.disarm_all()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    launches = lib.kernel_launches() - launches0
    clk = clocks.stop()
    lib.KernelTimer.disarm_all()
    lib.check_errors()

    step_ms = sum(a.elapsed_time(b) for a, b in zip(ev0, ev1)) / K
    step_ms_t = torch.tensor([step_ms], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(step_ms_t, op=torch.distributed.ReduceOp.MAX)
    step_ms_max = float(step_ms_t.item())
    tokens_per_step = sum(cfg.B * (cfg.T - k) for k in range(1, cfg.D + 1))
    value = world * tokens_per_step / (step_ms_max / 1e3)

    head_ms = [x for t in sampled.values() for x in t.durations_ms()]  # inside the timed region

    # per-kernel breakdown: a separate pass of KB steps with every kernel class's timer armed
    btimers = {name: lib.KernelTimer(name, n * KB) for name, n in launches_per_step}
    torch.cuda.synchronize()
    for t in btimers.values():
        t.arm()
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b_ms = 0.0
    for i in range(KB):
        flush()
        b0.record()
        step(W + K + i)
        b1.record()
        b1.synchronize()
        b_ms += b0.elapsed_time(b1)
    lib.KernelTimer.disarm_all()
    lib.check_errors()
    kern = {name: t.durations_ms() for name, t in btimers.items()}
    kern["head_ce_gemm"] = head_ms
    kern_steps = {name: KB for name in kern}
    kern_steps["head_ce_gemm"] = n_sampled
    counts = out["sums_counts"][1::2].cpu().numpy()  # supervised rows per term (same every step)
    peaks, peak_src = load_peaks()
    # algorithmic FLOPs of the head GEMM: 2 d V per supervised row, for main + each depth
    head_flops_step = 2.0 * cfg.d * cfg.V * float(counts.sum())
    head_ms_step = sum(head_ms) / n_sampled
    head_launch_flops = head_flops_step / (cfg.D + 1)
    head_launch_ms = head_ms_step / (cfg.D + 1)
    achieved = head_launch_flops / (head_launch_ms / 1e3) / 1e12
    peak = tensor_peak(peaks)
    traffic = recorded_traffic()
    roofline = {"bound": "tensor", "kernel": "gemm_tc_kernel<256, EPI_CE> (shared head + online CE)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic,
                "peak_source": "bf16_tflops (burst) of measured MEASURED_PEAKS.json: the kernel runs inside "
                               "a ~2 ms step at the maximum SM clock" if peak_src == "measured"
                               else "fallback 1.9 PFLOP/s burst",
                "algorithmic_flops_per_launch": head_launch_flops, "avg_launch_ms": head_launch_ms}

    # per-kernel table: algorithmic FLOPs per step and achieved TFLOP/s
    M = cfg.B * cfg.T
    d, f = cfg.d, cfg.ffn
    state_rows = float(tokens_per_step)  # rows with state over depths (upper bound used for the metric)
    per_row = {"gate_up_gemm": 4 * d * f, "down_gemm": 2 * d * f, "qkv_gemm": 6 * d * d, "o_gemm": 2 * d * d,
               "proj_gemm": 4 * d * d}
    breakdown = {}
    for name, ms in kern.items():
        tot = sum(ms) / kern_steps[name]
        entry = {"ms_per_step": tot, "launches_per_step": len(ms) / kern_steps[name]}
        if name in per_row:
            fl = per_row[name] * state_rows
            entry["tflops"] = fl / (tot / 1e3) / 1e12 if tot > 0 else None
            entry["frac_of_peak"] = entry["tflops"] / peak if entry["tflops"] else None
        if name == "head_ce_gemm":
            entry["tflops"] = achieved
            entry["frac_of_peak"] = achieved / peak
        if name == "prologue":  # gather E[x_{t+k}], read h^{k-1}, write c = [h; e] normalised: 8 d bytes per row
            hbm = float(load_peaks()[0].get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
            entry["gbs"] = 8.0 * cfg.d * state_rows / (tot / 1e3) / 1e9 if tot > 0 else None
            entry["frac_of_hbm"] = entry["gbs"] / hbm if entry["gbs"] else None
        breakdown[name] = entry

    # spec_verify: rows/s and algorithmic HBM bytes (decision scalars + the one sampled row pair or row)
    vo = vouts[W:W + K].cpu().numpy()
    acc, st = vo[:, 0], vo[:, 3]
    # the calls timed are those of the breakdown pass: their bytes
    vb = vouts[W + K:].cpu().numpy()
    b_acc, b_tok = vb[:, 0], vb[:, 1]
    b_rej = (b_acc < vcfg.gamma) & (b_tok >= 0)
    b_bonus = (b_acc == vcfg.gamma) & (b_tok >= 0)
    examined = np.minimum(b_acc + 1, vcfg.gamma)
    vbytes = (8.0 * examined + 8.0 * vcfg.V * b_rej + 4.0 * vcfg.V * b_bonus).sum(axis=1)  # per call
    v_ms = kern["spec_verify"]
    v_ms_mean = sum(v_ms) / len(v_ms)
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    v_gbs = float(vbytes.mean()) / (v_ms_mean / 1e3) / 1e9
    # floor for one pass over this many bytes: a read-only reduction over a buffer of the same size,
    # timed alike (L2 flushed first)
    nb = int(vbytes.mean()) // 16 * 16
    src_buf = torch.ones(nb // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    read_ms = []
    for _ in range(12):
        flush()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        torch.sum(src_buf, dim=0, out=sink)
        c1.record()
        torch.cuda.synchronize()
        read_ms.append(c0.elapsed_time(c1))
    read_us = 1e3 * sorted(read_ms[2:])[len(read_ms[2:]) // 2]
    del src_buf
    # what the same event pair reads around a kernel that does nothing (a one-element fill after
    # the same flush): launch latency and event overhead that every timed launch carries
    floor_ms = []
    for _ in range(40):
        flush()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        sink.fill_(0.0)
        c1.record()
        torch.cuda.synchronize()
        floor_ms.append(c0.elapsed_time(c1))
    floor_us = 1e3 * sorted(floor_ms[5:])[len(floor_ms[5:]) // 2]
    net_us = 1e3 * v_ms_mean - floor_us
    # the same calls replayed from a CUDA graph (48 calls over four input sets of 298 MB each, so
    # every call reads rows no recent call touched): per-call time without the launch and event
    # overhead of an isolated call
    gsets = [vin] + [synth.make_verify_inputs(vcfg, seed + 100 + s_, device=dev) for s_ in range(3)]
    gouts = [{k: torch.empty(vcfg.R, dtype=torch.int32, device=dev)
              for k in ("accepted", "next_token", "n_emit", "status")} for _ in gsets]
    n_graph = 48

    def graph_calls():
        for i in range(n_graph):
            v = gsets[i % len(gsets)]
            lib.spec_verify(v["p"], v["q"], v["draft"], seed=7 + rank, offset=5000 + i, out=gouts[i % len(gsets)])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up off the capture
        graph_calls()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        graph_calls()
    graph_ms = []
    for _ in range(5):
        flush()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        graph.replay()
        c1.record()
        torch.cuda.synchronize()
        graph_ms.append(c0.elapsed_time(c1) / n_graph)
    lib.check_errors()
    graph_us = 1e3 * sorted(graph_ms)[len(graph_ms) // 2]
    del graph, gsets, gouts
    verify = {"rows_per_s": world * vcfg.R * (vcfg.gamma + 1) / (v_ms_mean / 1e3),
              "same_size_read_us": read_us,
              "requests_per_s": world * vcfg.R / (v_ms_mean / 1e3), "us_per_call": 1e3 * v_ms_mean,
              "algorithmic_bytes_per_call": float(vbytes.mean()), "achieved_gbs": v_gbs, "peak_gbs": hbm_peak,
              "frac": v_gbs / hbm_peak, "mean_accepted": float(acc.mean()), "status_nonzero": int((st != 0).sum()),
              "event_floor_us": floor_us,
              "us_per_call_graph": graph_us,
              "frac_graph": float(vbytes.mean()) / (graph_us / 1e6) / 1e9 / hbm_peak,
              "frac_net_of_event_floor": (float(vbytes.mean()) / (net_us / 1e6) / 1e9 / hbm_peak) if net_us > 0 else None}

    # whole-step roofline (the metric's "% of roofline")
    step_rl = step_roofline(cfg, batch["seg"], counts, float(vbytes.mean()), step_ms_max, peaks)

    # decode-shaped draft step (its own workload, measured beside the step)
    draft = measure_draft(args, dev, rank, peaks)
    # DeepSeek-V3-width single depth (its own workload, measured beside the step)
    dsv3 = measure_dsv3(args, dev, rank, peaks)
    # training step (forward + backward) on the mid workload
    train = measure_train(args, dev, rank, peaks, chain, x, weights, cfg)

    # end to end through the public API: pinned host inputs -> device, result -> host, every step
    e2e = measure_e2e(cfg, vcfg, chain, batch, x, vin, args.e2e_steps, dev, rank, world, tokens_per_step)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, 1, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
                "ms_per_step": step_ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded; random-init weights of the workload's shapes)",
                "config": workload_config(), "roofline": roofline, "step_roofline": step_rl,
                "spec_verify": verify,
                "spec_verify_rows_per_s": verify["rows_per_s"], "kernels": breakdown,
                "kernels_pass": {"steps": KB, "ms_per_step_all_timers": b_ms / KB,
                                 "note": "per-kernel times other than head_ce_gemm come from this separate pass "
                                         "with an event pair around every launch"},
                "draft_step": draft, "dsv3_width": dsv3, "train_step": train,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
                "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
                "clock_samples": clk["samples"], "wall_s_timed_region": t_wall,
                "loss": float(out["losses"][0].item())}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_draft(args, dev, rank, peaks):
    """mtp_draft_step on the self-speculative decode workload (32 requests,
    module cache 8192 x d=7168, 56x128 heads, ffn 18432, V=129280) followed by
    gamma=1 verification of its draws; L2 flushed before every timed call.
    Algorithmic bytes: block weights + head + the 32 caches (K and V) + q."""
    import torch

    from deepseek_sequential_mtp_gb300 import lib, synth

    if args.draft_steps <= 0:
        return None
    cfg = synth.DRAFT_C5
    if args.draft_requests != cfg.R:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_R{args.draft_requests}", R=args.draft_requests)
    inp = synth.make_draft_inputs(cfg, 11 + rank, device=dev)
    step = lib.DraftStep(cfg, inp["weights"], device=dev)
    vcfg = synth.VerifyConfig(name="verify_R32_g1", R=cfg.R, gamma=1, V=cfg.V)
    vin = synth.make_verify_inputs(vcfg, 13 + rank, device=dev)
    out = {"q": torch.empty((cfg.R, cfg.V), dtype=torch.float32, device=dev),
           "y": torch.empty(cfg.R, dtype=torch.int32, device=dev)}
    vout = {k: torch.empty(cfg.R, dtype=torch.int32, device=dev)
            for k in ("accepted", "next_token", "n_emit", "status")}
    flush = L2Flush(dev)

    def call(i):
        step(inp["parent_hidden"], inp["frontier"], inp["pos"], inp["kv_k"], inp["kv_v"], inp["ctx_len"],
             seed=3, offset=i, out=out)

    for i in range(3):
        call(i)
        lib.spec_verify(vin["p"], out["q"].view(cfg.R, 1, cfg.V), out["y"].view(cfg.R, 1), seed=4, offset=i,
                        out=vout)
    torch.cuda.synchronize()
    lib.check_errors()
    n = args.draft_steps
    e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
          torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush()
        e[i][0].record()
        call(100 + i)
        e[i][1].record()
        lib.spec_verify(vin["p"], out["q"].view(cfg.R, 1, cfg.V), out["y"].view(cfg.R, 1), seed=4, offset=100 + i,
                        out=vout)
        e[i][2].record()
    torch.cuda.synchronize()
    lib.check_errors()
    d_ms = sorted(a.elapsed_time(b) for a, b, _ in e)[n // 2]
    v_ms = sorted(b.elapsed_time(c) for _, b, c in e)[n // 2]
    d, f, V, R = cfg.d, cfg.ffn, cfg.V, cfg.R
    weight_bytes = 2.0 * (2 * d * d + 4 * d * d + 3 * d * f)
    head_bytes = 2.0 * V * d
    cache_bytes = 2.0 * 2 * R * cfg.ctx * d
    q_bytes = 4.0 * R * V
    total = weight_bytes + head_bytes + cache_bytes + q_bytes
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = total / (d_ms / 1e3) / 1e9
    res = {"workload": f"draft step R={cfg.R}, cache 8192 x d=7168 (56x128), ffn 18432, V=129280 + gamma=1 verify",
           "ms_median": d_ms, "verify_ms_median": v_ms, "algorithmic_bytes": total,
           "achieved_gbs": gbs, "peak_gbs": hbm_peak, "frac": gbs / hbm_peak,
           "bound": "hbm", "steps": n, "l2": "flushed before every timed call (256 MiB written then read)"}
    del out, vout, step, vin

    # the same step with the module's linear maps in FP8 block-scaled form
    # (e4m3 codes + one fp32 scale per 128 x 128 block; head and cache bf16)
    if args.draft_fp8:
        f8 = synth.make_fp8_block(inp["weights"])
        step8 = lib.DraftStep(cfg, inp["weights"], device=dev, fp8=f8)
        out8 = {"q": torch.empty((cfg.R, cfg.V), dtype=torch.float32, device=dev),
                "y": torch.empty(cfg.R, dtype=torch.int32, device=dev)}

        def call8(i):
            step8(inp["parent_hidden"], inp["frontier"], inp["pos"], inp["kv_k"], inp["kv_v"], inp["ctx_len"],
                  seed=3, offset=i, out=out8)

        for i in range(3):
            call8(i)
        torch.cuda.synchronize()
        lib.check_errors()
        e8 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            flush()
            e8[i][0].record()
            call8(300 + i)
            e8[i][1].record()
        torch.cuda.synchronize()
        lib.check_errors()
        f_ms = sorted(a.elapsed_time(b) for a, b in e8)[n // 2]
        n_w = 2 * d * d + 4 * d * d + 3 * d * f
        blocks = sum(((r + 127) // 128) * ((k + 127) // 128)
                     for r, k in ((d, 2 * d), (d, d), (d, d), (d, d), (d, d), (f, d), (f, d), (d, f)))
        f_bytes = 1.0 * n_w + 4.0 * blocks + head_bytes + cache_bytes + q_bytes
        res["fp8"] = {"ms_median": f_ms, "algorithmic_bytes": f_bytes,
                      "achieved_gbs": f_bytes / (f_ms / 1e3) / 1e9,
                      "frac": f_bytes / (f_ms / 1e3) / 1e9 / hbm_peak,
                      "speedup_vs_bf16_weights": d_ms / f_ms, "steps": n,
                      "note": "module linear maps as e4m3 + fp32 128x128 block scales (1 B per weight); "
                              "head, norms and cache bf16"}
        del step8, out8, f8

    # recurrent round of gamma draft steps, then gamma-position verification of its draws
    g = args.draft_gamma
    if g > 1:
        rnd = lib.DraftRound(cfg, inp["weights"], g, device=dev)
        rin = synth.make_verify_inputs(synth.VerifyConfig(name=f"verify_R{cfg.R}_g{g}", R=cfg.R, gamma=g, V=cfg.V),
                                       15 + rank, device=dev)
        rout = {"q": torch.empty((cfg.R, g, cfg.V), dtype=torch.float32, device=dev),
                "y": torch.empty((cfg.R, g), dtype=torch.int32, device=dev)}
        vout = {k: torch.empty(cfg.R, dtype=torch.int32, device=dev)
                for k in ("accepted", "next_token", "n_emit", "status")}

        def round_call(i):
            rnd(inp["parent_hidden"], inp["frontier"], inp["pos"], inp["kv_k"], inp["kv_v"], inp["ctx_len"],
                seed=5, offset=i, out=rout)

        round_call(0)
        torch.cuda.synchronize()
        nr = max(3, n // g)
        er = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(nr)]
        for i in range(nr):
            flush()
            er[i][0].record()
            round_call(200 + i)
            er[i][1].record()
            lib.spec_verify(rin["p"], rout["q"], rout["y"], seed=6, offset=200 + i, out=vout)
            er[i][2].record()
        torch.cuda.synchronize()
        lib.check_errors()
        r_ms = sorted(a.elapsed_time(b) for a, b, _ in er)[nr // 2]
        rv_ms = sorted(b.elapsed_time(c) for _, b, c in er)[nr // 2]
        r_bytes = g * (weight_bytes + head_bytes + cache_bytes + q_bytes)
        res["round"] = {"gamma": g, "ms_median": r_ms, "verify_ms_median": rv_ms,
                        "drafted_tokens_per_s": cfg.R * g / (r_ms / 1e3), "algorithmic_bytes": r_bytes,
                        "achieved_gbs": r_bytes / (r_ms / 1e3) / 1e9,
                        "frac": r_bytes / (r_ms / 1e3) / 1e9 / hbm_peak, "calls": nr,
                        "note": "gamma recurrent steps of one module; the cache is streamed once per step"}
    return res


def measure_dsv3(args, dev, rank, peaks):
    """mtp_chain_loss on the DeepSeek-V3-width workload (B=1, T=4096, d=7168,
    56x128 heads, ffn 18432, V=129280, D=1, main + depth head): tokens/s and
    each GEMM class's TFLOP/s against the measured sustained bf16 peak.
    Algorithmic FLOPs count rows with state (T-1 at depth 1) and, for the
    heads, the supervised rows.  L2 flushed before every timed call."""
    import torch

    from deepseek_sequential_mtp_gb300 import lib, synth

    if args.c3_steps <= 0:
        return None
    cfg = synth.DSV3_BF16
    seed = 21 + rank
    batch = synth.make_batch(cfg, seed)
    x = {k: torch.from_numpy(v).to(dev) for k, v in batch.items()}
    h0 = synth.make_h0(cfg, seed, device=dev)
    chain = lib.Chain(cfg, synth.make_weights(cfg, seed + 1, device=dev), device=dev)
    out = {"sums_counts": torch.empty(2 * (cfg.D + 1), dtype=torch.float64, device=dev),
           "losses": torch.empty(cfg.D + 2, dtype=torch.float32, device=dev)}
    flush = L2Flush(dev)

    def call():
        chain.loss(x["tokens"], x["seg"], x["pos"], h0, den="fixed", with_main=True, out=out)

    for _ in range(2):
        call()
    torch.cuda.synchronize()
    lib.check_errors()
    n = args.c3_steps
    classes = ("head_ce_gemm", "gate_up_gemm", "down_gemm", "qkv_gemm", "o_gemm", "proj_gemm", "attention",
               "prologue")
    timers = {c: lib.KernelTimer(c, n * (cfg.D + 1)) for c in classes}
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for t in timers.values():
        t.arm()
    for i in range(n):
        flush()
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize()
    lib.KernelTimer.disarm_all()
    lib.check_errors()
    ms = sorted(a.elapsed_time(b) for a, b in ev)[n // 2]
    counts = out["sums_counts"][1::2].cpu().numpy()
    rows = float(sum(cfg.B * (cfg.T - k) for k in range(1, cfg.D + 1)))
    d, f, V = cfg.d, cfg.ffn, cfg.V
    peak = tensor_peak(peaks)
    flops = {"head_ce_gemm": 2.0 * d * V * float(counts.sum()), "gate_up_gemm": 4.0 * d * f * rows,
             "down_gemm": 2.0 * d * f * rows, "qkv_gemm": 6.0 * d * d * rows, "o_gemm": 2.0 * d * d * rows,
             "proj_gemm": 4.0 * d * d * rows}
    kernels = {}
    for c, t in timers.items():
        tot = sum(t.durations_ms()) / n
        e = {"ms_per_call": tot}
        if c in flops and tot > 0:
            e["tflops"] = flops[c] / (tot / 1e3) / 1e12
            e["frac_of_peak"] = e["tflops"] / peak
        kernels[c] = e
    head_launch_ms = kernels["head_ce_gemm"]["ms_per_call"] / (cfg.D + 1)
    head_launch_flops = flops["head_ce_gemm"] / (cfg.D + 1)
    head_tf = head_launch_flops / (head_launch_ms / 1e3) / 1e12 if head_launch_ms > 0 else None
    roofline = {"bound": "tensor", "kernel": "gemm_tc_kernel<256, EPI_CE> (shared head + online CE)",
                "achieved": head_tf, "peak": peak, "unit": "TFLOP/s",
                "frac": head_tf / peak if head_tf else None, "traffic": None,
                "algorithmic_flops_per_launch": head_launch_flops, "avg_launch_ms": head_launch_ms,
                "note": "dominant kernel of this workload (main + depth-1 heads); traffic not captured at this size"}
    return {"workload": "mtp_chain dsv3_width_D1 (B=1, T=4096, d=7168, 56x128 heads, ffn 18432, V=129280, "
                        "one packed boundary at 2048, main + depth-1 heads)",
            "tokens_per_s": rows / (ms / 1e3), "ms_per_call": ms, "steps": n, "kernels": kernels,
            "roofline": roofline, "peak_tflops": peak,
            "l2": "flushed before every timed call (256 MiB written then read)"}


def measure_train(args, dev, rank, peaks, chain, x, weights, cfg):
    """mtp_chain_loss_grad on the step's workload: the forward and the
    gradients of h^0 and of every weight (fp32, added into zeroed buffers).
    Algorithmic FLOPs = 3 x the forward's (rows with state for the block and
    projection GEMMs, supervised rows for the heads); the head logits are
    recomputed twice and the gate/up pre-activations once, which is extra work
    not counted.  L2 flushed before every timed step."""
    import torch

    from deepseek_sequential_mtp_gb300 import lib

    if args.train_steps <= 0:
        return None
    z = lambda t: torch.zeros(tuple(t.shape), dtype=torch.float32, device=dev)  # noqa: E731
    grads = {k: z(weights[k]) for k in ("embed", "head", "out_norm")}
    grads["h0"] = torch.zeros((cfg.B, cfg.T, cfg.d), dtype=torch.float32, device=dev)
    for k in ("hnorm", "enorm", "eh_proj", "attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up",
              "w_down"):
        grads[k] = [z(t) for t in weights[k]]
    out = {"sums_counts": torch.empty(2 * (cfg.D + 1), dtype=torch.float64, device=dev),
           "losses": torch.empty(cfg.D + 2, dtype=torch.float32, device=dev)}
    flush = L2Flush(dev)

    def call():
        chain.loss_grad(x["tokens"], x["seg"], x["pos"], x["h0"], grads, den="fixed", with_main=True, out=out)

    for _ in range(2):
        call()
    torch.cuda.synchronize()
    lib.check_errors()
    n = args.train_steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush()
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize()
    lib.check_errors()
    ms = sorted(a.elapsed_time(b) for a, b in ev)[n // 2]
    counts = out["sums_counts"][1::2].cpu().numpy()
    rows = float(sum(cfg.B * (cfg.T - k) for k in range(1, cfg.D + 1)))
    d, f, V = cfg.d, cfg.ffn, cfg.V
    fwd = (4 * d * d + 6 * d * d + 2 * d * d + 4 * d * f + 2 * d * f) * rows + 2.0 * d * V * float(counts.sum())
    peak = tensor_peak(peaks)
    tflops = 3.0 * fwd / (ms / 1e3) / 1e12
    return {"workload": "mtp_chain_loss_grad on the step's mid workload (all gradients)", "ms_median": ms,
            "tokens_per_s": rows / (ms / 1e3), "algorithmic_tflop": 3.0 * fwd / 1e12, "achieved_tflops": tflops,
            "frac_of_peak": tflops / peak, "steps": n,
            "l2": "flushed before every timed step (256 MiB written then read)"}


def measure_e2e(cfg, vcfg, chain, batch, x, vin, steps, dev, rank, world, tokens_per_step):
    """End to end through the public API: every step copies its inputs from
    pinned host memory (chain tokens/seg/pos/h0, verify p/q/drafts), runs the
    chain loss and spec_verify, and reads the losses and verify outputs back
    into pinned host memory.  Input copies are double-buffered on a second
    stream, so step i+1's copy overlaps step i's kernels, as an input pipeline
    would, and the results are read back on a third stream after an event, so
    the next step's kernels do not queue behind those small copies; the wall
    clock covers all copies, kernels and read-backs of the `steps` steps."""
    import torch

    from deepseek_sequential_mtp_gb300 import lib

    host = {k: torch.from_numpy(v).pin_memory() for k, v in batch.items()}
    host["h0"] = x["h0"].cpu().pin_memory()
    hv = {k: v.cpu().pin_memory() for k, v in vin.items()}
    bufs = [({k: torch.empty_like(v) for k, v in x.items()}, {k: torch.empty_like(v) for k, v in vin.items()})
            for _ in range(2)]
    n = max(steps, 1)
    res_l = [torch.empty(cfg.D + 2, dtype=torch.float32).pin_memory() for _ in range(n)]
    res_v = [torch.empty((4, vcfg.R), dtype=torch.int32).pin_memory() for _ in range(n)]
    h2d = sum(t.numel() * t.element_size() for t in list(host.values()) + list(hv.values()))
    d2h = res_l[0].numel() * 4 + res_v[0].numel() * 4
    comp = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    # step results are read back on a stream of their own, so the next step's kernels do not
    # queue behind the small device-to-host copies
    d2h_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    outs = [None, None]  # device outputs of the step that last used each slot

    def issue_copy(i):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(free[b])  # the step that last used this buffer has finished with it
            for k in bufs[b][0]:
                bufs[b][0][k].copy_(host[k], non_blocking=True)
            for k in bufs[b][1]:
                bufs[b][1][k].copy_(hv[k], non_blocking=True)
            ready[b].record(copy_stream)

    def run(n_steps, base):
        issue_copy(0)
        for i in range(n_steps):
            if i + 1 < n_steps:
                issue_copy(i + 1)
            b = i % 2
            comp.wait_event(ready[b])
            dx, dv = bufs[b]
            if outs[b] is not None:  # the read-back of this slot's previous outputs has finished
                comp.wait_event(done[b])
            o = chain.loss(dx["tokens"], dx["seg"], dx["pos"], dx["h0"], den="fixed", with_main=True)
            v = lib.spec_verify(dv["p"], dv["q"], dv["draft"], seed=7 + rank, offset=base + i)
            outs[b] = (o, v)
            free[b].record(comp)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(free[b])
                res_l[i].copy_(o["losses"], non_blocking=True)
                o["losses"].record_stream(d2h_stream)
                for j, kk in enumerate(("accepted", "next_token", "n_emit", "status")):
                    res_v[i][j].copy_(v[kk], non_blocking=True)
                    v[kk].record_stream(d2h_stream)
                done[b].record(d2h_stream)

    run(min(2, n), 10 ** 6)  # warm-up
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(n, 2 * 10 ** 6)
    torch.cuda.synchronize()
    per = (time.perf_counter() - t0) / n
    return {"value": world * tokens_per_step / per, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": 1e3 * per, "steps": n,
            "note": "every step copies its chain inputs (tokens, seg, pos, h0) and verify inputs (p, q, drafts) "
                    "from pinned host memory and reads its losses and verify outputs back; input copies are "
                    "double-buffered on a second stream so step i+1's copy overlaps step i's kernels, and results "
                    "are read back on a third stream so the next step's kernels do not wait for those copies"}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.impl == "cpu-one-core":
        run_one_core(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
