#!/usr/bin/env python
"""Benchmark: scored tokens/s of the fused linear logprob on the Qwen3-8B-shaped head.

One step = one pass of the whole scoring path over one batch of synthetic input:
RMSNorm -> LM-head GEMM with fused per-vocab-tile softmax statistics -> fixed-order
merge (logprob, lse, top-1) for T = 32768 rows (8 samples x 4096 tokens, d = 4096,
V = 151936, temperature 0.7), followed by the three-way compare of that batch's
generation / replay / trainer scores (8 sequences, TIS cap 2.0).  The step scores
the trainer set (C); A and B are recorded before the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints ONE JSON line on rank 0.  N > 1 runs under torchrun: every rank scores its
own batch (weak scaling, no data-path collective); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "scored tokens/s, fused logprob at d=4096,V=151936; % of bf16 tensor peak"
WORKLOAD = ("Qwen3-8B-shaped head: T=32768 rows (8 samples x 4096: 1024 shared prompt + 3072 "
            "response), d=4096, V=151936, temperature 0.7, three-way compare with TIS cap 2.0")
L2_NOTE = "inputs larger than L2 (W 1.245 GB + hidden 268 MB per step vs 129 MB L2)"

# DRAM bytes per lmhead_lse launch of this workload (T=32768, d=4096, V=151936),
# measured by a one-pass ncu capture of the full-size launch: 9.236 GB read +
# 0.315 GB written.  Valid only for the kernel sources hashed here (code lines
# only: comments and blank lines do not enter the hash) and for T = 32768.
TRAFFIC_CAPTURE = dict(sources={"lmhead_lse.cu": "a8d9cc34432250f6",
                                "tim_common.cuh": "68164e18e0c655eb"},
                       T=32768, bytes=9.236027904e9 + 314.873088e6)


def code_hash(path: str) -> str:
    """sha256 (16 hex digits) of a C++ source with // comments and blank lines removed."""
    import hashlib
    import re
    with open(path) as f:
        text = f.read()
    lines = []
    for line in text.splitlines():
        line = re.sub(r"//.*$", "", line).rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def traffic_per_launch(T):
    csrc = os.path.join(ROOT, "rollout_logprob_consistency_gb300", "csrc")
    for name, h in TRAFFIC_CAPTURE["sources"].items():
        if code_hash(os.path.join(csrc, name)) != h:
            return None   # the kernel changed since the counters were taken
    return TRAFFIC_CAPTURE["bytes"] if T == TRAFFIC_CAPTURE["T"] else None


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-extras", action="store_true")
    p.add_argument("--profile-shape", default=None,
                   help="T,d,V: only run --profile-iters tim_logprob calls of this shape "
                        "(small case for ncu captures), print nothing")
    p.add_argument("--profile-iters", type=int, default=3)
    p.add_argument("--profile-variant", default="bf16",
                   choices=["bf16", "fp8", "fp32", "backward", "processed", "diag"],
                   help="with --profile-shape: which head variant to run")
    p.add_argument("--score-workload", default=None,
                   choices=["tiny", "qwen3_1p7b", "qwen3_8b", "long_5120"],
                   help="instead of the benchmark step: time tim_logprob on the trainer rows "
                        "of this parity workload and the oracle on a bounded row sample, print "
                        "one JSON line (not the benchmark contract line)")
    p.add_argument("--cpu-rows", type=int, default=1024,
                   help="rows of the workload the oracle scores for the CPU baseline")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm_gbs=pk["hbm_gbs"], bf16=pk["bf16_tflops"],
                    bf16_sustained=pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------------------ clocks

class NvmlSampler:
    """SM clock, power and clock-event reasons of this process's GPU, read through NVML
    (queries only; no setting is changed) every ``period_s`` on a background thread
    while the timed region runs."""

    # nvmlClocksEventReason bits
    REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
               (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))

    def __init__(self, gpu_uuid, period_s=0.01, lib=None):
        import ctypes
        import threading
        self.ok = False
        self.rows = []
        if lib is None:
            try:
                lib = ctypes.CDLL("libnvidia-ml.so.1")
            except OSError:
                return
        self.lib = lib
        if lib.nvmlInit_v2() != 0:
            return
        self.dev = ctypes.c_void_p()
        found = False
        if gpu_uuid:
            u = gpu_uuid if gpu_uuid.upper().startswith("GPU-") else "GPU-" + gpu_uuid
            found = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.dev)) == 0
        if not found:
            n = ctypes.c_uint()
            if lib.nvmlDeviceGetCount_v2(ctypes.byref(n)) != 0 or n.value != 1 or \
                    lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.dev)) != 0:
                lib.nvmlShutdown()
                return
        self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        self.smax = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(
            self.dev, 1, ctypes.byref(mx)) == 0 else None
        self.ok = True
        self.period = period_s
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def _sample(self):
        import ctypes
        clk, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk)) != 0:   # NVML_CLOCK_SM
            return None
        power = mw.value / 1e3 if self.lib.nvmlDeviceGetPowerUsage(self.dev, ctypes.byref(mw)) == 0 else 0.0
        reasons = rs.value if self.reason_fn(self.dev, ctypes.byref(rs)) == 0 else 0
        return dict(t=time.perf_counter(), sm=float(clk.value), power=power, reasons=reasons)

    def _run(self):
        while not self._stop.is_set():
            r = self._sample()
            if r is not None:
                self.rows.append(r)
            self._stop.wait(self.period)

    def stop(self):
        if not self.ok:
            return None
        self._stop.set()
        self._thread.join(timeout=5)
        self.lib.nvmlShutdown()
        return self.summarize(self.rows, self.smax, self.period)

    @classmethod
    def summarize(cls, rows, smax, period):
        """Median / min / max SM clock, 100 MHz histogram, clock-event reasons seen and
        power of the samples (all taken inside the timed region)."""
        if not rows:
            return None
        reasons = sorted({name for r in rows for bit, name in cls.REASONS if r["reasons"] & bit})
        bins = {}
        for r in rows:
            key = f"{int(r['sm'] // 100) * 100}-{int(r['sm'] // 100) * 100 + 99}"
            bins[key] = bins.get(key, 0) + 1
        span = rows[-1]["t"] - rows[0]["t"]
        return dict(source="nvml", period_ms=1e3 * period,
                    sm_mhz=statistics.median(r["sm"] for r in rows),
                    sm_max_mhz=smax or max(r["sm"] for r in rows), reasons=reasons,
                    samples=len(rows), samples_under_load=len(rows),
                    sampled_span_s=round(span, 3),
                    sm_mhz_bins=dict(sorted(bins.items())),
                    sm_mhz_min=min(r["sm"] for r in rows), sm_mhz_max=max(r["sm"] for r in rows),
                    power_w_max=max(r["power"] for r in rows),
                    power_w_median=statistics.median(r["power"] for r in rows))


def start_clock_record(torch, rank):
    """In-process NVML sampling (10 ms) where NVML loads, else nvidia-smi (200 ms)."""
    if rank != 0:
        return None
    s = NvmlSampler(gpu_uuid(torch))
    return s if s.ok else ClockSampler(gpu_uuid(torch))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid):
        self.proc = None
        self.out = os.path.join("/tmp", f"tim_clocks_{os.getpid()}.csv")
        index = self._index_of(gpu_uuid)
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if index is not None:
                cmd += ["-i", str(index)]
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    @staticmethod
    def _index_of(gpu_uuid):
        """nvidia-smi index of the GPU this process uses (matched by UUID)."""
        try:
            r = subprocess.run(["nvidia-smi", "--query-gpu=index,uuid", "--format=csv,noheader"],
                               capture_output=True, text=True, timeout=20)
        except (OSError, subprocess.TimeoutExpired):
            return None
        rows = [ln.split(",") for ln in r.stdout.strip().splitlines() if "," in ln]
        if gpu_uuid:
            key = gpu_uuid.lower().replace("gpu-", "")
            for idx, uuid in rows:
                if uuid.strip().lower().replace("gpu-", "") == key:
                    return int(idx)
        return int(rows[0][0]) if len(rows) == 1 else None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.out) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                     power=float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                                     hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
                except ValueError:
                    continue
        os.remove(self.out)
        if not rows:
            return None
        load = [r for r in rows if r["power"] > 0.5 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in load),
                    sm_max_mhz=max(r["smax"] for r in load), reasons=sorted(reasons),
                    samples=len(rows), samples_under_load=len(load),
                    power_w_max=max(r["power"] for r in rows),
                    power_w_median=statistics.median(r["power"] for r in load))


def gpu_uuid(torch):
    try:
        return str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        return None


# ------------------------------------------------------------------------------ distributed

def dist_setup(n, timeout_s: float = 600.0):
    """Join the process group (one rank per GPU).  A rank that dies or never joins makes
    the others' next collective fail after ``timeout_s`` instead of waiting forever."""
    if n <= 1 and "WORLD_SIZE" not in os.environ:
        return 0, 1, 0, None
    import datetime
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    backend = "nccl" if os.environ.get("TIM_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
    dist.init_process_group(backend=backend, timeout=datetime.timedelta(seconds=timeout_s))
    return rank, world, local, dist


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device):
    if dist is None:
        return
    import torch
    if dist.get_backend() == "nccl":
        dist.barrier(device_ids=[torch.cuda.current_device()])
    else:
        dist.barrier()


# ------------------------------------------------------------------------------ CPU oracle

def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(b, rows):
    """fp64 oracle on ``rows`` of the workload (trainer set) + the compare of those rows."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    out = oracle.oracle_logprob(b.hidden_train[rows], b.head.gamma, b.head.W, b.token_ids[rows],
                                b.temperature, b.eps)
    lp = out["logprob"].astype(np.float32)
    oracle.oracle_compare(lp, lp, lp, np.array([0, len(rows)], dtype=np.int64),
                          np.ones(len(rows), np.uint8), b.tis_cap)
    return time.perf_counter() - t0


def reference_arm(args):
    """--impl reference: the fp64 CPU oracle on this workload, bounded per step."""
    import numpy as np
    import synth
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return 0
    b = synth.make_qwen3_8b()
    # one oracle row block per step: its fixed cost (widening W to fp64) is then
    # shared by 128 rows, about 2 s per step on 16 cores
    rows_per_step = 128
    g = np.random.default_rng(77)
    for _ in range(args.warmup):
        time_oracle(b, np.sort(g.choice(b.T, rows_per_step, replace=False)))
    total = 0.0
    for _ in range(args.steps):
        total += time_oracle(b, np.sort(g.choice(b.T, rows_per_step, replace=False)))
    value = rows_per_step * args.steps / total
    sample = (f"{rows_per_step} seeded rows of the workload per step, scored by the fp64 oracle "
              f"(RMSNorm, bf16 rounding, fp64 GEMM over V=151936, log-sum-exp) plus the compare")
    line = dict(impl="reference", metric=METRIC, value=value, unit="tokens/s", n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * total / args.steps,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic", config=dict(workload=WORKLOAD, T=b.T, d=b.d, V=b.V,
                                              temperature=b.temperature, l2=L2_NOTE),
                cpu_baseline=dict(value=value, unit="tokens/s", cores=cpu_cores(), kind="oracle",
                                  sample=sample),
                e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0),
                gpu_launches=0)
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ GPU arm

def profile_variant(args, tim, b, hid, gam, W, ids, out):
    """--profile-iters calls of the FP8 head, the FP32 head or the backward (weights
    prepared once beforehand, as a caller would)."""
    import torch
    T, d, V = b.T, b.head.d, b.head.V
    if args.profile_variant == "fp8":
        W8, sW = tim.quantize_fp8_rows(W)
        ws = tim.Workspace(int(tim.lib().tim_logprob_fp8_workspace_size(T, d, V)))
        for _ in range(args.profile_iters):
            tim.logprob_fp8(hid, gam, W8, sW, ids, 0.7, b.eps, out=out, workspace=ws, check=False)
    elif args.profile_variant == "fp32":
        Wb, Wsm = tim.split_tf32(W.float().contiguous())
        ws = tim.Workspace(int(tim.lib().tim_logprob_fp32_workspace_size(T, d, V)))
        for _ in range(args.profile_iters):
            tim.logprob_fp32(hid, gam, Wb, Wsm, ids, 0.7, b.eps, out=out, workspace=ws,
                             check=False)
    elif args.profile_variant == "processed":
        ws = tim.Workspace(int(tim.lib().tim_processed_logprob_workspace_size(T, d, V)))
        for _ in range(args.profile_iters):
            tim.processed_logprob(hid, gam, W, ids, 0.7, b.eps, 50, 0.95, out=out, workspace=ws,
                                  check=False)
    elif args.profile_variant == "diag":
        import numpy as np
        tim.logprob(hid, gam, W, ids, 0.7, b.eps, out=out)
        S = 8 if T >= 8 else 1
        offs = torch.from_numpy(np.linspace(0, T, S + 1).astype(np.int64)).cuda()
        mask = torch.ones(T, dtype=torch.uint8, device="cuda")
        ws = tim.Workspace(int(tim.lib().tim_compare_diag_workspace_size(T, S)))
        noisy = out[0] + 1e-3 * torch.randn(T, device="cuda")
        for _ in range(args.profile_iters):
            tim.compare_diag(out[0], out[0], noisy, offs, mask, 2.0, 0.5, 2.0,
                             top1=(out[2], out[2], out[2]), workspace=ws, check=False,
                             to_host=False)
    else:
        tim.logprob(hid, gam, W, ids, 0.7, b.eps, out=out)
        ws = tim.Workspace(int(tim.lib().tim_logprob_backward_workspace_size(T, d, V)))
        g = torch.ones(T, dtype=torch.float32, device="cuda")
        dy = torch.empty(T, d, dtype=torch.float32, device="cuda")
        dW = torch.empty(V, d, dtype=torch.float32, device="cuda")
        for _ in range(args.profile_iters):
            tim.logprob_backward(hid, gam, W, ids, out[1], g, 0.7, b.eps, out_dy=dy, out_dW=dW,
                                 workspace=ws, check=False)
    ws.check(f"profile {args.profile_variant}")
    torch.cuda.synchronize()
    return 0


def profile_case(args):
    """A few tim_logprob calls of one shape, for ncu captures of the kernels."""
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import synth
    import rollout_logprob_consistency_gb300 as tim
    T, d, V = (int(x) for x in args.profile_shape.split(","))
    b = synth.make_custom(T=T, d=d, V=V, temperature=0.7, tag="prof")

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    hid, gam, W = bf16(b.hidden_gen), bf16(b.head.gamma), bf16(b.head.W)
    ids = torch.from_numpy(b.token_ids).cuda()
    out = (torch.empty(T, device="cuda"), torch.empty(T, device="cuda"),
           torch.empty(T, dtype=torch.int32, device="cuda"))
    if args.profile_variant != "bf16":
        return profile_variant(args, tim, b, hid, gam, W, ids, out)
    ws = tim.Workspace(tim.logprob_workspace_size(T, d, V))
    for _ in range(args.profile_iters):
        tim.logprob(hid, gam, W, ids, 0.7, b.eps, out=out, workspace=ws, check=False)
    ws.check("profile case")
    # the three-way compare of the scored rows as 8 equal sequences (all tokens active)
    S = 8 if T >= 8 else 1
    offs = torch.from_numpy(np.linspace(0, T, S + 1).astype(np.int64)).cuda()
    mask = torch.ones(T, dtype=torch.uint8, device="cuda")
    cws = tim.Workspace(tim.compare_workspace_size(T, S))
    for _ in range(args.profile_iters):
        tim.compare(out[0], out[0], out[0], offs, mask, 2.0, workspace=cws, check=False,
                    to_host=False)
    cws.check("profile compare")
    torch.cuda.synchronize()
    return 0


def score_workload(args):
    """--score-workload: tokens/s of one scoring call over a whole parity workload (CUDA
    events, back-to-back calls after warm-up) and of the oracle on a bounded seeded sample."""
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import synth
    import rollout_logprob_consistency_gb300 as tim
    make = dict(tiny=synth.make_tiny, qwen3_1p7b=synth.make_qwen3_1p7b,
                qwen3_8b=synth.make_qwen3_8b, long_5120=synth.make_long_5120)[args.score_workload]
    b = make()
    T, d, V = b.T, b.head.d, b.head.V

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    hid, gam = bf16(b.hidden_train), bf16(b.head.gamma)
    W = bf16(b.W_train if b.W_train is not None else b.head.W)
    ids = torch.from_numpy(b.token_ids).cuda()
    ws = tim.Workspace(tim.logprob_workspace_size(T, d, V))
    out = (torch.empty(T, device="cuda"), torch.empty(T, device="cuda"),
           torch.empty(T, dtype=torch.int32, device="cuda"))
    for _ in range(max(args.warmup, 3)):
        tim.logprob(hid, gam, W, ids, b.temperature, b.eps, out=out, workspace=ws, check=False)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        tim.logprob(hid, gam, W, ids, b.temperature, b.eps, out=out, workspace=ws, check=False)
    e1.record()
    torch.cuda.synchronize()
    ws.check("score workload")
    ms = e0.elapsed_time(e1) / args.steps
    peaks = load_peaks()
    tflops = 2.0 * T * d * V / (ms / 1e3) / 1e12
    gbps = (2.0 * V * d + 2.0 * T * d) / (ms / 1e3) / 1e9
    frac = max(tflops / peaks["bf16_sustained"], gbps / peaks["hbm_gbs"])
    n_or = min(T, args.cpu_rows)
    rows = np.sort(np.random.default_rng(99).choice(T, n_or, replace=False))
    import oracle
    t0 = time.perf_counter()
    oracle.oracle_logprob(b.hidden_train[rows], b.head.gamma,
                          b.W_train if b.W_train is not None else b.head.W, b.token_ids[rows],
                          b.temperature, b.eps)
    dt = time.perf_counter() - t0
    print(json.dumps(dict(workload=b.name, T=T, d=d, V=V, ms_per_call=round(ms, 4),
                          tokens_per_s=round(T / (ms / 1e3), 1), TFLOPs=round(tflops, 1),
                          GBps=round(gbps, 1), roofline_frac=round(frac, 3),
                          peak_source=peaks["source"], oracle_rows=int(n_or),
                          oracle_s=round(dt, 2), oracle_tokens_per_s=round(n_or / dt, 1),
                          host_cores=cpu_cores())), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    if args.score_workload:
        return score_workload(args)
    if args.profile_shape:
        return profile_case(args)
    import numpy as np
    import torch

    rank, world, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    import synth
    import rollout_logprob_consistency_gb300 as tim

    peaks = load_peaks()
    b = synth.make_qwen3_8b(seed=rank)
    T, d, V = b.T, b.d, b.V
    tau, eps = b.temperature, b.eps
    stream = torch.cuda.current_stream()

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    W = bf16(b.head.W)
    gam = bf16(b.head.gamma)
    hid_gen = bf16(b.hidden_gen)
    hid_train = bf16(b.hidden_train)
    ids = torch.from_numpy(b.token_ids).to(dev)
    offs = torch.from_numpy(b.seq_offsets).to(dev)
    mask = torch.from_numpy(b.mask).to(dev)
    ws = tim.Workspace(tim.logprob_workspace_size(T, d, V), dev)
    cws = tim.Workspace(tim.compare_workspace_size(T, b.n_seq), dev)

    def new_out():
        return (torch.empty(T, dtype=torch.float32, device=dev),
                torch.empty(T, dtype=torch.float32, device=dev),
                torch.empty(T, dtype=torch.int32, device=dev))

    A = new_out()
    Bo = new_out()
    C = new_out()
    tim.logprob(hid_gen, gam, W, ids, tau, eps, out=A, workspace=ws)
    tim.logprob(hid_gen, gam, W, ids, tau, eps, out=Bo, workspace=ws)
    stats_buf = torch.empty(b.n_seq * tim.SEQ_STATS_DTYPE.itemsize, dtype=torch.uint8, device=dev)
    tis_w = torch.empty(T, dtype=torch.float32, device=dev)

    def step(evs=None):
        tim.logprob_stages(hid_train, gam, W, ids, tau, eps, C, ws, stream, events=evs)
        tim.compare(A[0], Bo[0], C[0], offs, mask, b.tis_cap, out_stats=stats_buf,
                    out_tis_w=tis_w, workspace=cws, check=False, to_host=False)

    for _ in range(max(args.warmup, 3)):
        step()
    ws.check("warmup")
    cws.check("warmup compare")

    ev_all = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = start_clock_record(torch, rank)
    barrier(dist, dev)
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        step(ev_all[k])
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(dist, dev)
    clk = clocks.stop() if clocks is not None else None
    ws.check("timed steps")
    cws.check("timed compare")
    total_ms = max_over_ranks(start.elapsed_time(stop), dist, dev)
    gemm_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev_all)
    norm_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev_all)
    fin_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev_all)
    ms_per_step = total_ms / args.steps
    value = world * T * args.steps / (total_ms / 1e3)

    flops = 2.0 * T * d * V
    achieved_tflops = flops / (gemm_ms / 1e3) / 1e12
    # the burst peak (a GEMM timed alone for a short while) for a timed region under
    # 2 s, the sustained one (seconds under the power cap) for longer regions
    short_region = total_ms < 2000.0
    peak = peaks["bf16"] if short_region else peaks["bf16_sustained"]
    peak_other = peaks["bf16_sustained"] if short_region else peaks["bf16"]

    # ---------------------------------------------------------------- end to end (host buffers)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_hid = pin(b.hidden_train.view(np.int16))
    h_ids = pin(b.token_ids)
    h_A = A[0].cpu().pin_memory()
    h_B = Bo[0].cpu().pin_memory()
    h_mask = pin(b.mask)
    h_offs = pin(b.seq_offsets)
    h_out = [torch.empty(T, dtype=torch.float32).pin_memory(),
             torch.empty(T, dtype=torch.float32).pin_memory(),
             torch.empty(T, dtype=torch.int32).pin_memory(),
             torch.empty(stats_buf.numel(), dtype=torch.uint8).pin_memory()]
    # two device input slots: the host->device copies of step k+1 run on a copy stream
    # while step k computes (inputs are still copied every step, inside the timed region)
    slots = []
    for _ in range(2):
        slots.append(dict(
            hid=torch.empty(T, d, dtype=torch.int16, device=dev),
            ids=torch.empty(T, dtype=torch.int32, device=dev),
            A=torch.empty(T, dtype=torch.float32, device=dev),
            B=torch.empty(T, dtype=torch.float32, device=dev),
            mask=torch.empty(T, dtype=torch.uint8, device=dev),
            offs=torch.empty(b.n_seq + 1, dtype=torch.int64, device=dev),
            ev_in=torch.cuda.Event(), ev_done=torch.cuda.Event()))
    copy_stream = torch.cuda.Stream(device=dev)
    h2d = sum(x.numel() * x.element_size() for x in (h_hid, h_ids, h_A, h_B, h_mask, h_offs))
    d2h = sum(x.numel() * x.element_size() for x in h_out)

    def e2e_step(k):
        sl = slots[k % 2]
        copy_stream.wait_event(sl["ev_done"])          # step k-2 finished with this slot
        with torch.cuda.stream(copy_stream):
            for key, src in (("hid", h_hid), ("ids", h_ids), ("A", h_A), ("B", h_B),
                             ("mask", h_mask), ("offs", h_offs)):
                sl[key].copy_(src, non_blocking=True)
            sl["ev_in"].record(copy_stream)
        stream.wait_event(sl["ev_in"])
        tim.logprob(sl["hid"].view(torch.bfloat16), gam, W, sl["ids"], tau, eps, out=C,
                    workspace=ws, check=False)
        tim.compare(sl["A"], sl["B"], C[0], sl["offs"], sl["mask"], b.tis_cap,
                    out_stats=stats_buf, out_tis_w=tis_w, workspace=cws, check=False,
                    to_host=False)
        for dst, src in zip(h_out, (C[0], C[1], C[2], stats_buf)):
            dst.copy_(src, non_blocking=True)
        sl["ev_done"].record(stream)

    for k in range(3):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_steps = max(3, args.steps)
    barrier(dist, dev)
    start.record(stream)
    copy_stream.wait_event(start)
    for k in range(e2e_steps):
        e2e_step(k)
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(dist, dev)
    ws.check("e2e")
    e2e_ms = max_over_ranks(start.elapsed_time(stop), dist, dev)
    e2e_value = world * T * e2e_steps / (e2e_ms / 1e3)

    # ---------------------------------------------------------------- compare alone
    c_a, c_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        tim.compare(A[0], Bo[0], C[0], offs, mask, b.tis_cap, out_stats=stats_buf, out_tis_w=tis_w,
                    workspace=cws, check=False, to_host=False)
    c_a.record(stream)
    for _ in range(50):
        tim.compare(A[0], Bo[0], C[0], offs, mask, b.tis_cap, out_stats=stats_buf, out_tis_w=tis_w,
                    workspace=cws, check=False, to_host=False)
    c_b.record(stream)
    torch.cuda.synchronize()
    cws.check("compare timing")
    cmp_us = 1e3 * c_a.elapsed_time(c_b) / 50
    cmp_bytes = T * (3 * 4 + 1 + 4) + (b.n_seq + 1) * 8 + b.n_seq * tim.SEQ_STATS_DTYPE.itemsize
    compare_info = dict(us=round(cmp_us, 2), bytes=cmp_bytes,
                        GBps=round(cmp_bytes / cmp_us / 1e3, 1), sequences=b.n_seq)

    # ---------------------------------------------------------------- next-row paths on this workload
    extras = None
    if rank == 0 and world == 1 and not args.no_extras:   # N = 1 runs report these
        extras = {}
        pout = (torch.empty(T, device=dev), torch.empty(T, device=dev),
                torch.empty(T, dtype=torch.int32, device=dev))
        pws = tim.Workspace(int(tim.lib().tim_processed_logprob_workspace_size(T, d, V)), dev)
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tim.processed_logprob(hid_train, gam, W, ids, tau, eps, 50, 0.95, out=pout,
                              workspace=pws, check=False)
        e_a.record(stream)
        for _ in range(3):
            tim.processed_logprob(hid_train, gam, W, ids, tau, eps, 50, 0.95, out=pout,
                                  workspace=pws, check=False)
        e_b.record(stream)
        torch.cuda.synchronize()
        pws.check("processed")
        pms = e_a.elapsed_time(e_b) / 3
        extras["processed_topk50_topp0.95"] = dict(ms=round(pms, 3),
                                                   tokens_per_s=round(T / (pms / 1e3), 1))
        del pws
        dws = tim.Workspace(int(tim.lib().tim_compare_diag_workspace_size(T, b.n_seq)), dev)
        dout = torch.empty(b.n_seq * tim.SEQ_DIAG_DTYPE.itemsize, dtype=torch.uint8, device=dev)
        tops = (A[2], Bo[2], C[2])
        tim.compare_diag(A[0], Bo[0], C[0], offs, mask, b.tis_cap, 0.5, 2.0, top1=tops, out=dout,
                         workspace=dws, check=False, to_host=False)
        e_a.record(stream)
        for _ in range(10):
            tim.compare_diag(A[0], Bo[0], C[0], offs, mask, b.tis_cap, 0.5, 2.0, top1=tops,
                             out=dout, workspace=dws, check=False, to_host=False)
        e_b.record(stream)
        torch.cuda.synchronize()
        dws.check("diag")
        extras["compare_diag_us"] = round(1e3 * e_a.elapsed_time(e_b) / 10, 2)
        # the whole batch as one sequence: 24576 active tokens, more than a quantile CTA
        # holds in shared memory, so the keys past 16384 are kept in the workspace
        offs1 = torch.tensor([0, T], dtype=torch.int64, device=dev)
        dws1 = tim.Workspace(int(tim.lib().tim_compare_diag_workspace_size(T, 1)), dev)
        dout1 = torch.empty(tim.SEQ_DIAG_DTYPE.itemsize, dtype=torch.uint8, device=dev)
        tim.compare_diag(A[0], Bo[0], C[0], offs1, mask, b.tis_cap, 0.5, 2.0, top1=tops, out=dout1,
                         workspace=dws1, check=False, to_host=False)
        e_a.record(stream)
        for _ in range(10):
            tim.compare_diag(A[0], Bo[0], C[0], offs1, mask, b.tis_cap, 0.5, 2.0, top1=tops,
                             out=dout1, workspace=dws1, check=False, to_host=False)
        e_b.record(stream)
        torch.cuda.synchronize()
        dws1.check("diag one sequence")
        extras["compare_diag_one_sequence_us"] = dict(
            us=round(1e3 * e_a.elapsed_time(e_b) / 10, 2), active_tokens=int(b.mask.sum()),
            note="quantiles over 16384 shared-memory keys plus the rest kept in the workspace")
        # FP8 (e4m3) head: W quantised once per weight version (untimed), then whole calls
        W8, sW8 = tim.quantize_fp8_rows(W)
        fws = tim.Workspace(int(tim.lib().tim_logprob_fp8_workspace_size(T, d, V)), dev)
        tim.logprob_fp8(hid_train, gam, W8, sW8, ids, tau, eps, out=pout, workspace=fws,
                        check=False)
        e_a.record(stream)
        for _ in range(5):
            tim.logprob_fp8(hid_train, gam, W8, sW8, ids, tau, eps, out=pout, workspace=fws,
                            check=False)
        e_b.record(stream)
        torch.cuda.synchronize()
        fws.check("fp8 head")
        fms = e_a.elapsed_time(e_b) / 5
        fp8_peak = 2.0 * peaks["bf16_sustained"] if peaks.get("bf16_sustained") else None
        extras["fp8_e4m3_head"] = dict(
            ms=round(fms, 3), tokens_per_s=round(T / (fms / 1e3), 1),
            call_TFLOPs=round(2.0 * T * d * V / (fms / 1e3) / 1e12, 1),
            peak_TFLOPs=fp8_peak, peak_note="2 x measured sustained bf16 (nominal fp8:bf16 ratio)")
        del fws, W8, sW8
        # FP32 head: W (fp32 here: the bf16 W widened) split once per weight version (untimed)
        Wb32, Ws32 = tim.split_tf32(W.view(torch.bfloat16).float().contiguous())
        f32ws = tim.Workspace(int(tim.lib().tim_logprob_fp32_workspace_size(T, d, V)), dev)
        tim.logprob_fp32(hid_train, gam, Wb32, Ws32, ids, tau, eps, out=pout, workspace=f32ws,
                         check=False)
        e_a.record(stream)
        for _ in range(2):
            tim.logprob_fp32(hid_train, gam, Wb32, Ws32, ids, tau, eps, out=pout, workspace=f32ws,
                             check=False)
        e_b.record(stream)
        torch.cuda.synchronize()
        f32ws.check("fp32 head")
        f32ms = e_a.elapsed_time(e_b) / 2
        tf32_peak = 0.5 * peaks["bf16_sustained"] if peaks.get("bf16_sustained") else None
        extras["fp32_tf32x3_head"] = dict(
            ms=round(f32ms, 3), tokens_per_s=round(T / (f32ms / 1e3), 1),
            fp32_equiv_TFLOPs=round(2.0 * T * d * V / (f32ms / 1e3) / 1e12, 1),
            tensor_TFLOPs=round(3 * 2.0 * T * d * V / (f32ms / 1e3) / 1e12, 1),
            tensor_peak_TFLOPs=tf32_peak,
            peak_note="tf32 = 0.5 x measured sustained bf16 (nominal ratio); three tf32 products "
                      "per multiply-add")
        del f32ws, Wb32, Ws32
        # backward of the linear logprob (recompute + G + dL/dy + dL/dW), upstream gradient 1
        gup = torch.ones(T, dtype=torch.float32, device=dev)
        lse_c = C[1]                      # the trainer-set lse of the timed steps
        bws = tim.Workspace(int(tim.lib().tim_logprob_backward_workspace_size(T, d, V)), dev)
        dy_b = torch.empty(T, d, dtype=torch.float32, device=dev)
        dW_b = torch.empty(V, d, dtype=torch.float32, device=dev)
        tim.logprob_backward(hid_train, gam, W, ids, lse_c, gup, tau, eps, out_dy=dy_b,
                             out_dW=dW_b, workspace=bws, check=False)
        e_a.record(stream)
        for _ in range(2):
            tim.logprob_backward(hid_train, gam, W, ids, lse_c, gup, tau, eps, out_dy=dy_b,
                                 out_dW=dW_b, workspace=bws, check=False)
        e_b.record(stream)
        torch.cuda.synchronize()
        bws.check("backward")
        bms = e_a.elapsed_time(e_b) / 2
        # the RMSNorm backward that carries dy on to the hidden states and gamma
        rws = tim.Workspace(int(tim.lib().tim_rmsnorm_backward_workspace_size(T, d)), dev)
        dh_b = torch.empty(T, d, dtype=torch.float32, device=dev)
        dg_b = torch.empty(d, dtype=torch.float32, device=dev)
        tim.rmsnorm_backward(hid_train, gam, dy_b, eps, out_dh=dh_b, out_dgamma=dg_b,
                             workspace=rws, check=False)
        e_a.record(stream)
        for _ in range(5):
            tim.rmsnorm_backward(hid_train, gam, dy_b, eps, out_dh=dh_b, out_dgamma=dg_b,
                                 workspace=rws, check=False)
        e_b.record(stream)
        torch.cuda.synchronize()
        rws.check("rmsnorm backward")
        rms_ms = e_a.elapsed_time(e_b) / 5
        rms_bytes = T * d * (2 + 4 + 4) + T * d * (2 + 4)   # rows pass + dgamma pass
        extras["backward_dy_dW"] = dict(
            ms=round(bms, 3), tokens_per_s=round(T / (bms / 1e3), 1),
            TFLOPs=round(3 * 2.0 * T * d * V / (bms / 1e3) / 1e12, 1),
            note="three GEMMs (logit recompute writing G once, G.W and G^T.y reading G, W and y in place); workspace "
                 f"{bws.nbytes / 1e9:.1f} GB",
            rmsnorm_backward_ms=round(rms_ms, 3),
            rmsnorm_backward_GBps=round(rms_bytes / (rms_ms / 1e3) / 1e9, 1))
        del bws, dy_b, dW_b, rws, dh_b, dg_b
        # the other two scoring workloads, whole tim_logprob calls: the Qwen3-1.7B-shaped
        # head (T = 8192, d = 2048, tau = 1.0) and the long-rollout head (T = 131072,
        # d = 5120, tau = 0.7).  Inputs are drawn on the device (seeded torch generator)
        # with the workloads' shapes and value distributions; token ids are uniform here
        # (the ids do not enter the time).
        for name, (Tw, dw, tw) in (("qwen3_1p7b", (8192, 2048, 1.0)),
                                   ("long_5120", (131072, 5120, 0.7))):
            gen = torch.Generator(device=dev)
            gen.manual_seed(1234)
            Ww = (torch.randn(V, dw, generator=gen, device=dev) * (2.0 / dw ** 0.5)).to(torch.bfloat16)
            hw = torch.randn(Tw, dw, generator=gen, device=dev).to(torch.bfloat16)
            gw = (1.0 + 0.05 ** 0.5 * torch.randn(dw, generator=gen, device=dev)).to(torch.bfloat16)
            iw = torch.randint(0, V, (Tw,), generator=gen, device=dev, dtype=torch.int32)
            wsw = tim.Workspace(tim.logprob_workspace_size(Tw, dw, V), dev)
            ow = (torch.empty(Tw, device=dev), torch.empty(Tw, device=dev),
                  torch.empty(Tw, dtype=torch.int32, device=dev))
            for _ in range(2):
                tim.logprob(hw, gw, Ww, iw, tw, eps, out=ow, workspace=wsw, check=False)
            reps = 5 if Tw > 16384 else 20
            e_a.record(stream)
            for _ in range(reps):
                tim.logprob(hw, gw, Ww, iw, tw, eps, out=ow, workspace=wsw, check=False)
            e_b.record(stream)
            torch.cuda.synchronize()
            wsw.check(name)
            wms = e_a.elapsed_time(e_b) / reps
            wtf = 2.0 * Tw * dw * V / (wms / 1e3) / 1e12
            extras[name] = dict(T=Tw, d=dw, V=V, temperature=tw, ms=round(wms, 3),
                                tokens_per_s=round(Tw / (wms / 1e3), 1), TFLOPs=round(wtf, 1),
                                frac_of_burst=round(wtf / peaks["bf16"], 3),
                                frac_of_sustained=round(wtf / peaks["bf16_sustained"], 3),
                                note="whole tim_logprob calls (RMSNorm, LM head, finalize); "
                                     "inputs drawn on the device, seeded")
            del Ww, hw, gw, iw, wsw, ow
        torch.cuda.empty_cache()
        G = 8
        e_a.record(stream)
        for _ in range(2):
            tim.logprob_vocab_parallel_emulated(hid_train, gam, W, ids, G, tau, eps)
        e_b.record(stream)
        torch.cuda.synchronize()
        vms = e_a.elapsed_time(e_b) / 2
        extras["vocab_parallel_G8_emulated_on_1_gpu"] = dict(
            ms=round(vms, 3), note="the 8 shards run one after another on one GPU; on 8 GPUs "
            "each rank would run one shard plus the merge")

    # ---------------------------------------------------------------- decode-shaped rows (HBM bound)
    decode = None
    if not args.no_decode and rank == 0 and world == 1:
        decode = {}
        for M in (1, 7, 64, 128, 200, 256, 320, 384, 448, 512, 513, 1024):
            wsm = tim.Workspace(tim.logprob_workspace_size(M, d, V), dev)
            outm = (torch.empty(M, device=dev), torch.empty(M, device=dev),
                    torch.empty(M, dtype=torch.int32, device=dev))
            hm, im = hid_gen[:M].contiguous(), ids[:M].contiguous()
            for _ in range(5):
                tim.logprob_stages(hm, gam, W, im, tau, eps, outm, wsm, stream)
            iters = 50
            # whole tim_logprob calls back to back (no events between the stages)
            t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t_a.record(stream)
            for it in range(iters):
                tim.logprob(hm, gam, W, im, tau, eps, out=outm, workspace=wsm, check=False)
            t_b.record(stream)
            # the same calls stage by stage with events, for the GEMM kernel alone
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(iters)]
            for it in range(iters):
                tim.logprob_stages(hm, gam, W, im, tau, eps, outm, wsm, stream, events=evs[it])
            torch.cuda.synchronize()
            wsm.check(f"decode M={M}")
            call_us = 1e3 * t_a.elapsed_time(t_b) / iters
            gemm_us = 1e3 * statistics.median(e[1].elapsed_time(e[2]) for e in evs)
            nbytes = 2.0 * V * d + 2.0 * M * d
            # roofline time: the larger of the W (+ hidden) read at the measured copy
            # bandwidth and 2 M d V FLOP at the measured burst bf16 peak
            roof_us = max(nbytes / peaks["hbm_gbs"] / 1e3, 2.0 * M * d * V / peaks["bf16"] / 1e6)
            decode[f"M{M}"] = dict(call_us=round(call_us, 2), gemm_us=round(gemm_us, 2),
                                   call_GBps=round(nbytes / call_us / 1e3, 1),
                                   gemm_GBps=round(nbytes / gemm_us / 1e3, 1),
                                   gemm_frac_of_hbm=round(nbytes / gemm_us / 1e3 / peaks["hbm_gbs"], 3),
                                   call_frac_of_hbm=round(nbytes / call_us / 1e3 / peaks["hbm_gbs"], 3),
                                   roofline_us=round(roof_us, 2),
                                   call_frac_of_roofline=round(roof_us / call_us, 3),
                                   gemm_frac_of_roofline=round(roof_us / gemm_us, 3))

    # ---------------------------------------------------------------- CPU baseline (oracle)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = np.sort(np.random.default_rng(99).choice(T, args.cpu_rows, replace=False))
        dt = time_oracle(b, rows)
        cpu = dict(value=args.cpu_rows / dt, unit="tokens/s", cores=cpu_cores(), kind="oracle",
                   sample=f"{args.cpu_rows} seeded rows of this workload (trainer set) scored by "
                          f"the fp64 numpy oracle plus their compare; {dt:.1f} s")

    if rank == 0:
        line = dict(
            metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=args.steps,
            warmup=max(args.warmup, 3), ms_per_step=ms_per_step, higher_is_better=True,
            scaling="weak", vs_baseline=None, dtype="bf16", data="synthetic",
            config=dict(workload=WORKLOAD, T=T, d=d, V=V, temperature=tau, l2=L2_NOTE,
                        parallelism=f"dp{world} (independent row batches per GPU)"),
            roofline=dict(bound="tensor", achieved=achieved_tflops, peak=peak, unit="TFLOP/s",
                          frac=achieved_tflops / peak, traffic=traffic_per_launch(T),
                          traffic_unit="DRAM bytes per launch (one-pass ncu capture of this launch)",
                          algorithmic_bytes=2.0 * V * d + 2.0 * T * d,
                          kernel="lmhead_lse_kernel",
                          peak_source=(f"{peaks['source']} bf16 "
                                       f"{'burst' if short_region else 'sustained'}"
                                       f" (timed region {total_ms / 1e3:.2f} s)"),
                          frac_secondary=achieved_tflops / peak_other,
                          peak_secondary=peak_other,
                          peak_secondary_source=(f"{peaks['source']} bf16 "
                                                 f"{'sustained' if short_region else 'burst'}"),
                          tflops_per_sm_ghz=(achieved_tflops / (clk["sm_mhz"] / 1e3)
                                             if clk and clk.get("sm_mhz") else None),
                          step_frac=(value / world) * 2.0 * d * V / 1e12 / peak),
            stage_ms=dict(rmsnorm=norm_ms, lmhead_lse=gemm_ms, finalize=fin_ms,
                          compare=ms_per_step - norm_ms - gemm_ms - fin_ms),
            cpu_baseline=cpu,
            e2e=dict(value=e2e_value, unit="tokens/s", h2d_bytes_per_step=h2d,
                     d2h_bytes_per_step=d2h, steps=e2e_steps,
                     note="pinned host buffers; the copies of step k+1 overlap step k"),
            # per step: RMSNorm, LM head, finalize, the compare's part numbering, compare
            gpu_launches=5 * args.steps,
            clocks=clk,
            compare=compare_info,
            decode_shapes=decode,
            next_rows=extras,
        )
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
