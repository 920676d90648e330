"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long]

One step = one ``attn_fwd`` call over one batch of the workload (the whole
hot path: a single fused kernel).  ``--path fp8`` times ``attn_fwd_fp8`` on
the workload's inputs quantised to e4m3, ``--path bwd`` times ``attn_bwd``,
``--path kvcache --nq Q`` times ``attn_fwd_kvcache`` with Q new queries against
the workload's K/V as the cache (its roofline is HBM bandwidth) -- the same
JSON line, with their own metric names.  The default workload is the long-sequence
causal configuration the throughput target is stated on: B=1, H=32, N=16384,
d=128, bf16, causal, Q,K,V ~ N(0,1) with 1% of the K rows scaled by 8.

Prints ONE JSON line (rank 0).  ``value`` is TFLOP/s with the inputs resident
in HBM (4*B*H*N^2*d FLOPs, halved for causal, counted per rank and summed over
ranks, divided by the slowest rank's time); ``e2e`` is the same metric through
the public API with pinned host buffers, the host->device copies of Q, K, V
and the device->host copies of O and LSE inside the timed region.

--impl reference times the fp64 CPU oracle (as it stands) on the host cores,
on bounded row samples of the same workload.  Under torchrun only rank 0 does
that; the other ranks exit without work.
"""
from __future__ import annotations

import argparse
import glob
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_attention_51_gb300 import workloads as wl  # noqa: E402

METRIC = "attention fwd TFLOP/s (bf16, causal/non-causal) and % of GB300 dense BF16 peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# The GB300 dense bf16 figure from NVIDIA's specification, reported beside the
# measured peak (which the roofline uses).
SPEC_BF16_TFLOPS = 2500.0
SPEC_SOURCE = ("NVIDIA GB300 NVL72 specification: 360 PFLOP/s bf16 with 2:4 sparsity "
               "/ 72 GPUs / 2 (dense)")
# Length of the untimed soak before the timed region, and of the default
# timed region.
SOAK_S = 1.0
# Device buffer sets the end-to-end loop rotates through.
E2E_SETS = 3
# The sources that build the bf16 forward kernel this benchmark times: a
# committed DRAM-traffic figure is used only while they hash to what was
# profiled.
KERNEL_SOURCES = ["exact_attention_51_gb300/csrc/attn_fwd_kernel.cuh",
                  "exact_attention_51_gb300/csrc/ptx.cuh",
                  "exact_attention_51_gb300/csrc/launch.cuh",
                  "exact_attention_51_gb300/csrc/fwd_dispatch.h",
                  "exact_attention_51_gb300/csrc/attn_fwd_d*.cu",
                  "exact_attention_51_gb300/csrc/attn_api.cu"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for pat in KERNEL_SOURCES:
        for f in sorted(glob.glob(os.path.join(ROOT, pat))):
            h.update(os.path.basename(f).encode())
            h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str, causal: bool):
    """DRAM bytes per launch from a committed ncu capture, if the kernel
    sources still hash to what was profiled."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    key = f"{workload}-{'causal' if causal else 'full'}"
    e = d.get(key)
    if not e or e.get("kernel_source_sha") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------ second bounds

L2_BYTES = 129 * 1024 * 1024
L2_FLUSH_BYTES = 256 * 1024 * 1024
# Exponentials per clock per SM on GB300 (its special-function units run ex2
# at twice the B200 rate); the unit count of the device, at the SM clock
# sampled during the run, gives the second (ALU) bound of the softmax.
EX2_PER_CLK_PER_SM = 32


def percentiles(xs):
    if not xs:
        return None
    ys = sorted(xs)
    pick = lambda f: ys[min(len(ys) - 1, int(round(f * (len(ys) - 1))))]
    return {"p10": pick(0.1), "p50": pick(0.5), "p90": pick(0.9), "n": len(ys)}


def exp_bound(w, causal, ms, clocks, per_score=1.0):
    """Exponentials per step (per_score per visible score) against the SFU
    rate."""
    import torch
    exps = per_score * w.B * w.H * w.N * w.N * (0.5 if causal else 1.0)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = (clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz") or 2070.0
    peak = EX2_PER_CLK_PER_SM * sms * mhz * 1e6
    achieved = exps / (ms * 1e-3)
    return {"exps": exps, "achieved_per_s": achieved, "peak_per_s": peak, "frac": achieved / peak,
            "peak_source": f"{EX2_PER_CLK_PER_SM} ex2/clk/SM x {sms} SMs x {mhz:.0f} MHz"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples with host arrival times."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", gpu_id, "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [(t, s) for t, s in self.samples if t0 <= t <= t1 + 0.06]
        if not rows:  # timed region shorter than one sampling interval
            before = [(t, s) for t, s in self.samples if t <= t1 + 0.06]
            rows = before[-1:]
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, s in rows:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = max(smax, float(f[2]))
            except ValueError:
                continue
            for name, flag in zip(names, f[5:9]):
                if flag.lower() in ("active", "0x1", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": smax or None, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[device_index]
        return str(device_index)


# ---------------------------------------------------------------- CPU oracle

def row_flops(w: wl.Workload, causal: bool, rows) -> float:
    """Algorithmic FLOPs of the listed rows (4*d per visible key)."""
    if not causal:
        return 4.0 * w.d * w.N * len(rows)
    return float(sum(4.0 * w.d * ((r % w.N) + 1) for r in rows))


def time_oracle_tiny_one_thread(reps: int = 20):
    """Median wall time (us) of the oracle on one thread over the whole tiny
    workload (B=1 H=2 N=128 d=64, non-causal), and its TFLOP/s."""
    import oracle
    orc = oracle.Oracle()
    w = wl.WORKLOADS["tiny"]
    q, k, v = wl.workload_inputs(w)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        orc.attn_bf16(q, k, v, False, w.scale, nthreads=1)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return t * 1e6, w.flops(False) / t / 1e12


def time_oracle(w, causal, q, k, v, target_s: float, seed: int):
    """Oracle throughput (TFLOP/s) on seeded random row samples, grown until
    one sample takes about `target_s` seconds; returns (tflops, seconds, rows,
    threads)."""
    import numpy as np
    import oracle
    orc = oracle.Oracle()
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.H * w.N
    n = 256
    while True:
        rows = sorted(rng.choice(total_rows, size=min(n, total_rows), replace=False).tolist())
        t0 = time.perf_counter()
        orc.attn_bf16_rows(q, k, v, causal, w.scale, rows)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or len(rows) == total_rows:
            return row_flops(w, causal, rows) / dt / 1e12, dt, len(rows), orc.max_threads()
        n = int(len(rows) * min(8.0, max(1.5, target_s / max(dt, 1e-3))))


# ---------------------------------------------------------------- main arms

def reduce_max_over_ranks(values, device):
    """Element-wise max of `values` over all ranks (identity when not
    distributed).  The only collective in the benchmark; the data path has
    none."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_tflops(flops_per_rank: float, world: int, slowest_ms: float) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return world * flops_per_rank / (slowest_ms * 1e-3) / 1e12


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, w, causal):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    q, k, v = wl.workload_inputs(w)
    import numpy as np
    import oracle
    orc = oracle.Oracle()
    rng = np.random.default_rng(12345)
    total_rows = w.B * w.H * w.N
    # size each step to ~2 s of oracle work so K + W steps stay within minutes
    n = 256
    while True:
        rows = sorted(rng.choice(total_rows, size=min(n, total_rows), replace=False).tolist())
        t0 = time.perf_counter()
        orc.attn_bf16_rows(q, k, v, causal, w.scale, rows)
        dt = time.perf_counter() - t0
        if dt >= 1.0 or len(rows) == total_rows:
            break
        n = int(len(rows) * min(8.0, max(1.5, 2.0 / max(dt, 1e-3))))
    n = len(rows)
    times, flops = [], []
    for step in range(args.warmup + args.steps):
        rows = sorted(rng.choice(total_rows, size=n, replace=False).tolist())
        t0 = time.perf_counter()
        orc.attn_bf16_rows(q, k, v, causal, w.scale, rows)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            flops.append(row_flops(w, causal, rows))
    value = sum(flops) / sum(times) / 1e12
    sample = (f"{n} seeded random rows of {w.describe(causal)} per step "
              f"(full workload: {total_rows} rows)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.describe(causal), "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": causal, "sample_rows_per_step": n},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": orc.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


class BenchPath:
    """One benchmarked entry point: its host inputs (copied in every e2e
    step), the device buffers of one step, the call, and its accounting."""

    def __init__(self, name, metric, dtype, flops, launches, kernel, peak_mult, host_inputs,
                 make_outputs, make_scratch, call, out_names):
        self.name, self.metric, self.dtype = name, metric, dtype
        self.flops, self.launches, self.kernel, self.peak_mult = flops, launches, kernel, peak_mult
        self.host_inputs = host_inputs      # dict name -> CPU tensor
        self.make_outputs = make_outputs    # dev -> dict name -> device tensor
        self.make_scratch = make_scratch    # dev -> device scratch tensor or None
        self.call = call                    # (inputs, outputs, scratch, stream) -> None
        self.out_names = out_names          # outputs copied back in the e2e loop
        self.min_bytes = None               # HBM-bound paths: bytes read and written at least

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host_inputs.values())


def make_path(args, w, causal, ea, dev):
    import torch
    scale = w.scale
    if args.path == "fwd":
        q, k, v = wl.workload_inputs(w)
        splits = 1 if args.splits is None else args.splits
        if splits == 0:
            splits = ea.attn_fwd_splitkv_num_splits(
                w.B, w.H, w.N, w.d, causal, torch.cuda.get_device_properties(dev).multi_processor_count)
        ws_bytes = ea.attn_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.d, splits) if splits > 1 else 0

        def call(i, o, scratch, st):
            if splits > 1:
                ea.attn_fwd_splitkv(i["q"], i["k"], i["v"], causal=causal, num_splits=splits,
                                    out=o["o"], lse=o["lse"], workspace=scratch, stream=st)
            else:
                ea.attn_fwd(i["q"], i["k"], i["v"], causal=causal, out=o["o"], lse=o["lse"], stream=st)
        p = BenchPath("fwd", METRIC, "bf16", w.flops(causal), 2 if splits > 1 else 1,
                      f"attn_fwd_kernel<{w.d},{str(causal).lower()}>", 1.0,
                      {"q": q, "k": k, "v": v},
                      lambda d: {"o": torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=d),
                                 "lse": torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=d)},
                      lambda d: torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=d),
                      call, ["o", "lse"])
        p.splits = splits
        return p
    if args.path == "kvcache":
        # Nq new queries against the workload's K/V as a cache of Nk = N keys
        # (bottom-right causal), e.g. a decoding step: HBM-bound.
        nq = args.nq
        _, k, v = wl.workload_inputs(w)
        q = wl.make_inputs(w.B, w.H, nq, w.d, w.dist, w.seed + 700)[0]
        splits = 0 if args.splits is None else args.splits
        if splits == 0:
            splits = ea.attn_fwd_kvcache_num_splits(
                w.B, w.H, nq, w.N, w.d, causal, torch.cuda.get_device_properties(dev).multi_processor_count)
        ws_bytes = ea.attn_fwd_splitkv_workspace_size(w.B, w.H, nq, w.d, splits) if splits > 1 else 0
        # visible (query, key) pairs: query i of nq sees keys j <= i + N - nq
        pairs = w.N * nq - (nq * (nq - 1) // 2 if causal else 0)

        def call(i, o, scratch, st):
            ea.attn_fwd_kvcache(i["q"], i["k"], i["v"], causal=causal, num_splits=splits, out=o["o"],
                                lse=o["lse"], workspace=scratch, stream=st)
        p = BenchPath("kvcache", f"attention fwd with a KV cache ({nq} queries against N keys) "
                      "TFLOP/s and HBM GB/s", "bf16", 4.0 * w.B * w.H * pairs * w.d,
                      2 if splits > 1 else 1,
                      f"attn_fwd_kernel<{w.d},{str(causal).lower()}>" + (" + merge" if splits > 1 else ""),
                      1.0, {"q": q, "k": k, "v": v},
                      lambda d: {"o": torch.empty((w.B, w.H, nq, w.d), dtype=torch.bfloat16, device=d),
                                 "lse": torch.empty((w.B, w.H, nq), dtype=torch.float32, device=d)},
                      lambda d: torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=d),
                      call, ["o", "lse"])
        p.splits = splits
        # Q, K, V read and O, LSE written once
        p.min_bytes = w.B * w.H * (2 * nq * w.d * 2 + 2 * w.N * w.d * 2 + nq * 4)
        return p
    if args.path == "fp8":
        q8, k8, v8, sc = wl.make_inputs_e4m3(w.B, w.H, w.N, w.d, w.dist, w.seed, w.k_outlier_frac)
        ws_bytes = ea.attn_fwd_fp8_workspace_size(w.B, w.H, w.N, w.d)  # > 0: V read transposed

        def call(i, o, scratch, st):
            ea.attn_fwd_fp8(i["q"], i["k"], i["v"], *sc, causal=causal, out=o["o"], lse=o["lse"],
                            workspace=scratch, stream=st)
        p = BenchPath("fp8", "attention fwd TFLOP/s (e4m3 Q/K/V, per-tensor scales) and % of "
                      "GB300 dense FP8 peak", "e4m3", w.flops(causal), 2 if ws_bytes else 1,
                      f"attn_fwd_kernel<{w.d},{str(causal).lower()},e4m3>"
                      + (" + V transpose" if ws_bytes else ""),
                      2.0,  # dense fp8 : bf16 tensor rate (4.5 : 2.25 PFLOP/s nominal)
                      {"q": q8, "k": k8, "v": v8},
                      lambda d: {"o": torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=d),
                                 "lse": torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=d)},
                      lambda d: torch.empty(ws_bytes, dtype=torch.uint8, device=d) if ws_bytes else None,
                      call, ["o", "lse"])
        p.splits = 1
        return p
    # backward: Q, K, V, the forward's O and LSE, and dO are the inputs
    q, k, v = wl.workload_inputs(w)
    g = wl.make_inputs(w.B, w.H, w.N, w.d, w.dist, w.seed + 500)[0]
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o, lse = ea.attn_fwd(qd, kd, vd, causal=causal)
    o_h, lse_h = o.cpu(), lse.cpu()
    del qd, kd, vd, o, lse
    ws_bytes = ea.attn_bwd_workspace_size(w.B, w.H, w.N)

    def call(i, o, scratch, st):
        ea.attn_bwd(i["q"], i["k"], i["v"], i["o"], i["lse"], i["do"], causal=causal,
                    dq=o["dq"], dk=o["dk"], dv=o["dv"], workspace=scratch, stream=st)
    p = BenchPath("bwd", "attention bwd TFLOP/s (bf16; 2.5x the forward's algorithmic FLOPs) and % "
                  "of GB300 dense BF16 peak", "bf16", 2.5 * w.flops(causal), 4 if w.d == 256 else 3,
                  "attn_bwd: row statistics + dV + dK + dQ kernels" if w.d == 256 else
                  "attn_bwd: row statistics + dK/dV + dQ kernels", 1.0,
                  {"q": q, "k": k, "v": v, "o": o_h, "lse": lse_h, "do": g},
                  lambda d: {n: torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=d)
                             for n in ("dq", "dk", "dv")},
                  lambda d: torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=d),
                  call, ["dq", "dk", "dv"])
    p.splits = 1
    return p


def run_ours(args, w, causal):
    import torch
    import torch.distributed as dist

    import exact_attention_51_gb300 as ea
    from exact_attention_51_gb300 import build as eabuild

    ws, rank, local = dist_setup()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    eabuild.build()
    ea.load_library()

    path = make_path(args, w, causal, ea, dev)
    ins = {n: t.to(dev) for n, t in path.host_inputs.items()}
    outs = path.make_outputs(dev)
    scratch = path.make_scratch(dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws > 1:
            dist.barrier()

    def step(st=None):
        path.call(ins, outs, scratch, st)

    # ---- device-resident timing
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, detail = ea.attn_fwd_device_status()
    if st != ea.ATTN_OK:
        raise RuntimeError(f"device wait timed out during warm-up (code {detail:#x})")
    # the length of one step, to size the soak and the default step count
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_a.record(stream)
    for _ in range(3):
        step()
    ev_b.record(stream)
    torch.cuda.synchronize(dev)
    est_ms = reduce_max_over_ranks([max(ev_a.elapsed_time(ev_b) / 3, 1e-3)], dev)[0]
    if args.steps is None:  # default: a timed region of about SOAK_S
        args.steps = min(1000, max(20, int(math.ceil(SOAK_S * 1e3 / est_ms))))
    soak_steps = min(20000, int(math.ceil(args.soak_seconds * 1e3 / est_ms)))

    # Inputs and outputs smaller than twice L2 would be served from L2 on
    # repeated launches: then every step is timed on its own, after a write
    # of L2_FLUSH_BYTES that evicts them.
    io_bytes = path.h2d_bytes() + sum(t.numel() * t.element_size() for t in outs.values())
    flush = io_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev) if flush else None
    sampler = ClockSampler(gpu_id_for(local))
    time.sleep(0.3)  # let nvidia-smi start printing
    per_step = []
    # Untimed soak right before the timed region: about SOAK_S of back-to-back
    # steps, so that the timed steps start at the clocks and power of a
    # sustained run and the clock samples cover more than a few steps.
    barrier()
    t_soak0 = time.monotonic()
    for _ in range(soak_steps):
        step()
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.monotonic()
    if flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            flush_buf.zero_()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        per_step = [a.elapsed_time(b) for a, b in evs]
        ms = sum(per_step) / len(per_step)
    else:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        ms = ev0.elapsed_time(ev1) / args.steps
    t_host1 = time.monotonic()
    barrier()
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)
    clocks_soak = sampler.summary(t_soak0, t_host0)
    if not flush:
        # step-by-step spread, outside the timed region above
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(args.steps, 50))]
        for a, b in evs:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        per_step = [a.elapsed_time(b) for a, b in evs]
    del flush_buf
    st, detail = ea.attn_fwd_device_status()
    if st != ea.ATTN_OK:
        raise RuntimeError(f"device wait timed out in the timed region (code {detail:#x})")

    # ---- end to end: pinned host buffers, copies inside the timed region.
    # E2E_SETS device buffer sets; step i copies its inputs in on an H2D
    # stream, computes on the compute stream and copies the results out on a
    # D2H stream, so the copies of one step overlap the kernels and the
    # copies of the neighbouring steps (the copy engines and the SMs are
    # separate hardware).  With three sets the H2D stream never waits for a
    # step's results to leave before it loads the step after next.
    nset = E2E_SETS
    pinned = {n: t.pin_memory() for n, t in path.host_inputs.items()}
    back = [{n: torch.empty(outs[n].shape, dtype=outs[n].dtype).pin_memory() for n in path.out_names}
            for _ in range(nset)]
    bufs = [dict(ins={n: torch.empty_like(t) for n, t in ins.items()}, outs=path.make_outputs(dev),
                 scratch=path.make_scratch(dev)) for _ in range(nset)]
    del ins, outs, scratch
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nset)]
    ev_done = [torch.cuda.Event() for _ in range(nset)]
    ev_free = [torch.cuda.Event() for _ in range(nset)]
    for e in ev_free:
        e.record(s_d2h)

    def e2e_step(i):
        b = bufs[i % nset]
        s_h2d.wait_event(ev_free[i % nset])
        with torch.cuda.stream(s_h2d):
            for n, t in pinned.items():
                b["ins"][n].copy_(t, non_blocking=True)
            ev_in[i % nset].record(s_h2d)
        stream.wait_event(ev_in[i % nset])
        path.call(b["ins"], b["outs"], b["scratch"], stream)
        ev_done[i % nset].record(stream)
        s_d2h.wait_event(ev_done[i % nset])
        with torch.cuda.stream(s_d2h):
            for n in path.out_names:
                back[i % nset][n].copy_(b["outs"][n], non_blocking=True)
            ev_free[i % nset].record(s_d2h)

    for i in range(max(1, min(args.warmup, 3))):
        e2e_step(i)
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_d2h)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    st, detail = ea.attn_fwd_device_status()
    if st != ea.ATTN_OK:
        raise RuntimeError(f"device wait timed out in the end-to-end loop (code {detail:#x})")
    h2d = path.h2d_bytes()
    d2h = sum(back[0][n].numel() * back[0][n].element_size() for n in path.out_names)

    # ---- max over ranks
    ms, e2e_ms = reduce_max_over_ranks([ms, e2e_ms], dev)

    if rank == 0:
        peaks, peak_src = load_peaks()
        # A timed region that follows the soak runs at the clocks of a
        # sustained load (under the power cap), so its denominator is the
        # sustained cuBLAS figure; without a soak the steps are timed as a
        # burst.  Both fractions are reported.
        sustained = soak_steps > 0
        burst_peak = peaks["bf16_tflops"] * path.peak_mult
        sust_peak = peaks["bf16_tflops_sustained"] * path.peak_mult
        peak = sust_peak if sustained else burst_peak
        achieved = path.flops / (ms * 1e-3) / 1e12
        min_bytes = path.min_bytes or (w.min_hbm_bytes() if path.name == "fwd" else None)
        traffic = load_traffic(args.workload, causal) if path.name == "fwd" else None
        q_bytes = w.B * w.H * w.N * w.d * 2
        line = {
            "metric": path.metric,
            "value": whole_job_tflops(path.flops, ws, ms),
            "unit": "TFLOP/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": path.dtype,
            "data": "synthetic",
            "config": {"workload": w.describe(causal), "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": causal, "scale": w.scale, "path": path.name,
                       "l2": ("L2 flushed (%d MiB write) before each step; per-step CUDA "
                              "events" % (L2_FLUSH_BYTES >> 20)) if flush else
                             ("inputs larger than L2 (3 x %d MiB bf16), no flush" % (q_bytes >> 20)),
                       "parallelism": f"replicas x{ws} (independent batches, no collective)",
                       "kv_splits": path.splits},
            "pct_of_peak": 100.0 * achieved / peak,
            "pct_of_spec_peak": 100.0 * achieved / (SPEC_BF16_TFLOPS * path.peak_mult),
            "spec_peak": {"tflops": SPEC_BF16_TFLOPS * path.peak_mult,
                          "frac": achieved / (SPEC_BF16_TFLOPS * path.peak_mult),
                          "source": SPEC_SOURCE + (" x 2 (fp8 : bf16)" if path.peak_mult == 2.0
                                                   else "")},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": traffic,
                         "peak_source": f"{peak_src} bf16 " + (
                             "sustained (timed steps follow a soak at the power cap)" if sustained
                             else "burst") + (
                             " x 2 (nominal fp8 : bf16 rate)" if path.peak_mult == 2.0 else ""),
                         "frac_of_burst_peak": achieved / burst_peak,
                         "frac_of_sustained_peak": achieved / sust_peak,
                         "kernel": path.kernel},
            "latency_ms": percentiles(per_step),
            "exp_bound": (exp_bound(w, causal, ms, clocks, 2.0 if path.name == "bwd" else 1.0)
                          if path.name != "kvcache" else None),
            "hbm": {"min_bytes": min_bytes,
                    "achieved_gbs": min_bytes / (ms * 1e-3) / 1e9,
                    "frac": min_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                    "peak_source": f"{peak_src} copy"} if min_bytes else None,
            "clocks": clocks,
            "soak": {"steps": soak_steps, "seconds": t_host0 - t_soak0, "clocks": clocks_soak,
                     "what": "untimed back-to-back steps right before the timed region"},
            "e2e": {"value": whole_job_tflops(path.flops, ws, e2e_ms), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps": e2e_steps,
                    "how": "pinned host buffers; H2D, kernels and D2H on three streams, "
                           f"{E2E_SETS} device buffer sets rotating across steps"},
            "gpu_launches": args.steps * path.launches,
        }
        if path.name == "fwd":
            line["pct_of_bf16_peak"] = line["pct_of_peak"]
        if path.name == "kvcache":
            # a few queries against a long cache: the bytes, not the tensor
            # core, bound it
            gbs = min_bytes / (ms * 1e-3) / 1e9
            line["config"]["nq"] = args.nq
            line["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                                "peak_source": f"{peak_src} copy", "kernel": path.kernel}
        if ws == 1 and not args.no_cpu_baseline and path.name == "fwd":
            q_h, k_h, v_h = (path.host_inputs[n] for n in ("q", "k", "v"))
            tf, secs, nrows, cores = time_oracle(w, causal, q_h, k_h, v_h, args.cpu_seconds, 99)
            line["cpu_baseline"] = {
                "value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                "sample": f"{nrows} seeded random rows of {w.describe(causal)} "
                          f"({secs:.1f} s of fp64 oracle work)"}
            us1, tf1 = time_oracle_tiny_one_thread()
            line["cpu_baseline"]["tiny_one_thread"] = {
                "us": us1, "value": tf1, "unit": "TFLOP/s", "cores": 1,
                "sample": "the whole tiny workload, B=1 H=2 N=128 d=64 non-causal, median of 20"}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: as many as fill about one second, at least 20)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--causal", choices=["default", "0", "1"], default="default")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--soak-seconds", type=float, default=SOAK_S,
                    help="untimed back-to-back steps right before the timed region (0: none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["fwd", "fp8", "bwd", "kvcache"], default="fwd",
                    help="fwd: attn_fwd (bf16, the headline); fp8: attn_fwd_fp8 on the "
                         "workload's inputs quantised to e4m3; bwd: attn_bwd; kvcache: "
                         "attn_fwd_kvcache, --nq queries against the workload's K/V")
    ap.add_argument("--nq", type=int, default=16,
                    help="queries of the kvcache path (the workload's N is the key length)")
    ap.add_argument("--splits", type=int, default=None,
                    help="1: attn_fwd; >1: attn_fwd_splitkv with that many key splits; "
                         "0: the split count of the split model (default: 1 for fwd, 0 for "
                         "kvcache)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = wl.WORKLOADS[args.workload]
    causal = w.causal[-1] if args.causal == "default" else args.causal == "1"
    if args.path == "fp8" and w.d not in (64, 128, 256):
        ap.error("--path fp8 needs a d = 64, 128 or 256 workload")
    if args.path == "bwd" and w.d not in (64, 128, 256):
        ap.error("--path bwd needs a d = 64, 128 or 256 workload")
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        if args.path != "fwd":
            ap.error("--impl reference times the forward oracle only")
        return run_reference(args, w, causal)
    return run_ours(args, w, causal)


if __name__ == "__main__":
    sys.exit(main())
