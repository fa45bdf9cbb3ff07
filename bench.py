#!/usr/bin/env python3
"""Benchmark of the GB300 SGEMM library; prints one JSON line.

Default workload: FP32 SGEMM M=N=K=4092 (not a tile multiple), alpha=1,
beta=0.5, A, B, C uniform[-1,1) from seed 1 -- the configuration the headline
metric "SGEMM TFLOP/s at 4092^3 FP32" is quoted on.  One step is one sgemm()
call through the C ABI (validate -> choose kernel -> encode TMA descriptors ->
launch the FFMA kernel), with the operands resident in HBM.

  value        2*M*N*K*steps*world / max-over-ranks device time (TFLOP/s)
  e2e          the same through sgemm_host, the C ABI's host-buffer entry
               point: each step copies A, B, C host->device from pinned
               memory and C back, overlapped with the compute in row panels
  roofline     the FFMA kernel against the FP32 FFMA peak
               (SMs x 128 lanes x 2 FLOP x max SM clock): "bound": "alu"
  cpu_baseline the fp64 oracle on host cores on a bounded row sample
  parity       the timed launch's result against the oracle (every element)
  secondary    128^3 (time only), decode shapes (GB/s vs measured HBM copy
               bandwidth, B rotating through buffers larger than L2 together),
               8192^3 on all four arithmetics, the prefill GEMMs and medium
               shapes, on the seeded synthetic inputs of each workload, each
               with its own parity check

`--impl reference` times the oracle itself (the reference arm).  Under
torchrun each rank runs an independent replica (weak scaling); timing is the
max over ranks.
"""

from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SGEMM TFLOP/s at 4092³ FP32 (% of FP32 peak); GB/s (% HBM) on M≤16 shapes"
L2_BYTES = 129 * 10**6
# Best figure the pages print for this metric and workload: cuBLAS FP32 on an
# RTX A6000 at 4092^3, 23,249.6 GFLOP/s ("CUDA 矩阵乘法优化：从朴素 Kernel 到接近
# cuBLAS", results table).  Another machine: context, not the target.
PAGES_BEST_TFLOPS = 23.2496

# --mode names -> the binding's arithmetic mode
MODES = {"fp32": lambda sg: sg.MODE_FP32, "3xtf32": lambda sg: sg.MODE_3XTF32,
         "tf32": lambda sg: sg.MODE_TF32, "bf16": lambda sg: sg.MODE_BF16}

KERNEL_SOURCES = {
    "ffma_tma": ["dense_fp32_matrix_row_gb300/csrc/ffma_tma.cu",
                 "dense_fp32_matrix_row_gb300/csrc/ffma_tuning.inc",
                 "dense_fp32_matrix_row_gb300/csrc/common.cuh"],
    "decode": ["dense_fp32_matrix_row_gb300/csrc/decode.cu",
               "dense_fp32_matrix_row_gb300/csrc/common.cuh"],
    "tf32x3": ["dense_fp32_matrix_row_gb300/csrc/tf32x3.cu",
               "dense_fp32_matrix_row_gb300/csrc/common.cuh"],
}


_TOKENS = re.compile(r'"(?:\\.|[^"\\])*"|//[^\n]*|/\*.*?\*/', re.S)


def _code_only(text: str) -> str:
    """C++ source without its comments and with whitespace collapsed, so that
    editing a comment does not count as changing a kernel."""
    text = _TOKENS.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return " ".join(text.split())


def source_hash(kernel: str) -> str:
    """Hash of the code (comments excluded) of the files a kernel is built from."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        p = os.path.join(ROOT, rel)
        if os.path.exists(p):
            h.update(_code_only(open(p, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "_source": "fallback"}


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel, {}).get(workload)
    if not d or d.get("source_hash") != source_hash(kernel):
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="sgemm_bench_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0: float, t1: float):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10], parts[5]))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])),
                "sm_max_mhz": float(max(r[2] for r in inside)),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------ helpers
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier_max(value: float, world: int, device=None) -> float:
    """Max of `value` over all ranks (a timing scalar, not data).  Works on the
    NCCL group the bench uses on GPUs and on a gloo group (CPU tensors)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    if dist.get_backend() != "nccl":
        device = "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


def time_oracle(M, N, K, alpha, beta, A, B, C0, budget_s: float, threads: int = 0):
    """Time the oracle on a leading row sample sized to ~budget_s seconds.
    Returns (flop/s, rows, seconds, threads)."""
    import oracle
    orc = oracle.default()
    probe = max(1, min(M, 8))
    t = time.perf_counter()
    orc.sgemm(A, B, C0, alpha=alpha, beta=beta, rows=np.arange(probe), threads=threads)
    per_row = (time.perf_counter() - t) / probe
    rows = int(max(1, min(M, budget_s / max(per_row, 1e-9))))
    t = time.perf_counter()
    orc.sgemm(A, B, C0, alpha=alpha, beta=beta, rows=np.arange(rows), threads=threads)
    dt = time.perf_counter() - t
    return 2.0 * rows * N * K / dt, rows, dt, (threads or orc.max_threads())


def workload_config(name, w, extra=None):
    cfg = {"workload": f"{name}: FP32 SGEMM M={w['M']} N={w['N']} K={w['K']} row-major, "
                       f"alpha={w['alpha']} beta={w['beta']}, seed {w['seed']}",
           "M": w["M"], "N": w["N"], "K": w["K"], "alpha": w["alpha"], "beta": w["beta"]}
    cfg.update(extra or {})
    return cfg


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import synth
    name = args.workload
    A, B, C0, w = synth.workload_inputs(name)
    M, N, K = w["M"], w["N"], w["K"]
    import oracle
    orc = oracle.default()
    # Size each step so the whole run stays near args.ref_budget seconds.
    probe = max(1, min(M, 4))
    t = time.perf_counter()
    orc.sgemm(A, B, C0, alpha=w["alpha"], beta=w["beta"], rows=np.arange(probe))
    per_row = (time.perf_counter() - t) / probe
    steps_total = args.steps + args.warmup
    rows = int(max(1, min(M, args.ref_budget / steps_total / max(per_row, 1e-9))))
    sel = [np.arange(s * rows, s * rows + rows) % M for s in range(steps_total)]
    for s in range(args.warmup):
        orc.sgemm(A, B, C0, alpha=w["alpha"], beta=w["beta"], rows=sel[s])
    t0 = time.perf_counter()
    for s in range(args.warmup, steps_total):
        orc.sgemm(A, B, C0, alpha=w["alpha"], beta=w["beta"], rows=sel[s])
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K * args.steps
    value = flops / dt / 1e12
    sample = (f"{rows} of {M} rows of C per step ({rows * N * K * 2 / 1e9:.2f} GFLOP), "
              f"{args.steps} timed steps after {args.warmup} warm-up")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(name, w, {"parallelism": "host cores, OpenMP over rows"}),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": orc.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def timed_steps(fn, steps, stream):
    """Run fn() `steps` times on `stream`, each bracketed by CUDA events.
    Returns (total ms first-start..last-end, mean per-launch ms)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    total = evs[0][0].elapsed_time(evs[-1][1])
    per = float(np.mean([s.elapsed_time(e) for s, e in evs]))
    return total, per


def roofline_for(kid, M, N, K, beta, per_launch_ms, kernel_ms, sms, peaks):
    """(bound, achieved, peak, unit, peak_source) of the main line: the FFMA
    path against the FP32 FFMA peak (the tile kernel's own time when
    kernel_ms is given, else the whole call), the tensor-core paths against
    the tensor peak of their operand type (3xTF32 counts its three TF32
    products), the decode path against the measured copy bandwidth."""
    import dense_fp32_matrix_row_gb300 as sg
    from dense_fp32_matrix_row_gb300 import accounting as acc
    flops = acc.gemm_flops(M, N, K)
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    peak = acc.ffma_peak_tflops(sms, mhz)
    achieved = flops / ((kernel_ms or per_launch_ms) * 1e-3) / 1e12
    bound, unit = "alu", "TFLOP/s"
    peak_source = (f"{sms} SMs x 128 FP32 lanes x 2 FLOP x {mhz:.0f} MHz "
                   f"({peaks.get('_source', 'measured')} max clock)")
    if kid in (sg.KERNEL_TF32X3, sg.KERNEL_TF32, sg.KERNEL_BF16):
        bound = "tensor"
        if kid == sg.KERNEL_BF16:
            peak, peak_source = peaks["bf16_tflops"], "measured bf16 GEMM burst"
        else:
            peak = acc.tf32_peak_from_bf16(peaks["bf16_tflops"])
            peak_source = "measured bf16 GEMM burst x 1.1/2.25 (nominal TF32/BF16 ratio)"
        if kid == sg.KERNEL_TF32X3:
            achieved *= 3      # three TF32 products per useful product
    if kid == sg.KERNEL_DECODE:
        # M <= 16: bound by streaming B, measured against the copy bandwidth
        bound, unit = "hbm", "GB/s"
        achieved = acc.min_traffic_bytes(M, N, K, beta != 0.0) / (per_launch_ms * 1e-3) / 1e9
        peak, peak_source = peaks["hbm_gbs"], "measured HBM copy bandwidth"
    return bound, achieved, peak, unit, peak_source


def gate_err(got, ref, A, B, K, alpha, beta, C0, bias=None):
    """The acceptance gate as a number (<= 1e-6 passes): per element,
    |C - C_ref| against 1e-6*|alpha|*K*max|A|*max|B| plus, where beta != 0
    or a bias is added, 2^-22*(|beta*C0| + |bias| + |C_ref|) (the FP32
    rounding of those terms).  With beta = 0 and no bias it is
    max|C - C_ref| / (|alpha|*K*max|A|*max|B|) verbatim."""
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    diff = np.abs(got - ref)
    if diff.size == 0:
        return 0.0
    if np.isnan(diff).any():
        return float("inf")
    prod = 1e-6 * abs(alpha) * K * float(np.abs(A).max()) * float(np.abs(B).max())
    bound = np.full(diff.shape, prod)
    if (beta != 0.0 and C0 is not None) or bias is not None:
        t = np.abs(ref)
        if beta != 0.0 and C0 is not None:
            t = t + abs(beta) * np.abs(C0.astype(np.float64))
        if bias is not None:
            t = t + np.abs(bias.astype(np.float64)).reshape(1, -1)
        bound += 2.0 ** -22 * t
    return 1e-6 * float((diff / bound).max()) if prod > 0 else float(diff.max())


def sample_index(n: int, stride: int = 61):
    """Every stride-th index plus the last (stride 61 < every tile edge, so
    every tile row / column band is hit)."""
    return np.unique(np.r_[np.arange(0, n, stride), [n - 1]])


def parity_check(A, B, C0, alpha, beta, got, inputs="fp32", full_below_flop=4e10):
    """Compare a result with the fp64 oracle: every element when the product
    is small enough, else a cross of sampled rows and sampled columns (every
    61st plus the last), which covers every output tile.  Returns a dict."""
    import oracle
    M, K = A.shape
    N = B.shape[1]
    c0 = C0 if beta != 0.0 else None
    if 2.0 * M * N * K <= full_below_flop:
        ref = oracle.sgemm(A, B, c0, alpha=alpha, beta=beta, inputs=inputs)
        err = gate_err(got, ref, A, B, K, alpha, beta, c0)
        checked = f"all {M * N} elements"
    else:
        rows, cols = sample_index(M), sample_index(N)
        ref_r = oracle.sgemm(A, B, c0, alpha=alpha, beta=beta, rows=rows, inputs=inputs)
        Bc = np.ascontiguousarray(B[:, cols])
        c0c = np.ascontiguousarray(c0[:, cols]) if c0 is not None else None
        ref_c = oracle.sgemm(A, Bc, c0c, alpha=alpha, beta=beta, inputs=inputs)
        err = max(gate_err(got[rows], ref_r, A, B, K, alpha, beta, c0[rows] if c0 is not None else None),
                  gate_err(got[:, cols], ref_c, A, B, K, alpha, beta, c0c))
        checked = f"{rows.size} full rows + {cols.size} full columns (every 61st and the last)"
    return {"checked": checked, "normwise_err": err, "gate": 1e-6, "pass": bool(err <= 1e-6)}


def secondary(sg, torch, stream, dev, peaks, steps=20, warmup=3, check=True):
    """Device-timed secondary shapes on the seeded synthetic inputs of the
    named workloads (synth), each parity-checked against the oracle on its
    first call.  "ms" is per call in a replayed CUDA graph of `steps` calls;
    "ms_eager" per call with an event pair around each eager call."""
    import synth
    out = {}
    # the FP32 FFMA peak (SMs x 128 lanes x 2 FLOP x max clock), and the
    # measured bf16 x the nominal TF32 / BF16 ratio, burst and sustained
    ffma_peak = (torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2
                 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12)
    tf32_peak = peaks["bf16_tflops"] * 1.1 / 2.25
    tf32_peak_s = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * 1.1 / 2.25
    tf32_peak = peaks["bf16_tflops"] * 1.1 / 2.25   # measured bf16 x nominal tf32/bf16

    def capture(fns):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for f in fns:
                f()
        return graph

    def replay_ms(graph, n):
        """ms per call of one replay of a graph of n calls."""
        with torch.cuda.stream(stream):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def graph_ms(fns):
        """Mean ms per call of the calls `fns` captured in one CUDA graph:
        the median of three replays after one warm replay."""
        graph = capture(fns)
        replay_ms(graph, len(fns))
        ms = float(np.median([replay_ms(graph, len(fns)) for _ in range(3)]))
        del graph
        return ms

    def bench_shape(A, B, C0, alpha, beta, mode=sg.MODE_FP32, activation="none", rotate=1,
                    inputs="fp32", bias_seed=None, burst=False):
        """Parity of the first call, then timing.  With rotate > 1 the calls
        cycle through that many copies of B (distinct device buffers), so no
        call finds its B in L2 from the call before.  With `burst` (the
        tensor-core lines, whose speed depends on how long the GPU has been
        under load): "ms" is the graph replayed after a second of idling,
        "ms_sustained" the graph replayed again after about a second of
        back-to-back calls, and "ms_eager" follows, still under load."""
        M, K = A.shape
        N = B.shape[1]
        dA = torch.from_numpy(A).to(dev)
        dBs = [torch.from_numpy(B).to(dev) for _ in range(rotate)]
        dC = torch.from_numpy(C0).to(dev) if C0 is not None else torch.empty((M, N), device=dev)
        bias = None
        if activation != "none":
            bias = synth.matrix(1, N, seed=bias_seed, stream=3, dist="normal").reshape(-1)
        dbias = torch.from_numpy(bias).to(dev) if bias is not None else None
        fns = [(lambda dB=dB: sg.sgemm(dA, dB, dC, alpha, beta, stream=stream, tensor_cores=mode,
                                       bias=dbias, activation=activation)) for dB in dBs]
        res = {"shape": [M, N, K]}
        with torch.cuda.stream(stream):
            fns[0]()
        st = sg.status(stream)
        if check and activation == "none":
            res["parity"] = parity_check(A, B, C0, alpha, beta, dC.cpu().numpy(), inputs)
        elif check:
            import oracle
            rows = sample_index(M)
            ref = oracle.sgemm(A, B, C0 if beta != 0.0 else None, alpha=alpha, beta=beta,
                               rows=rows, bias=bias, act=activation, inputs=inputs)
            got = dC.cpu().numpy()[rows]
            err = gate_err(got, ref, A, B, K, alpha, beta,
                           C0[rows] if C0 is not None else None, bias)
            res["parity"] = {"checked": f"{rows.size} full rows", "normwise_err": err,
                             "gate": 1e-6, "pass": bool(err <= 1e-6)}
        for i in range(warmup):
            with torch.cuda.stream(stream):
                fns[i % rotate]()
        torch.cuda.synchronize()
        if burst:
            graph = capture([fns[i % rotate] for i in range(steps)])
            replay_ms(graph, steps)            # warm replay
            time.sleep(1.0)
            res["ms"] = replay_ms(graph, steps)
            t_end = time.time() + 1.0
            while time.time() < t_end:
                replay_ms(graph, steps)
            res["ms_sustained"] = replay_ms(graph, steps)
            del graph
        evs = []
        with torch.cuda.stream(stream):
            for i in range(steps):
                e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                e[0].record(stream)
                fns[i % rotate]()
                e[1].record(stream)
                evs.append(e)
        torch.cuda.synchronize()
        res["ms_eager"] = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        if not burst:
            res["ms"] = graph_ms([fns[i % rotate] for i in range(steps)])
        if rotate > 1:
            res["ms_same_buffer"] = graph_ms([fns[0]] * steps)
            res["b_buffers"] = rotate
        st = st or sg.status(stream)
        res["status"] = st
        kid = sg.select_kernel(M, N, K, alpha, dA.data_ptr(), K, dBs[0].data_ptr(), N, beta,
                               dC.data_ptr(), N, mode)
        res["kernel"] = sg.KERNEL_NAMES.get(kid, str(kid))
        del dA, dBs, dC, dbias
        return res

    def tflops(res, M, N, K, key="ms"):
        return 2.0 * M * N * K / (res[key] * 1e-3) / 1e12

    # 128^3: the overhead regime (a handful of tiles); time only, no roofline bar
    A, B, C0, w = synth.workload_inputs("sgemm_128")
    r = bench_shape(A, B, C0, w["alpha"], w["beta"])
    r["us"], r["us_eager"] = r["ms"] * 1e3, r["ms_eager"] * 1e3
    r["TFLOP/s"] = tflops(r, 128, 128, 128)
    r["note"] = "launch/overhead-bound: timed, no roofline bar"
    out["sgemm_128"] = r

    # decode: B (235 MB) streamed from HBM; three B buffers (705 MB > L2) rotate
    for M in (1, 4, 16):
        A, B, C0, w = synth.workload_inputs(f"decode_m{M}")
        N, K = w["N"], w["K"]
        r = bench_shape(A, B, C0, w["alpha"], w["beta"], rotate=3)
        nbytes = 4 * (M * K + K * N + M * N)
        r["GB/s"] = nbytes / (r["ms"] * 1e-3) / 1e9
        r["frac_hbm"] = r["GB/s"] / peaks["hbm_gbs"]
        r["GB/s_eager"] = nbytes / (r["ms_eager"] * 1e-3) / 1e9
        r["GB/s_same_buffer"] = nbytes / (r["ms_same_buffer"] * 1e-3) / 1e9
        r["TFLOP/s"] = tflops(r, M, N, K)
        r["l2"] = "B rotates through 3 buffers (705 MB > 129 MB L2); same-buffer figure as a side key"
        out[f"decode_m{M}"] = r
        del A, B

    # skinny products, 17 <= M <= 128 rows on the decode shapes' N and K (the
    # same B): HBM-bound below about 24 rows, FFMA-bound above
    for M in (32, 64, 128):
        A, B, C0, w = synth.workload_inputs(f"skinny_m{M}")
        N, K = w["N"], w["K"]
        r = bench_shape(A, B, C0, w["alpha"], w["beta"], rotate=3)
        nbytes = 4 * (M * K + K * N + M * N)
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e3
        t_alu = 2.0 * M * N * K / (ffma_peak * 1e12) * 1e3
        r["TFLOP/s"] = tflops(r, M, N, K)
        r["GB/s"] = nbytes / (r["ms"] * 1e-3) / 1e9
        r["bound"] = "alu" if t_alu >= t_hbm else "hbm"
        r["frac_bound"] = max(t_alu, t_hbm) / r["ms"]
        r["frac_ffma_peak"] = r["TFLOP/s"] / ffma_peak
        r["frac_hbm"] = r["GB/s"] / peaks["hbm_gbs"]
        r["l2"] = "B rotates through 3 buffers (705 MB > 129 MB L2)"
        out[f"skinny_m{M}"] = r
        del A, B

    # the compute-bound workloads on the FFMA path
    for name in ("sgemm_8192", "prefill_qkv", "prefill_up", "prefill_down"):
        A, B, C0, w = synth.workload_inputs(name)
        M, N, K = w["M"], w["N"], w["K"]
        r = bench_shape(A, B, C0, w["alpha"], w["beta"])
        r["TFLOP/s"] = tflops(r, M, N, K)
        r["frac_ffma_peak"] = r["TFLOP/s"] / ffma_peak
        out[name] = r
        if name == "prefill_up":
            # FFN-up with the fused epilogue act(X W + bias), SiLU
            r = bench_shape(A, B, C0, w["alpha"], w["beta"], activation="silu", bias_seed=w["seed"])
            r["TFLOP/s"] = tflops(r, M, N, K)
            r["frac_ffma_peak"] = r["TFLOP/s"] / ffma_peak
            r["epilogue"] = "bias + SiLU (sgemm_fused)"
            out["prefill_up_bias_silu"] = r
        if name == "sgemm_8192":
            # the tensor-core paths on the same operands: burst (after idling)
            # against the burst peak, sustained against the sustained peak
            r = bench_shape(A, B, C0, w["alpha"], w["beta"], mode=sg.MODE_3XTF32, burst=True)
            useful, useful_s = tflops(r, M, N, K), tflops(r, M, N, K, "ms_sustained")
            r.update({"TFLOP/s": useful, "tensor_TFLOP/s": 3 * useful, "tf32_peak": tf32_peak,
                      "frac_tf32_peak": 3 * useful / tf32_peak,
                      "frac_useful_ceiling": useful / (tf32_peak / 3),
                      "TFLOP/s_sustained": useful_s, "tf32_peak_sustained": tf32_peak_s,
                      "frac_tf32_peak_sustained": 3 * useful_s / tf32_peak_s,
                      "TFLOP/s_eager": tflops(r, M, N, K, "ms_eager")})
            out["sgemm_8192_3xtf32"] = r
            r = bench_shape(A, B, C0, w["alpha"], w["beta"], mode=sg.MODE_TF32, inputs="tf32",
                            burst=True)
            t, ts = tflops(r, M, N, K), tflops(r, M, N, K, "ms_sustained")
            r.update({"TFLOP/s": t, "tf32_peak": tf32_peak, "frac_tf32_peak": t / tf32_peak,
                      "TFLOP/s_sustained": ts, "tf32_peak_sustained": tf32_peak_s,
                      "frac_tf32_peak_sustained": ts / tf32_peak_s,
                      "TFLOP/s_eager": tflops(r, M, N, K, "ms_eager")})
            out["sgemm_8192_tf32"] = r
            r = bench_shape(A, B, C0, w["alpha"], w["beta"], mode=sg.MODE_BF16, inputs="bf16",
                            burst=True)
            t, ts = tflops(r, M, N, K), tflops(r, M, N, K, "ms_sustained")
            bf_s = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
            r.update({"TFLOP/s": t, "bf16_peak": peaks["bf16_tflops"],
                      "frac_bf16_peak": t / peaks["bf16_tflops"],
                      "TFLOP/s_sustained": ts, "bf16_peak_sustained": bf_s,
                      "frac_bf16_peak_sustained": ts / bf_s,
                      "TFLOP/s_eager": tflops(r, M, N, K, "ms_eager")})
            out["sgemm_8192_bf16"] = r
        del A, B

    # Medium shapes whose last wave is split along K, and skinny-M shapes.
    # Their operands (4-34 MB) stay in L2 between calls.
    mid = [("mid_1024", 1024, 1024, 1024), ("mid_1024x1024x8192", 1024, 1024, 8192),
           ("mid_512x512x8192", 512, 512, 8192), ("mid_2048", 2048, 2048, 2048)]
    for i, (name, M, N, K) in enumerate(mid):
        A = synth.matrix(M, K, seed=10 + i, stream=0, dist="normal")
        B = synth.matrix(K, N, seed=10 + i, stream=1, dist="normal")
        r = bench_shape(A, B, None, 1.0, 0.0)
        r["TFLOP/s"] = tflops(r, M, N, K)
        r["frac_ffma_peak"] = r["TFLOP/s"] / ffma_peak
        r["l2_resident"] = True
        r["data"] = f"A, B normal(0,1), seed {10 + i}"
        out[name] = r
    return out


def run_ours(args, world, rank, local):
    import torch
    import dense_fp32_matrix_row_gb300 as sg
    import synth
    from dense_fp32_matrix_row_gb300 import accounting as acc

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sg.build()
    peaks = measured_peaks()

    name = args.workload
    A, B, C0, w = synth.workload_inputs(name)
    M, N, K, alpha, beta = w["M"], w["N"], w["K"], w["alpha"], w["beta"]
    stream = torch.cuda.Stream(device=dev)
    dA = torch.from_numpy(A).to(dev)
    dB = torch.from_numpy(B).to(dev)
    dC = torch.from_numpy(C0).to(dev) if C0 is not None else torch.empty((M, N), device=dev)
    mode_name = args.mode or ("3xtf32" if args.tensor_cores else "fp32")
    tc = MODES[mode_name](sg)
    kid = sg.select_kernel(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                           dC.data_ptr(), N, tc)
    # kernels one sgemm() call launches: the FFMA path transposes A first (and
    # sums a divided tail in a kernel of its own), the tensor-core paths
    # convert A and B first
    launches_per_call = {sg.KERNEL_FFMA_TMA: 2, sg.KERNEL_TF32X3: 3, sg.KERNEL_TF32: 3,
                         sg.KERNEL_BF16: 3}.get(kid, 1)
    if kid == sg.KERNEL_FFMA_TMA:
        launches_per_call += sg.ffma_tail_plan(M, N, K)["tail_sum"]

    def step():
        sg.sgemm(dA, dB, dC, alpha, beta, stream=stream, tensor_cores=tc)

    # Parity of this exact launch configuration on sampled rows, before timing.
    with torch.cuda.stream(stream):
        step()
    st = sg.status(stream)
    if st != sg.OK:
        raise SystemExit(f"kernel status {sg.status_string(st)}")
    parity = None
    inputs = {"tf32": "tf32", "bf16": "bf16"}.get(mode_name, "fp32")
    if rank == 0 and not args.no_parity:
        parity = parity_check(A, B, C0, alpha, beta, dC.cpu().numpy(), inputs,
                              full_below_flop=2e11)

    clocks = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else
                          int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    if rank == 0:
        clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        total_ms, per_launch_ms = timed_steps(step, args.steps, stream)
    t_wall1 = time.time()
    # The tile kernel's own time: the same steps again, with the library's
    # CUDA events around each tile-kernel launch.  A pass of its own, because
    # events between the transpose and the tile kernel keep the tile kernel
    # from starting its set-up during the transpose's tail (0.4% per call).
    kernel_ms = None
    if kid == sg.KERNEL_FFMA_TMA and not args.no_kernel_timing:
        sg.kernel_timing(True)
        try:
            with torch.cuda.stream(stream):
                timed_steps(step, args.steps, stream)
        finally:
            sg.kernel_timing(False)
        k_total, k_n = sg.kernel_timing_result()
        kernel_ms = k_total / k_n if k_n == args.steps else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if rank == 0:
        clocks.stop()
    st = sg.status(stream)
    if st != sg.OK:
        raise SystemExit(f"kernel status {sg.status_string(st)}")
    total_ms = barrier_max(total_ms, world, dev)
    flops = acc.gemm_flops(M, N, K)
    value = aggregate_tflops(flops, args.steps, world, total_ms)

    # End to end through the C ABI's host-buffer entry point (sgemm_host):
    # pinned host A, B, C; the library copies B and row panels of A and C up,
    # multiplies each panel as it arrives and copies C back, every step.
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = (torch.from_numpy(C0) if C0 is not None else torch.zeros((M, N))).pin_memory()
    e2e_parity = None
    if rank == 0 and not args.no_parity:
        with torch.cuda.stream(stream):
            sg.sgemm_host(hA, hB, hC, alpha, beta, stream=stream, tensor_cores=tc)
        if sg.status(stream) != sg.OK:
            raise SystemExit("kernel status after sgemm_host")
        e2e_parity = parity_check(A, B, C0, alpha, beta, hC.numpy().copy(), inputs,
                                  full_below_flop=2e11)
        if C0 is not None:
            hC.copy_(torch.from_numpy(C0))

    def e2e_step():
        # C is read and written in place: each step starts from the last
        # result (alpha*A@B + beta*C stays bounded for |beta| < 1)
        sg.sgemm_host(hA, hB, hC, alpha, beta, stream=stream, tensor_cores=tc)

    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    with torch.cuda.stream(stream):
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms, _ = timed_steps(e2e_step, e2e_steps, stream)
    e2e_ms = barrier_max(e2e_ms, world, dev)
    e2e_value = aggregate_tflops(flops, e2e_steps, world, e2e_ms)
    h2d = 4 * (M * K + K * N + (M * N if beta != 0.0 else 0))
    d2h = 4 * M * N

    sec = None
    if rank == 0 and not args.no_secondary:
        with torch.cuda.stream(stream):
            sec = secondary(sg, torch, stream, dev, peaks, check=not args.no_parity)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    props = torch.cuda.get_device_properties(dev)
    bound, achieved, peak, unit, peak_source = roofline_for(
        kid, M, N, K, beta, per_launch_ms, kernel_ms, props.multi_processor_count, peaks)
    traffic = ncu_traffic("ffma_tma", name) if kid == sg.KERNEL_FFMA_TMA else None
    cpu = None
    if not args.no_cpu_baseline:
        fl, rows, secs, thr = time_oracle(M, N, K, alpha, beta, A, B, C0, args.cpu_budget)
        cpu = {"value": fl / 1e12, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"rows 0..{rows - 1} of {M} ({rows / M:.1%} of the {name} work), "
                         f"{secs:.1f} s of fp64 triple loops"}
    csum = clocks.summary(t_wall0, t_wall1)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGES_BEST_TFLOPS,
        "vs_baseline_ref": "pages' cuBLAS FP32 on an RTX A6000 at 4092^3 (23.25 TFLOP/s): "
                           "another machine, context only",
        "dtype": {"tf32": "tf32", "bf16": "bf16"}.get(mode_name, "f32"), "data": "synthetic",
        "config": workload_config(name, w, {
            "kernel": sg.KERNEL_NAMES.get(kid, str(kid)),
            "l2": f"operands {4 * (M * K + K * N + M * N) / 1e6:.0f} MB > L2 129 MB; no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_source,
                     "kernel": (("ffma_tma_kernel, CUDA events around each of its launches in a "
                                 "second pass of the timed steps (the call's transpose and tail sum "
                                 "excluded; per_call_ms and frac_per_call include them)") if kernel_ms else
                                ("transpose_tile_kernel<0> + ffma_tma_kernel + tail sum, timed together "
                                 "as one sgemm() call; traffic is ffma_tma_kernel's alone")
                                if kid == sg.KERNEL_FFMA_TMA else sg.KERNEL_NAMES.get(kid, str(kid))),
                     "kernel_ms": kernel_ms,
                     "per_call_ms": per_launch_ms},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "sgemm_host (C ABI): pinned host A, B, C; copies overlapped with the "
                       "compute in %d row panels" % -(-M // sg.host_panel_rows(M, N, K)),
                "parity": e2e_parity},
        "gpu_launches": args.steps * launches_per_call,
        "clocks": csum,
        "cpu_baseline": cpu,
        "parity": parity,
    }
    if kernel_ms:
        line["roofline"]["frac_per_call"] = flops / (per_launch_ms * 1e-3) / 1e12 / peak
    if csum and csum.get("sm_mhz") and bound == "alu":
        line["roofline"]["frac_at_sampled_clock"] = achieved / acc.ffma_peak_tflops(
            props.multi_processor_count, csum["sm_mhz"])
    if sec is not None:
        line["secondary"] = sec
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sgemm_4092")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds for --impl reference")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--no-kernel-timing", action="store_true",
                    help="time the whole sgemm() call only (no events around the tile kernel)")
    ap.add_argument("--tensor-cores", action="store_true",
                    help="time sgemm_3xtf32 instead of sgemm on the main workload (= --mode 3xtf32)")
    ap.add_argument("--mode", choices=sorted(MODES),
                    help="arithmetic of the main workload: sgemm (fp32), sgemm_3xtf32, sgemm_tf32, "
                         "sgemm_bf16")
    ap.add_argument("--print-source-hash", metavar="KERNEL")
    args = ap.parse_args()
    if args.print_source_hash:
        print(source_hash(args.print_source_hash))
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
