"""Benchmark: C = alpha*A*B + beta*C (FP16 inputs, FP32 accumulation) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 3] [--impl ours|reference]

One step is one call of the library's GEMM (mpgemm_run) on the named
workload, default the 8192^3 square GEMM (inputs larger than L2, so no flush
is needed between steps). Prints one JSON line (rank 0).

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize() on both sides, timed with CUDA events on the
launching stream; the maximum over ranks is taken. Several GPUs run
independent replicas (a GEMM of this size needs no collective), so
`value` = all ranks' FLOPs / the slowest rank's time ("weak" scaling).

Extra keys:
  roofline      the tensor-core kernel against the roof that binds it: the
                tensor peak (2MNK per launch over its event-timed duration,
                against the measured bf16 dense peak; the fp16 kind::f16 rate
                is the same) when the workload's arithmetic intensity is above
                the ridge point, else HBM (algorithmic bytes per launch over
                the same duration, against the measured copy bandwidth);
                roofline_alt holds the other roof;
  peak_theoretical  SMs x FLOP per cycle per SM x maximum SM clock, the
                per-SM factor measured on the device by the library's MMA-rate
                probe (mpgemm_probe_mma_rate);
  protocol      the median of 5 runs x 20 back-to-back launches and the
                coefficient of variation of the 5 runs;
  steady_state  alternating segments of about a second of back-to-back calls
                of ours and of cuBLAS, clocks sampled every 50 ms: TFLOP/s, SM
                clock, cycles per call (time x median SM clock) and power;
  e2e           the same metric through mpgemm_run_host with pinned HOST
                buffers: every step copies A and B in and C out;
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload;
  clocks        nvidia-smi samples taken during the timed region (or, when the
                timed region is shorter than the sampling interval, during the
                steady-state segments of ours, as the window key says).

--impl reference times the CPU oracle (the project's correctness reference)
on the same workload, metric and unit, one bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "TFLOP/s (2MNK/device time) fp16->fp32 GEMM; % of GB300 dense FP16 tensor peak"


# ----------------------------------------------------------------------------- counters

def gemm_flops(M: int, N: int, K: int) -> int:
    """2*M*N*K: one multiply and one add per (i, j, k)."""
    return 2 * M * N * K


def gemm_bytes(M: int, N: int, K: int, beta: float, a_bytes=2, b_bytes=2, c_bytes=4) -> int:
    """Algorithmic HBM bytes: A and B read once, C written once (and read once if beta != 0)."""
    c_traffic = M * N * c_bytes * (2 if beta != 0 else 1)
    return M * K * a_bytes + K * N * b_bytes + c_traffic


def roofline_pair(M: int, N: int, K: int, beta: float, kernel_ms: float, peaks: dict, traffic=None,
                  theoretical=None):
    """(binding roof, the other roof) of one tensor-core launch taking
    kernel_ms. The workload is HBM-bound when its arithmetic intensity
    (2MNK over the algorithmic bytes) is below the ridge point of the
    measured peaks (tensor FLOP/s over HBM bytes/s), tensor-bound otherwise
    ("02_mixed_precision_gemm" README, "Experimental Setup": the roofline
    against the dense tensor peak and the memory bandwidth)."""
    flops = gemm_flops(M, N, K)
    nbytes = gemm_bytes(M, N, K, beta)
    secs = kernel_ms / 1e3
    tensor_achieved = flops / secs / 1e12
    hbm_achieved = nbytes / secs / 1e9
    tensor = {"bound": "tensor", "achieved": round(tensor_achieved, 1), "peak": peaks["tflops"],
              "unit": "TFLOP/s", "frac": round(tensor_achieved / peaks["tflops"], 4), "traffic": traffic,
              "peak_kind": f"bf16 dense burst, {peaks['source']}",
              "frac_of_sustained": (round(tensor_achieved / peaks["tflops_sustained"], 4)
                                    if peaks.get("tflops_sustained") else None),
              "kernel": "gemm_tc_kernel", "algorithmic_flops": flops, "algorithmic_bytes": nbytes}
    if theoretical and theoretical.get("tflops"):
        tensor["peak_theoretical"] = theoretical["tflops"]
        tensor["frac_of_theoretical"] = round(tensor_achieved / theoretical["tflops"], 4)
    hbm = {"bound": "hbm", "achieved": round(hbm_achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": round(hbm_achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
           "peak_kind": f"HBM copy bandwidth, {peaks['source']}",
           "kernel": "gemm_tc_kernel", "algorithmic_bytes": nbytes}
    ridge = peaks["tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flops / nbytes < ridge:
        return hbm, tensor
    return tensor, hbm


def check_world(gpus: int, world: int):
    """--gpus N must match the ranks actually launched: N > 1 runs as N
    torchrun ranks (one replica per GPU), N == 1 as one process. A mismatch
    is an error, so the line never claims GPUs it did not use."""
    if gpus < 1:
        raise SystemExit(f"bench.py: --gpus {gpus} is not a GPU count")
    if gpus != world:
        raise SystemExit(f"bench.py: --gpus {gpus} but {world} rank(s) were launched; for N > 1 run "
                         f"python -m torch.distributed.run --nproc-per-node {gpus} bench.py --gpus {gpus}")


def workload_config(w, world: int) -> dict:
    """The workload as both arms report it (the same keys and values)."""
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "lda": w.lda, "ldb": w.ldb, "ldc": w.ldc,
            "alpha": w.alpha, "beta": w.beta, "inputs": w.dist, "parallelism": f"replicas x{world}"}


def _code_only(text: str) -> str:
    """C++ source without its comments and blank space (string literals in
    these files hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash() -> str:
    """Hash of what fixes the tensor-core kernel's memory traffic: its device
    code (comments and layout aside) and the tile configurations it is
    instantiated with. A stored ncu traffic figure is only reported while
    this hash matches."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixed_precision_dense_gb300", "csrc")
    for name in ("gemm_kernel.cuh", "ptx.cuh"):
        with open(os.path.join(csrc, name)) as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    with open(os.path.join(csrc, "mpgemm.cu")) as f:
        for line in f:
            if line.startswith("using Cfg"):
                h.update(_code_only(line).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"tflops": d["bf16_tflops"], "tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"tflops": 1900.0, "tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def traffic_path(workload_index: int) -> str:
    return os.path.join(ROOT, "profiles", f"gemm_tc_kernel_traffic_w{workload_index}.json")


def stored_traffic(workload_index: int, tile: str):
    """Per-launch DRAM bytes of the tensor-core kernel from a committed ncu
    summary, if it was taken on the current kernel sources and tile shape."""
    path = traffic_path(workload_index)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_hash") != source_hash() or d.get("tile") != tile:
        return None
    return d.get("dram_bytes_per_launch")


def record_traffic(args):
    """Write the per-launch DRAM traffic record of the tensor-core kernel
    from an ncu CSV log holding dram__bytes_read.sum, dram__bytes_write.sum
    and gpu__time_duration.sum of one launch (the workload's own tile shape,
    current sources)."""
    import csv

    import mixed_precision_dense_gb300 as mp
    w = workloads.WORKLOADS[args.workload]
    plan = mp.plan(w.M, w.N, w.K, w.alpha, 256, w.lda, 256, w.ldb, w.beta, 256, w.ldc, num_sms=args.num_sms,
                   tile_m=args.tile_m, tile_n=args.tile_n)
    metrics, kernel = {}, None
    with open(args.record_traffic) as f:
        rows = [r for r in csv.reader(line for line in f if not line.startswith("=="))]
    hdr = rows[0]
    ki, mi, vi = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value")
    for r in rows[1:]:
        if len(r) > vi and "gemm_tc_kernel" in r[ki]:
            kernel = r[ki]
            metrics[r[mi]] = float(r[vi].replace(",", ""))
    rd, wr = metrics["dram__bytes_read.sum"], metrics["dram__bytes_write.sum"]
    rec = {"kernel": kernel, "workload": w.name, "tile": f"{plan['tile_m']}x{plan['tile_n']}",
           "dram_bytes_read_per_launch": int(rd), "dram_bytes_write_per_launch": int(wr),
           "dram_bytes_per_launch": int(rd + wr), "ncu_duration_ns": int(metrics["gpu__time_duration.sum"]),
           "source_hash": source_hash(), "command": args.record_command}
    with open(traffic_path(args.workload), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec))


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_seconds: float, local_flops: float, group=None, device=None):
    """(max seconds over ranks, total flops over ranks)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return local_seconds, local_flops
    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    f = torch.tensor([local_flops], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(f, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(f.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock, power and throttle-reason samples with timestamps,
    every `interval_ms`; summarize() keeps the samples inside a host-time
    window."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int, interval_ms: int = 50):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.samples = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.samples = parse_clock_samples(out)
        return self.samples

    @staticmethod
    def summarize(samples, t0=None, t1=None) -> dict:
        inside = [x for x in samples if (t0 is None or x["t"] >= t0) and (t1 is None or x["t"] <= t1)]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "power_w": None, "power_w_max": None,
                    "samples": 0, "reasons": []}
        reasons = sorted({r for x in inside for r in x["reasons"]})
        return {"sm_mhz": statistics.median(x["sm"] for x in inside),
                "sm_max_mhz": max(x["smax"] for x in inside),
                "power_w": round(statistics.median(x["power"] for x in inside), 1),
                "power_w_max": max(x["power"] for x in inside),
                "samples": len(inside), "reasons": reasons}


def parse_clock_samples(text: str):
    """Rows of the ClockSampler query -> [{t, sm, smax, power, reasons}] (t in
    host epoch seconds; rows that do not parse are skipped)."""
    import datetime
    out = []
    for line in text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            sm, smax, power = float(parts[2]), float(parts[3]), float(parts[4])
        except ValueError:
            continue
        reasons = [n for n, flag in zip(ClockSampler.REASONS, parts[6:10]) if flag.lower().startswith("active")]
        out.append({"t": t, "sm": sm, "smax": smax, "power": power, "reasons": reasons})
    return out


# ----------------------------------------------------------------------------- CPU oracle timing

def cpu_model() -> str:
    """The host CPU as the OS names it (lscpu's model name, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def time_oracle_sample(w, ops, target_seconds: float, max_elements: int, seed: int):
    """Time the oracle on seeded sampled elements of the workload; returns
    (TFLOP/s-equivalent, seconds, elements, threads)."""
    import oracle
    threads = os.cpu_count() or 1
    A, B, C = ops.bits("A"), ops.bits("B"), ops.bits("C")
    n = 256
    while True:
        I, J = workloads.sample_indices(w.M, w.N, n, seed=seed, edges=False)
        t0 = time.perf_counter()
        oracle.elements(w.M, w.N, w.K, w.alpha, A, w.lda, B, w.ldb, w.beta, C, w.ldc, I, J,
                        threads=threads)
        dt = time.perf_counter() - t0
        if dt >= target_seconds or n >= max_elements:
            break
        n = min(max_elements, max(n * 2, int(n * target_seconds / max(dt, 1e-3))))
    return gemm_flops(1, n, w.K) / dt / 1e12, dt, n, threads


# ----------------------------------------------------------------------------- workloads

def select_workload(args):
    """The named workload, or (--shape MxNxK) the same recipe at another size."""
    import dataclasses
    w = workloads.WORKLOADS[args.workload]
    if not args.shape:
        return w, workloads.workload_operands(args.workload)
    M, N, K = (int(x) for x in args.shape.lower().split("x"))
    w = dataclasses.replace(w, name=f"{w.name}_recipe_at_{M}x{N}x{K}", M=M, N=N, K=K,
                            lda=K, ldb=N, ldc=N, full_check=False)
    ops = workloads.make_operands(M, N, K, lda=K, ldb=N, ldc=N, alpha=w.alpha, beta=w.beta,
                                  dist=w.dist, c_dist=w.c_dist, seed=w.seed_base)
    return w, ops


# ----------------------------------------------------------------------------- cuBLAS context

def _cublas_lib():
    import ctypes
    import glob
    cands = []
    try:
        import nvidia.cublas  # noqa: F401  (wheel-installed cuBLAS next to torch)
        import nvidia.cublas as nc
        cands += glob.glob(os.path.join(os.path.dirname(nc.__file__), "lib", "libcublas.so*"))
    except Exception:
        pass
    cands += sorted(glob.glob("/usr/local/cuda/lib64/libcublas.so*"), reverse=True)
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    return None


class CublasContext:
    """cublasGemmEx(FP16 A and B, FP32 C, CUBLAS_COMPUTE_32F, default algorithm)
    on the same buffers as our step. Row-major C = A*B is issued as the
    column-major product C^T = B^T * A^T, so no copies are needed. This is
    context measured by the harness only; the library does not use cuBLAS.
    `call` is None when cuBLAS cannot be loaded or refuses the problem."""
    CALL = ("cublasGemmEx(CUDA_R_16F, CUDA_R_16F, CUDA_R_32F, CUBLAS_COMPUTE_32F, "
            "CUBLAS_GEMM_DEFAULT), harness only")

    def __init__(self, w, A, B, C, stream):
        import ctypes
        self.call = None
        self._lib = _cublas_lib()
        self._h = ctypes.c_void_p()
        if self._lib is None or self._lib.cublasCreate_v2(ctypes.byref(self._h)) != 0:
            self._lib = None
            return
        lib, h = self._lib, self._h
        lib.cublasSetStream_v2(h, ctypes.c_void_p(stream.cuda_stream))
        alpha = ctypes.c_float(w.alpha)
        beta = ctypes.c_float(w.beta)
        CUDA_R_16F, CUDA_R_32F, COMPUTE_32F, GEMM_DEFAULT = 2, 0, 68, -1

        def call():
            return lib.cublasGemmEx(h, 0, 0, w.N, w.M, w.K, ctypes.byref(alpha),
                                    ctypes.c_void_p(B.data_ptr()), CUDA_R_16F, w.ldb,
                                    ctypes.c_void_p(A.data_ptr()), CUDA_R_16F, w.lda,
                                    ctypes.byref(beta), ctypes.c_void_p(C.data_ptr()), CUDA_R_32F,
                                    w.ldc, COMPUTE_32F, GEMM_DEFAULT)

        for _ in range(3):
            if call() != 0:
                return
        self.call = call

    def close(self):
        if self._lib is not None:
            self._lib.cublasDestroy_v2(self._h)
            self._lib = None
            self.call = None


def timed_loop(fn, stream, steps, flush=None):
    """Mean milliseconds per call of fn() over `steps` calls, CUDA events on
    `stream`. With `flush` (a tensor larger than L2), L2 is overwritten before
    every call and only the calls are timed."""
    import torch
    if flush is None:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
    ends[-1].synchronize()
    return sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps


def protocol_runs(fn, stream, flops, flush=None, runs=5, calls=20):
    """The measurement protocol of the "02_mixed_precision_gemm" README
    ("Results", "Reproducing"): the median of `runs` runs of `calls`
    back-to-back launches, with each run's TFLOP/s and the coefficient of
    variation of the runs."""
    ms = [timed_loop(fn, stream, calls, flush) for _ in range(runs)]
    tf = [flops / (m / 1e3) / 1e12 for m in ms]
    return {"runs": runs, "calls_per_run": calls, "tflops_median": round(statistics.median(tf), 2),
            "tflops_runs": [round(x, 1) for x in tf], "ms_median": round(statistics.median(ms), 5),
            "cv": round(statistics.pstdev(ms) / statistics.mean(ms), 5)}


def steady_state(arms: dict, stream, ms_guess: float, flops: float, device_index: int,
                 seconds: float = 1.0, rounds: int = 2):
    """Alternating segments of about `seconds` of back-to-back calls per arm
    (name -> callable), `rounds` times, with clocks, power and throttle
    reasons sampled every 50 ms. Long enough for the power cap to act (the
    driver's short burst is not). Per arm: TFLOP/s and ms per call (median of
    its segments), the median SM clock inside its segments and the cycles per
    call that time x clock gives, the median power and any throttle reason."""
    import torch
    sampler = ClockSampler(device_index, interval_ms=50).start()
    time.sleep(0.3)
    segs = []
    for _ in range(rounds):
        for name, fn in arms.items():
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            n = max(20, int(seconds * 1e3 / max(ms_guess, 1e-3)))
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            t0 = time.time()
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            e1.synchronize()
            t1 = time.time()
            segs.append((name, t0, t1, e0.elapsed_time(e1) / n, n))
    time.sleep(0.1)
    samples = sampler.stop()
    out = {"seconds_per_segment": seconds, "segments_per_arm": rounds, "clock_interval_ms": 50}
    for name in arms:
        mine = [x for x in segs if x[0] == name]
        ms = statistics.median(x[3] for x in mine)
        # skip the first 50 ms of a segment: the clock takes a moment to settle
        inside = [x for seg in mine for x in samples if seg[1] + 0.05 <= x["t"] <= seg[2]]
        clk = ClockSampler.summarize(inside)
        mhz = clk["sm_mhz"]
        out[name] = {"tflops": round(flops / (ms / 1e3) / 1e12, 1), "ms_per_call": round(ms, 5),
                     "calls_per_segment": mine[0][4], "sm_mhz": mhz,
                     "cycles_per_call": round(ms * 1e-3 * mhz * 1e6) if mhz else None,
                     "power_w": clk["power_w"], "clock_samples": clk["samples"], "reasons": clk["reasons"]}
    if "ours" in out and "cublas" in out:
        out["ours_over_cublas"] = round(out["ours"]["tflops"] / out["cublas"]["tflops"], 4)
        if out["ours"]["cycles_per_call"] and out["cublas"]["cycles_per_call"]:
            out["cycles_cublas_over_ours"] = round(out["cublas"]["cycles_per_call"] / out["ours"]["cycles_per_call"], 4)
    out["_samples"] = samples
    out["_segments"] = segs
    return out


def theoretical_peak(device, max_mhz=None):
    """SMs x FLOP per cycle per SM x maximum SM clock, the per-SM factor
    measured by the library's MMA-rate probe (one CTA per SM issuing 16384
    back-to-back 128 x 256 x 16 MMAs) and the maximum clock as nvidia-smi
    reports it (else MEASURED_PEAKS.json's)."""
    import torch

    import mixed_precision_dense_gb300 as mp
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mmas = 1 << 14
    out = torch.zeros(2 * sms, dtype=torch.int64, device=device)
    stream = torch.cuda.current_stream(device)
    mp.probe_mma_rate(sms, mmas, out.data_ptr(), stream.cuda_stream)
    stream.synchronize()
    res = out.cpu().tolist()
    cycles = [res[2 * i] for i in range(sms) if res[2 * i + 1] == 1]
    if not cycles:
        return None
    per_sm = statistics.median(mp.PROBE_FLOP_PER_MMA * mmas / c for c in cycles)
    if max_mhz is None:
        try:
            q = subprocess.run(["nvidia-smi", f"--id={device.index or 0}", "--query-gpu=clocks.max.sm",
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
            max_mhz = float(q.stdout.strip().splitlines()[0])
        except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
            path = os.path.join(ROOT, "MEASURED_PEAKS.json")
            max_mhz = json.load(open(path)).get("sm_max_mhz") if os.path.exists(path) else None
    if not max_mhz:
        return None
    return {"tflops": round(sms * per_sm * max_mhz * 1e6 / 1e12, 1), "sms": sms,
            "flop_per_clk_per_sm": round(per_sm, 1), "sm_max_mhz": max_mhz,
            "how": "mpgemm_probe_mma_rate: one CTA per SM, 16384 back-to-back kind::f16 "
                   "128 x 256 x 16 MMAs, %clock64 cycles; x SMs x max SM clock"}


# ----------------------------------------------------------------------------- our arm

def run_ours(args):
    import numpy as np
    import torch

    import mixed_precision_dense_gb300 as mp

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    mp.build()
    w, ops = select_workload(args)
    stream = torch.cuda.current_stream(device)
    A = ops.A.to(device)
    B = ops.B.to(device)
    C0 = ops.C.to(device)
    C = C0.clone()
    handle = mp.Handle()
    handle.set_option(mp.Option.TILE_M, args.tile_m)
    handle.set_option(mp.Option.TILE_N, args.tile_n)
    handle.set_option(mp.Option.SPLIT_K, args.split_k)

    def step():
        handle.run(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.lda, B.data_ptr(), w.ldb, w.beta,
                   C.data_ptr(), w.ldc, stream.cuda_stream)

    plan = mp.plan(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.lda, B.data_ptr(), w.ldb, w.beta,
                   C.data_ptr(), w.ldc, num_sms=torch.cuda.get_device_properties(device).multi_processor_count,
                   tile_m=args.tile_m, tile_n=args.tile_n)
    launches_per_step = 1 + plan["stage_a"] + plan["stage_b"]
    if (args.split_k > 1 or (args.split_k == 0 and plan["k_splits"] > 1)) and w.beta != 1.0:
        launches_per_step += 1      # the pass that applies beta before the slices add into C

    # correctness first, on a NaN-poisoned (beta == 0) or restored (beta != 0) C
    if w.beta == 0:
        C.fill_(float("nan"))
    step()
    st, info = handle.sync_status(stream.cuda_stream)
    if st != mp.Status.OK:
        raise RuntimeError(f"device reported {st.name} {info}")
    check = None
    if rank == 0 and not args.no_check:
        import oracle
        I, J = workloads.sample_indices(w.M, w.N, 2048, seed=w.seed_base + 3)
        ref, S = oracle.elements(w.M, w.N, w.K, w.alpha, ops.bits("A"), w.lda, ops.bits("B"), w.ldb,
                                 w.beta, ops.bits("C"), w.ldc, I, J)
        got = C.cpu().numpy()[I, J].astype(np.float64)
        ratio = np.abs(got - ref) / oracle.tolerance(S)
        if not np.all(ratio <= 1.0):
            raise AssertionError(f"bench correctness check failed: max err/tol {np.nanmax(ratio)}")
        check = float(np.max(ratio))
    C.copy_(C0)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    small = gemm_bytes(w.M, w.N, w.K, w.beta) < L2_BYTES
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=device) if small else None
    sampler = ClockSampler(local, interval_ms=20).start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(device)
    t_begin = time.time()
    local_ms = timed_loop(step, stream, args.steps, flush)
    torch.cuda.synchronize(device)
    t_end = time.time()
    barrier()
    timed_clocks = ClockSampler.summarize(sampler.stop(), t_begin, t_end)
    st, info = handle.sync_status(stream.cuda_stream)
    if st != mp.Status.OK:
        raise RuntimeError(f"device reported {st.name} {info}")
    local_s = local_ms * args.steps / 1e3
    flops = gemm_flops(w.M, w.N, w.K)
    max_s, flops_all = aggregate(local_s, flops * args.steps, device=device)
    value = flops_all / max_s / 1e12
    ms_per_step = max_s * 1e3 / args.steps

    # the dominant kernel alone: event-timed tensor-core launches (one per step
    # when no operand needs staging; otherwise the same kernel, same tile
    # and same reading of A, timed on operands staged beforehand)
    # (a split call's pass that applies beta stays in: it belongs to that call)
    kernel_ms = ms_per_step
    if plan["stage_a"] or plan["stage_b"]:
        kernel_ms = time_tc_kernel_only(w, A, B, C, stream, args.steps, plan, flush, args.split_k)
    peaks = measured_peaks()
    theory = None if args.no_probe else theoretical_peak(device)
    traffic = None if args.shape else stored_traffic(args.workload, f"{plan['tile_m']}x{plan['tile_n']}")
    roofline, roofline_alt = roofline_pair(w.M, w.N, w.K, w.beta, kernel_ms, peaks, traffic, theory)

    protocol = protocol_runs(step, stream, flops, flush)
    cublas, steady = None, None
    cub = None if args.no_cublas else CublasContext(w, A, B, C, stream)
    if cub is not None and cub.call is not None:
        cub_ms = timed_loop(cub.call, stream, args.steps, flush)
        cublas = {"value": round(flops / (cub_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                  "ms_per_step": round(cub_ms, 5), "call": CublasContext.CALL,
                  "ours_over_cublas": round(value / world / (flops / (cub_ms / 1e3) / 1e12), 4),
                  "protocol": protocol_runs(cub.call, stream, flops, flush)}
    if args.steady_seconds > 0:
        arms = {"ours": step}
        if cub is not None and cub.call is not None:
            arms["cublas"] = cub.call
        steady = steady_state(arms, stream, local_ms, flops, local, seconds=args.steady_seconds)
        steady["l2"] = "back to back on the same operands, no L2 flush"
    if cub is not None:
        cub.close()
    if timed_clocks["samples"] > 0 and (steady is None or t_end - t_begin >= 0.5):
        clocks = dict(timed_clocks, window="the timed region")
    elif steady is not None:
        segs = [x for x in steady["_segments"] if x[0] == "ours"]
        inside = [x for seg in segs for x in steady["_samples"] if seg[1] + 0.05 <= x["t"] <= seg[2]]
        clocks = dict(ClockSampler.summarize(inside),
                      window=(f"the steady-state segments of ours (the timed region, {args.steps} calls in "
                              f"{local_s * 1e3:.1f} ms, is too short for nvidia-smi's samples, which lag "
                              "by tens of ms)"),
                      timed_region=timed_clocks)
    else:
        clocks = dict(timed_clocks, window="the timed region")
    if steady is not None:
        steady.pop("_samples")
        steady.pop("_segments")

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(handle, w, ops, stream, device, args)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, n, threads = time_oracle_sample(w, ops, args.cpu_seconds, 1 << 20, w.seed_base + 5)
        cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{n} seeded elements of C (K = {w.K} MACs each) in {dt:.2f} s"}

    handle.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16 inputs, f32 accumulate", "data": "synthetic (seeded)",
            "config": workload_config(w, world),
            "l2": (f"L2 flushed between steps (a {2 * L2_BYTES // 2**20} MiB write before each "
                   "step, outside the timed calls)" if small else
                   f"inputs larger than L2 ({gemm_bytes(w.M, w.N, w.K, w.beta) / 2**20:.0f} MiB "
                   f"> {L2_BYTES // 2**20} MiB): no flush"),
            "launch": {"tile": f"{plan['tile_m']}x{plan['tile_n']}x{plan['tile_k']}", "grid": plan["grid"],
                       "k_splits": plan["k_splits"], "a_row_classes": plan["a_classes"],
                       "staged": {"A": plan["stage_a"], "B": plan["stage_b"]}},
            "pct_of_peak": round(100 * value / world / peaks["tflops"], 2),
            "pct_of_theoretical_peak": round(100 * value / world / theory["tflops"], 2) if theory else None,
            "peak_theoretical": theory,
            "roofline": roofline, "roofline_alt": roofline_alt, "protocol": protocol,
            "steady_state": steady, "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks,
            "context_cublas": cublas,
            "gpu_launches": launches_per_step * args.steps, "check_max_err_over_tol": check,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def time_tc_kernel_only(w, A, B, C, stream, steps, plan, flush=None, split_k=0):
    """Event-time the tensor-core launch alone: the operands that the call
    stages (plan["stage_a"], plan["stage_b"]) are copied to aligned buffers
    first, the others are used as they are (an unaligned A that the kernel
    reads in row classes stays so), and the tile shape is pinned to the
    call's own, so the launch timed is the step's kernel."""
    import torch

    import mixed_precision_dense_gb300 as mp
    M, N, K = w.M, w.N, w.K
    A2, lda, B2, ldb = A, w.lda, B, w.ldb
    if plan["stage_a"]:
        lda = (K + 7) // 8 * 8
        A2 = torch.zeros((M, lda), dtype=torch.float16, device=A.device)
        A2[:, :K] = A[:, :K]
    if plan["stage_b"]:
        ldb = (N + 7) // 8 * 8
        B2 = torch.zeros((K, ldb), dtype=torch.float16, device=B.device)
        B2[:, :N] = B[:, :N]
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, plan["tile_m"])
        h.set_option(mp.Option.TILE_N, plan["tile_n"])
        h.set_option(mp.Option.SPLIT_K, split_k)
        run = lambda: h.run(M, N, K, w.alpha, A2.data_ptr(), lda, B2.data_ptr(), ldb, w.beta, C.data_ptr(),
                            w.ldc, stream.cuda_stream)
        p2 = mp.plan(M, N, K, w.alpha, A2.data_ptr(), lda, B2.data_ptr(), ldb, w.beta, C.data_ptr(), w.ldc,
                     num_sms=torch.cuda.get_device_properties(A.device).multi_processor_count,
                     tile_m=plan["tile_m"], tile_n=plan["tile_n"])
        assert p2["stage_a"] == 0 and p2["stage_b"] == 0 and p2["a_classes"] == plan["a_classes"], p2
        for _ in range(3):
            run()
        ms = timed_loop(run, stream, steps, flush)
        st, info = h.sync_status(stream.cuda_stream)
        if st != mp.Status.OK:
            raise RuntimeError(f"device reported {st.name} {info}")
        return ms


# handles (and streams) the end-to-end leg rotates through
E2E_SLOTS = 3


def run_e2e(handle, w, ops, stream, device, args):
    """End to end through mpgemm_run_host on pinned host buffers: every step
    copies A and B (and C when beta != 0) to the device, runs the GEMM and
    copies C back. Three handles on three streams rotate, so one step's
    copy in, another's GEMM and a third's copy out can run at once (with two
    slots a step's copy in has to wait for the copy out two steps back); a
    step's slot is reused only after its stream has finished, i.e. after its
    result is in host memory."""
    import torch

    import mixed_precision_dense_gb300 as mp
    slots = E2E_SLOTS
    A_h = ops.A.pin_memory()
    B_h = ops.B.pin_memory()
    C_h = [ops.C.clone().pin_memory() for _ in range(slots)]
    handles = [handle] + [mp.Handle() for _ in range(slots - 1)]
    for h in handles[1:]:
        h.set_option(mp.Option.TILE_M, args.tile_m)
        h.set_option(mp.Option.TILE_N, args.tile_n)
        h.set_option(mp.Option.SPLIT_K, args.split_k)
    streams = [stream] + [torch.cuda.Stream(device) for _ in range(slots - 1)]
    steps = max(1, min(args.steps, args.e2e_steps))

    def enqueue(i):
        k = i % slots
        handles[k].run_host(w.M, w.N, w.K, w.alpha, A_h.data_ptr(), w.lda, B_h.data_ptr(), w.ldb,
                            w.beta, C_h[k].data_ptr(), w.ldc, streams[k].cuda_stream)

    for i in range(2 * slots):
        enqueue(i)
    torch.cuda.synchronize(device)
    barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        if i >= slots:
            streams[i % slots].synchronize()   # step i-slots's result is on the host; its slot is free
        enqueue(i)
    for st in streams:
        st.synchronize()
    dt = time.perf_counter() - t0
    for k in range(slots):
        st_, info = handles[k].sync_status(streams[k].cuda_stream)
        if st_ != mp.Status.OK:
            raise RuntimeError(f"device reported {st_.name} {info}")
    for h in handles[1:]:
        h.close()
    max_s, flops_all = aggregate(dt, gemm_flops(w.M, w.N, w.K) * steps, device=device)
    h2d = (w.M * w.K * 2 + w.K * w.N * 2) + (w.M * w.N * 4 if w.beta != 0 else 0)
    return {"value": round(flops_all / max_s / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": w.M * w.N * 4, "steps": steps,
            "ms_per_step": round(max_s * 1e3 / steps, 4),
            "api": f"mpgemm_run_host on pinned host buffers, {slots} handles on {slots} streams "
                   "rotating, host wall clock"}


# ----------------------------------------------------------------------------- the capstone gate

GATE_CASES = [  # "Day 80, Capstone 4: a tensor-core GEMM", "Independent gate"
    ("unit", 16, 16, 16, "int", "bitwise"),
    ("onefrag", 16, 8, 16, "int", "bitwise"),
    ("small", 128, 128, 128, "uniform", "tolerance"),
    ("odd", 611, 613, 617, "uniform", "tolerance"),
    ("skinny", 4096, 16, 4096, "uniform", "tolerance"),
    ("square", 1024, 1024, 1024, "normal", "tolerance"),
    ("adversarial", 256, 256, 256, "edge", "tolerance"),
    ("perf", 4096, 4096, 4096, "uniform", "sampled"),
]


def run_acc16_study(args):
    """FP16 accumulators against FP32 ("Day 72: Tensor cores with WMMA",
    Exercise: AccT = __half; "Day 80, Capstone 4", "Common failures"). For
    uniform[-1, 1) inputs at growing K, the FP16-accumulated C is compared
    with the FP32-accumulated C of the same library (parity-tested; its own
    error is at most about K * 2^-24 * S, negligible here) in units of
    S = sum_k |A_ik B_kj|, and against the parity tolerance 1e-3 * S + 1e-5.
    Then the pages' integer sizes, the 4096-term overflow and a sum growing
    by 15 per K = 16 step past 2048. Prints a markdown report."""
    import numpy as np
    import torch

    import mixed_precision_dense_gb300 as mp
    mp.build()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)

    def gemm(A, B, acc):
        M, K = A.shape
        N = B.shape[1]
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        with mp.Handle() as h:
            h.set_option(mp.Option.ACCUMULATOR, acc)
            h.run(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N, stream.cuda_stream)
            stream.synchronize()
            st, info = h.sync_status(stream.cuda_stream)
            if st != mp.Status.OK:
                raise RuntimeError(f"device reported {st.name} {info}")
        return C

    print("| inputs | K | max err / S (FP16 acc) | median err / S | elements over 1e-3 S + 1e-5 | max err / S (FP32 acc, vs FP64 of 2048 samples) |")
    print("|---|---|---|---|---|---|")
    M = N = 1024
    for lo, K in [(lo, K) for lo in (-1.0, 0.0) for K in (256, 1024, 2048, 4096, 8192, 16384)]:
        g = torch.Generator().manual_seed(900 + K + int(lo))
        A = (lo + torch.rand(M, K, generator=g) * (1 - lo)).half().to(dev)
        B = (lo + torch.rand(K, N, generator=g) * (1 - lo)).half().to(dev)
        c32, c16 = gemm(A, B, 32), gemm(A, B, 16)
        S = torch.matmul(A.float().abs(), B.float().abs())
        r = ((c16 - c32).abs() / S).flatten()
        over = int(((c16 - c32).abs() > 1e-3 * S + 1e-5).sum())
        # FP32 path against an FP64 product on a sample (host float64 arithmetic)
        idx = torch.randint(0, M * N, (2048,), generator=g)
        i, j = (idx // N).tolist(), (idx % N).tolist()
        a64, b64 = A.double().cpu(), B.double().cpu()
        exact = (a64[i] * b64[:, j].t()).sum(1)
        e32 = float(((c32.cpu().double().flatten()[idx] - exact).abs() / S.cpu().double().flatten()[idx]).max())
        print(f"| uniform[{lo:g}, 1) | {K} | {float(r.max()):.2e} | {float(r.median()):.2e} | {over} of {M * N} | {e32:.1e} |")

    print()
    for size in (256, 1024, 2048):
        g = torch.Generator().manual_seed(700 + size)
        A = torch.randint(-3, 4, (size, size), generator=g).half().to(dev)
        B = torch.randint(-2, 3, (size, size), generator=g).half().to(dev)
        same = bool(torch.equal(gemm(A, B, 16), gemm(A, B, 32)))
        print(f"- integer inputs in [-3, 3] x [-2, 2] at {size}^3: FP16-accumulated C "
              f"{'equals' if same else 'differs from'} the exact (FP32-accumulated) C")
    A = torch.full((256, 4096), 4.0, device=dev).half()
    B = torch.full((4096, 256), 4.0, device=dev).half()
    c16, c32 = gemm(A, B, 16), gemm(A, B, 32)
    print(f"- 4096 products of 4 x 4: FP32 gives {float(c32[0, 0]):.0f} everywhere: "
          f"{bool(torch.all(c32 == 65536.0))}; FP16 gives +inf everywhere: {bool(torch.all(torch.isinf(c16)))}")
    steps = 512
    A = torch.ones(128, 16 * steps, device=dev).half()
    B = torch.ones(16 * steps, 128, device=dev)
    B[15::16, :] = 0.0
    c16 = gemm(A, B.half(), 16)
    d = np.float16(0)
    for _ in range(steps):
        d = np.float16(d + np.float16(15))
    print(f"- a sum growing by 15 per K = 16 step, {steps} steps (exact {15 * steps}): FP16 accumulators give "
          f"{float(c16[0, 0]):.0f} (all elements equal: {bool(torch.all(c16 == c16[0, 0]))}); adding 15 and "
          f"rounding to FP16 once per step gives {float(d):.0f}")


def run_gate(args):
    """The gate's eight cases through mpgemm_solve (A row-major, B column-major,
    C row-major): every case checked against the CPU oracle (bit for bit for
    the exact small integers), then timed as the median of 5 runs x 20 calls
    (the protocol of the "02_mixed_precision_gemm" README), with cuBLAS GemmEx
    (FP16 in, FP32 out, COMPUTE_32F) on the same buffers and the coefficient of
    variation of the perf case's runs. Prints a markdown report."""
    import ctypes

    import numpy as np
    import torch

    import mixed_precision_dense_gb300 as mp
    import oracle
    mp.build()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    lib = _cublas_lib()
    cub = ctypes.c_void_p()
    if lib is not None and lib.cublasCreate_v2(ctypes.byref(cub)) == 0:
        lib.cublasSetStream_v2(cub, ctypes.c_void_p(stream.cuda_stream))
    else:
        lib = None
    rows = []
    for name, m, n, k, inputs, check in GATE_CASES:
        if inputs == "int":
            ops = workloads.make_operands(m, n, k, dist="int3", dist_b="int2", seed=500 + m + n + k,
                                          b_col_major=True)
        else:
            ops = workloads.make_operands(m, n, k, dist=inputs, seed=500 + m + n + k, b_col_major=True)
        A = ops.A.to(dev)
        B = ops.B.to(dev)
        C = torch.full((m, n), float("nan"), dtype=torch.float32, device=dev)

        def ours():
            mp.solve(A.data_ptr(), B.data_ptr(), C.data_ptr(), m, n, k, stream.cuda_stream)

        ours()
        stream.synchronize()
        got = C.cpu().double().numpy()
        A_bits, B_bits = ops.bits("A"), ops.bits("B")
        if check == "sampled":
            I, J = workloads.sample_indices(m, n, 20000, seed=501)
            ref, S = oracle.elements(m, n, k, 1.0, A_bits, k, B_bits, k, 0.0, None, n, I, J,
                                     b_col_major=True)
            err = float(np.max(np.abs(got[I, J] - ref) / oracle.tolerance(S)))
            verdict = f"max err/tol {err:.2e} on {I.size} elements" + (" PASS" if err <= 1 else " FAIL")
        else:
            ref, S = oracle.gemm(m, n, k, 1.0, A_bits, k, B_bits, k, 0.0, b_col_major=True)
            if check == "bitwise":
                ok = bool(np.array_equal(got, ref))
                verdict = "bit for bit " + ("PASS" if ok else "FAIL")
            else:
                err = float(np.max(np.abs(got - ref) / oracle.tolerance(S)))
                verdict = f"max err/tol {err:.2e}" + (" PASS" if err <= 1 else " FAIL")
        runs = []
        for _ in range(3):
            ours()
        for _ in range(5):
            runs.append(timed_loop(ours, stream, 20))
        ours_ms = statistics.median(runs)
        cv = statistics.pstdev(runs) / statistics.mean(runs)
        cub_ms = None
        if lib is not None:
            alpha, beta = ctypes.c_float(1.0), ctypes.c_float(0.0)

            def theirs():
                lib.cublasGemmEx(cub, 1, 0, n, m, k, ctypes.byref(alpha), ctypes.c_void_p(B.data_ptr()), 2, k,
                                 ctypes.c_void_p(A.data_ptr()), 2, k, ctypes.byref(beta),
                                 ctypes.c_void_p(C.data_ptr()), 0, n, 68, -1)

            for _ in range(3):
                theirs()
            cub_ms = statistics.median(timed_loop(theirs, stream, 20) for _ in range(5))
        rows.append((name, m, n, k, check, verdict, ours_ms, cub_ms, cv))
    if lib is not None:
        lib.cublasDestroy_v2(cub)
    print("| case | m, n, k | check | result | mpgemm_solve (us) | TFLOP/s | cuBLAS GemmEx (us) | % of cuBLAS | CV of 5 runs |")
    print("|---|---|---|---|---|---|---|---|---|")
    for name, m, n, k, check, verdict, ours_ms, cub_ms, cv in rows:
        tf = gemm_flops(m, n, k) / (ours_ms / 1e3) / 1e12
        pct = f"{100 * cub_ms / ours_ms:.1f} %" if cub_ms else "n/a"
        cubs = f"{cub_ms * 1e3:.2f}" if cub_ms else "n/a"
        print(f"| {name} | {m}, {n}, {k} | {check} | {verdict} | {ours_ms * 1e3:.2f} | {tf:.1f} | {cubs} | {pct} | {100 * cv:.2f} % |")
    print(f"\nGPU: {torch.cuda.get_device_name(dev)}; times are medians of 5 runs x 20 back-to-back calls; "
          "tolerance |err| <= 1e-3 * sum_k|A_ik B_kj| + 1e-5.")


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w, ops = select_workload(args)
    import oracle
    threads = os.cpu_count() or 1
    # one bounded sample per step, sized so warm-up + steps stay within a few minutes
    budget_s = 120.0
    per_step = max(1, min(512, int(budget_s / max(1, args.steps + args.warmup) * 2e9 / (2 * w.K))))
    A, B, C = ops.bits("A"), ops.bits("B"), ops.bits("C")

    def step(i):
        I, J = workloads.sample_indices(w.M, w.N, per_step, seed=w.seed_base + 100 + i, edges=False)
        oracle.elements(w.M, w.N, w.K, w.alpha, A, w.lda, B, w.ldb, w.beta, C, w.ldc, I, J,
                        threads=threads)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = gemm_flops(1, per_step, w.K) * args.steps / dt / 1e12
    sample = f"{per_step} seeded elements of C per step (K = {w.K} MACs each)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle: FP16 decoded, double sums)",
        "data": "synthetic (seeded)",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=3, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--shape", default="", help="MxNxK: the workload's recipe at another size")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--steady-seconds", type=float, default=1.0,
                    help="length of each steady-state segment (two per arm); 0 = none")
    ap.add_argument("--no-probe", action="store_true", help="skip the MMA-rate probe (theoretical peak)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-check", action="store_true")
    ap.add_argument("--no-cublas", action="store_true")
    ap.add_argument("--record-traffic", default="",
                    help="write the workload's stored ncu DRAM-traffic record from this ncu CSV log and exit")
    ap.add_argument("--record-command", default="", help="the ncu command that produced --record-traffic's log")
    ap.add_argument("--num-sms", type=int, default=152, help="SM count assumed by --record-traffic's plan")
    ap.add_argument("--tile-m", type=int, default=0, choices=[0, 128, 256],
                    help="force the tile height (0 = the library's choice)")
    ap.add_argument("--tile-n", type=int, default=0, choices=[0, 128, 256, 288, 320, 384, 512],
                    help="force the tile width (0 = the library's choice)")
    ap.add_argument("--split-k", type=int, default=0,
                    help="slices of K per tile (0 = the library's choice, 1 = never split)")
    ap.add_argument("--acc16-study", action="store_true",
                    help="compare FP16 with FP32 accumulation and print a report instead")
    ap.add_argument("--gate", action="store_true",
                    help="run the capstone gate's eight cases and print a report instead")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # at least three warm-up steps, whatever was asked
    if not (args.record_traffic or args.acc16_study or args.gate):
        check_world(args.gpus, dist_env()[0])
    if args.record_traffic:
        record_traffic(args)
    elif args.acc16_study:
        run_acc16_study(args)
    elif args.gate:
        run_gate(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
