"""SGEMM throughput benchmark (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one C = alpha*A*B + beta*C call on the workload (default: the
M = N = K = 4096 cube, uniform[-1, 1] inputs from seed 1, alpha = 0.5,
beta = 3). Inputs are resident on the device before timing; A + B + C
(201 MB at 4096) exceed the 129 MB L2, so no flush is needed between steps.
`value` is GFLOP/s (2*M*N*K per step) over exactly K timed steps bracketed by
a barrier and a device synchronisation, max over ranks; N > 1 runs
independent replicas (the path has no exchange step). `e2e` times the same
work from pinned host buffers: H2D of A, B, C, the call, D2H of C.
`--impl reference` times the CPU oracle (FP64 triple loop) on a bounded row
sample of the same workload; it runs on rank 0 only.

Besides the contract's keys the line carries the per-step statistics of the K
event-timed steps (mean, median, min, max, spread), the SM clock and clock-event
reasons sampled through NVML inside the timed window, and -- from the CPU
baseline leg, which computes the oracle's rows anyway -- `verified`: one call
of each timed path on a fresh C before any timing, checked against the oracle
on those rows and on sampled elements at the FP32 tolerance.
"""
from __future__ import annotations

import argparse
import contextlib
import datetime as _dt
import functools
import glob
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SGEMM GFLOP/s at M=N=K=4096 FP32 and % of GB300 FP32 FFMA peak (1 GPU)"
UNIT = "GFLOP/s"
FFMA_FLOP_PER_CLK_PER_SM = 256  # 128 FP32 lanes x 2 FLOP per fused multiply-add
L2_BYTES = 129 * 1024 * 1024


# ---- accounting (checked against the pages' printed numbers in tests) -------------
def gemm_flops(M, N, K):
    return 2 * M * N * K


def gflops(M, N, K, seconds):
    return gemm_flops(M, N, K) / seconds / 1e9


def gmem_accesses_per_result(K, BM, BN):
    """Global loads per output element for a BM x BN tile: K*(1/BM + 1/BN)."""
    return K * (1.0 / BM + 1.0 / BN)


def smem_loads_per_result(K, TM, TN):
    """Shared loads per output element for a TM x TN thread tile."""
    return K * (1.0 / TM + 1.0 / TN)


def min_bytes(M, N, K, beta):
    """Algorithmic bytes: read A and B once, write C (and read it if beta != 0)."""
    return 4 * (M * K + K * N + M * N * (2 if beta != 0 else 1))


def ffma_peak_tflops(sms, mhz):
    return sms * mhz * 1e6 * FFMA_FLOP_PER_CLK_PER_SM / 1e12


# Nominal dense tensor rates of GB300 (TF32 1.1 PF/s, BF16 2.25 PF/s): the
# TF32 peak is the measured BF16 cuBLAS peak times their ratio. The 3xTF32 path
# issues three TF32 products per FP32 product, so its useful-FLOP roof is a third.
TF32_OVER_BF16 = 1.1 / 2.25


def tf32x3_peak_tflops(peaks):
    """The 3xTF32 roof estimated from the measured BF16 peak (TF32 runs at
    half the BF16 rate, nominally), three TF32 products per FP32 product."""
    bf16 = peaks.get("bf16_tflops")
    return (float(bf16) * TF32_OVER_BF16 / 3.0) if bf16 else None


def tf32x3_roof(binding, peaks, pair=False):
    """(roof TFLOP/s, basis, measured TF32 TFLOP/s or None): the measured
    tcgen05 kind::tf32 throughput of this device / 3 (the library's probe
    kernels: cta_group::2 MMAs of CTA pairs when `pair`, the form the timed
    call ran, else one CTA per SM), else the BF16-derived estimate."""
    probe = binding.sgemm_diag_tf32_pair_mma_rate if pair else binding.sgemm_diag_tf32_mma_rate
    st, tf32 = probe(20000)
    if st == 0 and tf32 > 0:
        form = ("two-SM pairs, cta_group::2 M 256" if pair else "one CTA per SM, M 128")
        return (tf32 / 3.0, f"measured tcgen05.mma kind::tf32 throughput (probe kernel, {form}, "
                            "burst) / 3 TF32 products per FP32 product", tf32)
    return (tf32x3_peak_tflops(peaks), "measured bf16 peak x 1.1/2.25 (TF32/BF16 nominal) / 3 "
                                       "TF32 products per FP32 product", None)


# The sources that define the FFMA kernel the bench times and how it is
# configured (the other entry points and the C-ABI dispatch are left out).
FFMA_KERNEL_SOURCES = ("ffma_sgemm.cuh", "ptx.cuh", "schedule.hpp", "tile_config.hpp",
                       "configs.hpp", "configs.inc", "launch.cuh", "dispatch.hpp", "tuned_table.inc")


def kernel_source_hash():
    """Hash of the FFMA kernel's sources: a stored ncu traffic figure is used
    only while this is unchanged."""
    h = hashlib.sha256()
    files = set()
    for pat in FFMA_KERNEL_SOURCES:
        files.update(glob.glob(os.path.join(ROOT, "dense_fp32_gemm_gb300", "csrc", pat)))
    for f in sorted(files):
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")


def profiled_traffic(workload, tile_config, path=TRAFFIC_PATH):
    """DRAM bytes per launch of the FFMA kernel on this workload, from the
    committed ncu figures (profiles/traffic.json: one entry per workload with
    the kernel-source hash and tile configuration it was captured on), or None
    if there is none, the kernel sources changed since, or it was taken on
    another tile configuration."""
    try:
        table = json.load(open(path))
    except (OSError, ValueError):
        return None
    e = table.get("ffma_sgemm", {}).get(workload)
    if not isinstance(e, dict):
        return None
    if e.get("kernel_source_sha") != kernel_source_hash():
        return None
    if not e.get("tile_config") or not tile_config.startswith(e["tile_config"]):
        return None
    try:
        return float(e["dram_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


def step_stats(ms):
    """Mean, median, min, max and spread (max - min over the median, %) of
    per-step device times in milliseconds."""
    v = sorted(float(x) for x in ms)
    if not v:
        return None
    n = len(v)
    med = v[n // 2] if n % 2 else 0.5 * (v[n // 2 - 1] + v[n // 2])
    return {"mean": round(sum(v) / n, 5), "median": round(med, 5), "min": round(v[0], 5),
            "max": round(v[-1], 5), "spread_pct": round(100.0 * (v[-1] - v[0]) / med, 2) if med else None,
            "n": n}


# ---- NVTX ranges: name the bench's phases in profiler timelines ------------------------
@contextlib.contextmanager
def nvtx_range(name):
    import torch
    torch.cuda.nvtx.range_push(name)
    try:
        yield
    finally:
        torch.cuda.nvtx.range_pop()


# ---- clocks -------------------------------------------------------------------------
# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*) that hold the
# SM clock below what was asked for.
NVML_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
NVML_CLOCK_SM = 1


def summarize_clock_samples(samples, t0, t1, max_mhz, source, period_ms=None):
    """samples: (wall time, SM MHz, reason bits or None). Only the samples
    taken inside [t0, t1] count; with none inside, the clock is unknown."""
    inside = [x for x in samples if t0 <= x[0] <= t1]
    out = {"sm_mhz": None, "sm_max_mhz": max_mhz, "samples": len(inside), "reasons": [],
           "source": source}
    if period_ms is not None:
        out["period_ms"] = period_ms
    if not inside:
        out["reasons"] = ["no clock sample inside the timed window"]
        return out
    mhz = sorted(x[1] for x in inside)
    n = len(mhz)
    out["sm_mhz"] = mhz[n // 2] if n % 2 else 0.5 * (mhz[n // 2 - 1] + mhz[n // 2])
    out["sm_mhz_min"] = mhz[0]
    out["reasons"] = sorted({name for x in inside if x[2] is not None
                             for bit, name in NVML_REASON_BITS.items() if x[2] & bit})
    return out


class NvmlClockSampler:
    """SM clock and clock-event reasons of one GPU, read through NVML by a
    background thread every `period_s` seconds. The queries only read: no
    clock, limit or mode is set. `lib` replaces libnvidia-ml (tests)."""

    def __init__(self, pci_bus_id=None, index=0, period_s=0.002, lib=None):
        import ctypes
        import threading
        self.samples, self.err, self.period_s = [], None, period_s
        self._stop = threading.Event()
        self._thread = None
        self.lib, self.max_mhz = None, None
        try:
            nv = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            if pci_bus_id:
                rc = nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h))
            else:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(index)), ctypes.byref(h))
            if rc != 0:
                raise OSError(f"no NVML device handle (status {rc})")
            self._reasons = (getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None)
                             or nv.nvmlDeviceGetCurrentClocksThrottleReasons)
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.lib, self.h = nv, h
        except (OSError, AttributeError) as e:
            self.err = str(e)

    def poll(self):
        """One sample: (wall time, SM MHz, reason bits or None), or None."""
        import ctypes
        clk, bits = ctypes.c_uint(), ctypes.c_ulonglong()
        t = time.time()
        if self.lib.nvmlDeviceGetClockInfo(self.h, NVML_CLOCK_SM, ctypes.byref(clk)) != 0:
            return None
        r = int(bits.value) if self._reasons(self.h, ctypes.byref(bits)) == 0 else None
        return (t, float(clk.value), r)

    def _run(self):
        while not self._stop.is_set():
            x = self.poll()
            if x is not None:
                self.samples.append(x)
            self._stop.wait(self.period_s)

    def start(self):
        import threading
        if self.lib is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)

    def summary(self, t0, t1):
        if self.lib is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                    "reasons": [f"NVML unavailable: {self.err}"], "source": "nvml"}
        return summarize_clock_samples(self.samples, t0, t1, self.max_mhz, "nvml",
                                       period_ms=round(self.period_s * 1e3, 3))


def nvml_bus_id(props):
    """NVML's PCI bus id ("domain:bus:device.0") of a torch device, or None."""
    try:
        return f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    except AttributeError:
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while it runs (used
    when NVML cannot be loaded)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        self.path = os.path.join("/tmp", f"sgemm_clocks_{os.getpid()}.csv")
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                    "reasons": ["no clock sample inside the timed window"]}
        mhz = sorted(r[1] for r in inside)
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[4]) if v == "Active"})
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[2] for r in inside),
                "samples": len(inside), "reasons": reasons}


# ---- distributed helpers (replicas only) ------------------------------------------
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(flops_per_step_per_rank, steps, seconds_max, world):
    """Whole-job throughput: work of all ranks over the slowest rank's time."""
    return flops_per_step_per_rank * steps * world / seconds_max / 1e9


# ---- CPU oracle timing --------------------------------------------------------------
def oracle_rows_timing(w, A, B, C, rows, threads, keep=False):
    """Seconds the oracle takes for the first `rows` rows of C; with keep,
    also the rows it computed (reference values and magnitudes)."""
    import oracle
    Cn = None if w.beta == 0 else C.numpy()
    t0 = time.perf_counter()
    ref = oracle.sgemm_rows(w.M, w.N, w.K, w.alpha, A.numpy(), w.LDA, B.numpy(), w.LDB, w.beta, Cn,
                            w.LDC, 0, rows, threads=threads)
    dt = time.perf_counter() - t0
    return (dt, ref) if keep else dt


TOL_REL, TOL_ABS = 1e-5, 1e-30
TOLERANCE_RULE = "|C - C_ref| <= 1e-5 * (|alpha| sum_k |a_ik b_kj| + |beta| |c_ij|) + 1e-30"


def check_against_reference(gpu_rows, ref, mag, exact):
    """Compare GPU results with oracle values (float64 arrays of one shape):
    every element within the FP32 tolerance, and bit-exact (as floats) when
    `exact` (integer inputs). Returns (ok, worst error / bound, mismatches)."""
    import numpy as np
    g = np.asarray(gpu_rows, dtype=np.float64)
    err = np.abs(g - ref)
    bound = TOL_REL * mag + TOL_ABS
    ok = np.isfinite(g) & (err <= bound)
    if exact:
        ok &= (g == ref.astype(np.float32).astype(np.float64))
    worst = float(np.max(err / bound)) if err.size else 0.0
    return bool(ok.all()), worst, int(ok.size - int(ok.sum()))


def verify_sample(w, A, B, C, gpu_results, row_ref, n_elements=4096, seed=12345):
    """`gpu_results`: {path: flat C after one call on a fresh C}. Checks each
    against the oracle rows the CPU baseline computed (row_ref: first rows of C)
    and against n_elements seeded elements anywhere in C (the last row and
    column among them)."""
    import numpy as np

    import oracle
    ref_rows, mag_rows = row_ref
    nrows = ref_rows.shape[0]
    rng = np.random.default_rng(seed)
    ri = rng.integers(0, w.M, n_elements)
    ci = rng.integers(0, w.N, n_elements)
    ri[:3] = [w.M - 1, w.M - 1, 0]
    ci[:3] = [w.N - 1, 0, w.N - 1]
    Cn = None if w.beta == 0 else C.numpy()
    ref_el, mag_el = oracle.sgemm_elements(w.M, w.N, w.K, w.alpha, A.numpy(), w.LDA, B.numpy(),
                                           w.LDB, w.beta, Cn, w.LDC, ri, ci)
    exact = w.dist == "int3"
    out = {}
    for path, flat in gpu_results.items():
        g = np.asarray(flat, dtype=np.float32)
        rows = g[:nrows * w.LDC].reshape(nrows, w.LDC)[:, :w.N] if nrows else g[:0].reshape(0, w.N)
        ok_r, worst_r, bad_r = check_against_reference(rows, ref_rows, mag_rows, exact)
        ok_e, worst_e, bad_e = check_against_reference(g[ri * w.LDC + ci], ref_el, mag_el, exact)
        out[path] = {"ok": ok_r and ok_e, "rows_checked": int(nrows),
                     "elements_checked": int(n_elements), "mismatches": bad_r + bad_e,
                     "worst_error_over_bound": round(max(worst_r, worst_e), 6),
                     "bit_exact_required": exact}
    return out


def cpu_baseline(w, A, B, C, budget_s=10.0, gpu_results=None):
    """The oracle as it stands, on the host cores, over a growing row sample
    until about budget_s of CPU work has been timed. With gpu_results
    ({path: flat C from one call on a fresh C}), the rows it computed (plus a
    sample of elements) also check those results: the `verification` entry."""
    threads = len(os.sched_getaffinity(0))
    rows, spent, total_rows, row_ref = max(1, threads), 0.0, 0, None
    while True:
        rows = min(rows, w.M)
        dt, ref = oracle_rows_timing(w, A, B, C, rows, threads, keep=True)
        if dt >= budget_s / 4 or rows == w.M:
            spent, total_rows, row_ref = dt, rows, ref
            break
        rows = min(w.M, max(rows * 2, int(rows * (budget_s / 4) / max(dt, 1e-3))))
    value = gemm_flops(total_rows, w.N, w.K) / spent / 1e9
    # one core, on a few rows (about a second)
    one_rows = max(1, min(w.M, int(total_rows * 0.2 / max(threads, 1))))
    one_dt = oracle_rows_timing(w, A, B, C, one_rows, 1)
    out = {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
           "single_core_value": round(gemm_flops(one_rows, w.N, w.K) / one_dt / 1e9, 3),
           "cpu_model": cpu_model(),
           "sample": f"first {total_rows} of {w.M} rows of C ({w.N} columns, K={w.K}), "
                     f"{spent:.2f} s, FP64 i-j-k loop, rows split over {threads} threads; "
                     f"single core: first {one_rows} rows, {one_dt:.2f} s"}
    if gpu_results:
        out["verification"] = verify_sample(w, A, B, C, gpu_results, row_ref)
    return out


def cpu_model():
    """The host CPU's model name (lscpu), or the platform's processor string."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


# ---- arms ---------------------------------------------------------------------------
def run_reference(args, w):
    """Times the oracle (the CPU reference arm) on bounded row samples."""
    from dense_fp32_gemm_gb300.workloads import make_inputs
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return None
    A, B, C = make_inputs(w)
    threads = len(os.sched_getaffinity(0))
    # rows per step so that one step costs about 0.2 s of host time
    t = oracle_rows_timing(w, A, B, C, threads, threads)
    rows = max(1, min(w.M, int(threads * 0.2 / max(t, 1e-4))))
    for _ in range(args.warmup):
        oracle_rows_timing(w, A, B, C, rows, threads)
    spent = sum(oracle_rows_timing(w, A, B, C, rows, threads) for _ in range(args.steps))
    value = gemm_flops(rows, w.N, w.K) * args.steps / spent / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(spent / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{rows} rows of C per step ({w.N} columns, K={w.K})"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    return line


def workload_config(w):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "lda": w.LDA, "ldb": w.LDB,
            "ldc": w.LDC, "alpha": w.alpha, "beta": w.beta, "dist": w.dist, "seed": w.seed,
            "layout": "row-major",
            "l2": ("inputs larger than L2" if min_bytes(w.M, w.N, w.K, 1) > L2_BYTES
                   else "inputs smaller than L2 (no flush)")}


def run_ours(args, w):
    import torch

    from dense_fp32_gemm_gb300 import binding
    from dense_fp32_gemm_gb300.workloads import make_inputs

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count

    A, B, C = make_inputs(w)
    dA, dB, dC = A.to(dev), B.to(dev), C.to(dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def step(out=None):
        st = binding.sgemm(w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.LDA, dB.data_ptr(), w.LDB,
                           w.beta, (dC if out is None else out).data_ptr(), w.LDC, sh)
        if st != 0:
            raise RuntimeError(f"sgemm: {binding.sgemm_status_string(st)}")

    def step3(out=None):
        st3 = binding.sgemm_3xtf32(w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.LDA, dB.data_ptr(),
                                   w.LDB, w.beta, (dC if out is None else out).data_ptr(), w.LDC,
                                   sh)
        if st3 != 0:
            raise RuntimeError(f"sgemm_3xtf32: {binding.sgemm_status_string(st3)}")

    # one call of each timed path on a fresh C, before any timing; the CPU
    # baseline leg checks these results against the oracle
    fresh = {}
    if rank == 0 and args.cpu_baseline:
        for path, fn in (("ffma", step), ("3xtf32", step3)):
            if path == "3xtf32" and not args.tf32x3:
                continue
            out = C.to(dev)
            fn(out)
            torch.cuda.synchronize(dev)
            fresh[path] = out.cpu().numpy()
            del out

    sampler = None
    if rank == 0:
        sampler = NvmlClockSampler(pci_bus_id=nvml_bus_id(props)).start()
        if sampler.lib is None:
            visible = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
            sampler = ClockSampler(visible[local] if local < len(visible) else str(local))
            time.sleep(1.0)

    with nvtx_range("warmup"):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
    st, detail = binding.sgemm_poll_device_status(sh)
    if st != 0:
        raise RuntimeError(f"device status {st} detail {detail} after warm-up")

    # ---- timed region: exactly K steps -------------------------------------------
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with nvtx_range("timed_steps"):
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    t_wall1 = time.time()
    total_s = start.elapsed_time(end) / 1e3
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_s = sum(step_ms) / 1e3 / args.steps
    if sampler:
        sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    st, detail = binding.sgemm_poll_device_status(sh)
    if st != 0:
        raise RuntimeError(f"device status {st} detail {detail} after timing")
    tile_config = binding.sgemm_last_config()
    total_max = max_over_ranks(total_s, world)
    value = aggregate(gemm_flops(w.M, w.N, w.K), args.steps, total_max, world)

    # ---- the opt-in tensor-core path on the same workload (reported apart) ---------
    tf32x3 = None
    if args.tf32x3:
        for _ in range(args.warmup):
            step3()
        barrier(world)
        torch.cuda.synchronize(dev)
        s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev3 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        with nvtx_range("tf32x3_steps"):
            s3.record(stream)
            for i in range(args.steps):
                ev3[i][0].record(stream)
                step3()
                ev3[i][1].record(stream)
            e3.record(stream)
            torch.cuda.synchronize(dev)
        t3 = max_over_ranks(s3.elapsed_time(e3) / 1e3, world)
        st, detail = binding.sgemm_poll_device_status(sh)
        if st != 0:
            raise RuntimeError(f"device status {st} detail {detail} after the 3xTF32 steps")
        v3 = aggregate(gemm_flops(w.M, w.N, w.K), args.steps, t3, world)
        tf32x3 = {"value": round(v3, 1), "unit": UNIT, "ms_per_step": round(t3 / args.steps * 1e3, 4),
                  "step_ms": step_stats([a.elapsed_time(b) for a, b in ev3]),
                  "config": binding.sgemm_last_config(),
                  "note": "opt-in sgemm_3xtf32: split-operand TF32 on tcgen05, same FP32 tolerance; "
                          "includes its B-transpose pre-pass kernel"}

    # ---- end to end from pinned host buffers, through the C ABI ---------------------
    # sgemm_host copies A, B (and C, as beta != 0) from pinned host memory,
    # overlapping the copies with the multiplication, and copies C back; the
    # timed region covers all of it, every step.
    e2e_steps = max(3, min(args.steps, 20))
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = C.clone().pin_memory()

    def host_step():
        st2 = binding.sgemm_host(w.M, w.N, w.K, w.alpha, hA.data_ptr(), w.LDA, hB.data_ptr(),
                                 w.LDB, w.beta, hC.data_ptr(), w.LDC, sh)
        if st2 != 0:
            raise RuntimeError(f"sgemm_host: {binding.sgemm_status_string(st2)}")
    for _ in range(max(3, min(args.warmup, 10))):
        host_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with nvtx_range("e2e_steps"):
        e0.record(stream)
        for _ in range(e2e_steps):
            host_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = aggregate(gemm_flops(w.M, w.N, w.K), e2e_steps, e2e_s, world)
    h2d_bytes = 4 * (w.M * w.K + w.K * w.N + (w.M * w.N if w.beta != 0 else 0))
    d2h_bytes = 4 * w.M * w.N

    if rank != 0:
        return None
    peaks = measured_peaks()
    max_mhz = float(peaks.get("sm_max_mhz") or (clocks or {}).get("sm_max_mhz") or 2070.0)
    peak_tf = ffma_peak_tflops(sms, max_mhz)
    achieved_tf = gemm_flops(w.M, w.N, w.K) / kern_s / 1e12
    traffic = profiled_traffic(w.name, tile_config)
    sampled = (clocks or {}).get("sm_mhz")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_max / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w),
        "parallelism": f"replicas{world}", "tile_config": tile_config,
        "step_ms": step_stats(step_ms),
        "pct_of_ffma_peak": round(100 * achieved_tf / peak_tf, 2),
        "pct_of_ffma_peak_at_sampled_clock": (round(100 * achieved_tf / ffma_peak_tflops(sms, sampled), 2)
                                              if sampled else None),
        "roofline": {"bound": "alu", "achieved": round(achieved_tf, 3), "peak": round(peak_tf, 3),
                     "unit": "TFLOP/s", "frac": round(achieved_tf / peak_tf, 4),
                     "traffic": traffic,
                     "peak_basis": f"{sms} SMs x {max_mhz:.0f} MHz x 128 FFMA/clk x 2 "
                                   "(FP32 pipe; clock from MEASURED_PEAKS.json sm_max_mhz)",
                     "kernel_ms": round(kern_s * 1e3, 4)},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "steps": e2e_steps, "api": "sgemm_host (pinned host buffers, copies overlapped)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if tf32x3 is not None:
        p3, basis, tf32_measured = tf32x3_roof(binding, peaks,
                                               pair="pair=2sm" in tf32x3["config"])
        a3 = tf32x3["value"] / 1e3
        est = tf32x3_peak_tflops(peaks)
        tf32x3["roofline"] = {"bound": "tensor", "achieved": round(a3, 3),
                              "peak": round(p3, 3) if p3 else None, "unit": "TFLOP/s",
                              "frac": round(a3 / p3, 4) if p3 else None, "peak_basis": basis,
                              "tf32_mma_tflops_measured": (round(tf32_measured, 1)
                                                           if tf32_measured else None),
                              "peak_from_bf16_estimate": round(est, 3) if est else None}
        line["tf32x3"] = tf32x3
    if args.cpu_baseline:
        cb = cpu_baseline(w, A, B, C, budget_s=args.cpu_budget, gpu_results=fresh)
        ver = cb.pop("verification", None)
        line["cpu_baseline"] = cb
        line["verified"] = bool(ver) and all(v["ok"] for v in ver.values())
        line["verification"] = dict(ver or {}, rule=TOLERANCE_RULE,
                                    how="one call per path on a fresh C before any timing, "
                                        "against the oracle rows the CPU baseline computed "
                                        "and seeded single elements")
    else:
        line["verified"] = None
        line["verification"] = {"skipped": "--no-cpu-baseline (the oracle runs in that leg)"}
    return line


REPORT_WORKLOADS = ["square128", "square128_int", "square4096", "edges8191x1000x777",
                    "kdominant1024x1024x16384", "skinny16384x64x4096"] + \
    [f"sweep{n}" for n in (256, 512, 1024, 2048, 4096, 8192, 16384)]

# The pages' own measurements of their kernels at M = N = K = 4096 on an
# RTX 5080 (another GPU: context for the ladder lines, not a target):
# "Shared Memory Tiling", section "The Arithmetic"; "Vectorized Memory Access:
# 128-bit Loads and Stores", section "Mechanics"; "Warp Tiling: A Third Level
# of Tiling", section "Mechanics".
PAGES_LADDER_GFLOPS = {3: 4131.3, 7: 25130.5, 8: 29376.6}


def _mean_ms(call, reps):
    """Mean device time of `reps` back-to-back calls (one event pair)."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        call()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _per_call_ms(call, reps, flush=None):
    """Sorted device times of `reps` calls, one event pair around each; with
    `flush`, a write larger than L2 runs before every call (outside the
    events)."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        if flush is not None:
            flush()
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    return sorted(a.elapsed_time(b) for a, b in ev)


def _reps_for(call, budget_ms=200.0):
    import torch
    call()
    torch.cuda.synchronize()
    one = _mean_ms(call, 1)
    return max(10, int(budget_ms / max(one, 1e-3)))


def _timing_fields(call, reps, flush):
    """mean (back to back), the per-call distribution, and the per-call
    median with L2 flushed before each call."""
    ms = _mean_ms(call, reps)
    per = _per_call_ms(call, min(reps, 500))
    fl = _per_call_ms(call, min(reps, 100), flush=flush)
    return ms, {"ms_min": round(per[0], 5), "ms_median": round(per[len(per) // 2], 5),
                "ms_max": round(per[-1], 5),
                "spread_pct": round(100 * (per[-1] - per[0]) / per[len(per) // 2], 1),
                "ms_median_l2_flushed": round(fl[len(fl) // 2], 5)}


def _l2_flusher():
    import torch
    buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    return lambda: buf.fill_(1.0)


def run_report(args):
    """One JSON line per workload and path: device-timed GFLOP/s of the
    automatic configuration, its fraction of the FFMA peak (the opt-in 3xTF32
    path: of its tensor roof), the per-call time distribution and the time
    with L2 flushed before each call. Not the default line."""
    import torch

    from dense_fp32_gemm_gb300 import binding
    from dense_fp32_gemm_gb300.workloads import WORKLOADS, make_inputs
    props = torch.cuda.get_device_properties(0)
    peaks = measured_peaks()
    max_mhz = float(peaks.get("sm_max_mhz") or 2070.0)
    peak_tf = ffma_peak_tflops(props.multi_processor_count, max_mhz)
    # the 3xTF32 roof of each kernel form: single CTAs, and two-SM pairs
    roof3 = {False: tf32x3_roof(binding, peaks)[0], True: tf32x3_roof(binding, peaks, pair=True)[0]}
    s = torch.cuda.current_stream().cuda_stream
    flush = _l2_flusher()
    for name in REPORT_WORKLOADS:
        w = WORKLOADS[name]
        A, B, C = make_inputs(w)
        dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
        mb = min_bytes(w.M, w.N, w.K, w.beta)
        for path, fn in (("ffma", binding.sgemm), ("3xtf32", binding.sgemm_3xtf32)):
            def call(fn=fn):
                st = fn(w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.LDA, dB.data_ptr(), w.LDB, w.beta,
                        dC.data_ptr(), w.LDC, s)
                if st != 0:
                    raise RuntimeError(binding.sgemm_status_string(st))
            for _ in range(max(3, args.warmup)):
                call()
            torch.cuda.synchronize()
            reps = _reps_for(call)
            ms, dist = _timing_fields(call, reps, flush)
            st, _ = binding.sgemm_poll_device_status(s)
            tf = gemm_flops(w.M, w.N, w.K) / ms / 1e9
            line = {"workload": name, "path": path, "M": w.M, "N": w.N, "K": w.K,
                    "alpha": w.alpha, "beta": w.beta, "ms": round(ms, 5),
                    "gflops": round(tf * 1e3, 1)}
            if path == "ffma":
                line["pct_of_ffma_peak"] = round(100 * tf / peak_tf, 2)
            else:
                p3 = roof3["pair=2sm" in binding.sgemm_last_config()]
                line["pct_of_3xtf32_tensor_roof"] = round(100 * tf / p3, 2) if p3 else None
            line.update({"min_bytes": mb, "achieved_min_gbs": round(mb / ms / 1e6, 1),
                         "achieved_min_gbs_l2_flushed":
                             round(mb / dist["ms_median_l2_flushed"] / 1e6, 1)})
            line.update(dist)
            line.update({"reps": reps, "status": st, "config": binding.sgemm_last_config()})
            print(json.dumps(line), flush=True)
        del dA, dB, dC
        torch.cuda.empty_cache()


# Oracle timing per workload: whole problems up to 4096^3; at 8192^3 and
# 16384^3 a 256-row sample, extrapolated to the whole problem.
ORACLE_REPORT = ["square128", "square4096", "edges8191x1000x777", "kdominant1024x1024x16384",
                 "skinny16384x64x4096"] + [f"sweep{n}" for n in (256, 512, 1024, 2048, 8192, 16384)]
ORACLE_SAMPLE_ROWS = 256


def run_oracle_report(args):
    """The CPU oracle timed on the host cores (all of them, and one), one JSON
    line per workload. Runs on the host only."""
    from dense_fp32_gemm_gb300.workloads import WORKLOADS, make_inputs
    threads = len(os.sched_getaffinity(0))
    model = cpu_model()
    for name in ORACLE_REPORT:
        w = WORKLOADS[name]
        A, B, C = make_inputs(w)
        rows = w.M if w.M * w.N * w.K <= 4096 ** 3 else min(w.M, ORACLE_SAMPLE_ROWS)
        t_all = oracle_rows_timing(w, A, B, C, rows, threads)
        per_row_one_core = t_all * threads / rows
        rows1 = max(1, min(rows, int(1.0 / max(per_row_one_core, 1e-9))))
        t_one = oracle_rows_timing(w, A, B, C, rows1, 1)
        print(json.dumps({
            "workload": name, "M": w.M, "N": w.N, "K": w.K, "rows_timed": rows,
            "extrapolated": rows < w.M,
            "all_cores": threads, "all_core_gflops": round(gemm_flops(rows, w.N, w.K) / t_all / 1e9, 3),
            "all_core_s_whole_problem": round(t_all * w.M / rows, 3),
            "single_core_rows": rows1,
            "single_core_gflops": round(gemm_flops(rows1, w.N, w.K) / t_one / 1e9, 3),
            "single_core_s_whole_problem": round(t_one * w.M / rows1, 3),
            "cpu_model": model}), flush=True)
        del A, B, C


def run_ladder(args):
    """The pages' kernels 3, 7 and 8 next to the library's own kernel on one
    workload (default: the 4096 cube), one JSON line each."""
    import torch

    from dense_fp32_gemm_gb300 import binding
    from dense_fp32_gemm_gb300.workloads import WORKLOADS, make_inputs
    props = torch.cuda.get_device_properties(0)
    peaks = measured_peaks()
    max_mhz = float(peaks.get("sm_max_mhz") or 2070.0)
    peak_tf = ffma_peak_tflops(props.multi_processor_count, max_mhz)
    s = torch.cuda.current_stream().cuda_stream
    flush = _l2_flusher()
    w = WORKLOADS[args.workload]
    A, B, C = make_inputs(w)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    runs = [(f"ladder_kernel{k}", functools.partial(binding.sgemm_ladder, k), k)
            for k in binding.LADDER_KERNELS] + [("sgemm", binding.sgemm, None)]
    base_ms = None
    lines = []
    for path, fn, k in runs:
        def call(fn=fn):
            st = fn(w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.LDA, dB.data_ptr(), w.LDB, w.beta,
                    dC.data_ptr(), w.LDC, s)
            if st != 0:
                raise RuntimeError(binding.sgemm_status_string(st))
        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        if args.profile_once:
            # for a profiler: one more call per kernel, no timing
            call()
            torch.cuda.synchronize()
            print(json.dumps({"workload": w.name, "path": path, "calls": max(3, args.warmup) + 1,
                              "config": binding.sgemm_last_config()}), flush=True)
            continue
        reps = _reps_for(call, budget_ms=300.0)
        ms, dist = _timing_fields(call, reps, flush)
        tf = gemm_flops(w.M, w.N, w.K) / ms / 1e9
        line = {"workload": w.name, "path": path, "M": w.M, "N": w.N, "K": w.K, "ms": round(ms, 5),
                "gflops": round(tf * 1e3, 1), "pct_of_ffma_peak": round(100 * tf / peak_tf, 2)}
        line.update(dist)
        line.update({"reps": reps, "config": binding.sgemm_last_config()})
        if k is not None and w.M == w.N == w.K == 4096:
            line["pages_gflops_rtx5080"] = PAGES_LADDER_GFLOPS[k]
        if path == "sgemm":
            base_ms = ms
        lines.append(line)
    for line in lines if base_ms else []:
        line["time_vs_sgemm"] = round(line["ms"] / base_ms, 2)
        print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="square4096")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-tf32x3", dest="tf32x3", action="store_false",
                    help="skip timing the opt-in 3xTF32 tensor-core path")
    ap.add_argument("--report", action="store_true",
                    help="time every named workload and the sweep, one JSON line each")
    ap.add_argument("--ladder", action="store_true",
                    help="time the pages' kernels 3, 7, 8 and sgemm on --workload")
    ap.add_argument("--oracle-report", action="store_true",
                    help="time the CPU oracle on every workload (host only)")
    ap.add_argument("--profile-once", action="store_true",
                    help="with --ladder: warm-up calls plus one call per kernel, no timing")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.report:
        run_report(args)
        return
    if args.ladder:
        run_ladder(args)
        return
    if args.oracle_report:
        run_oracle_report(args)
        return
    from dense_fp32_gemm_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    line = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if line is not None:
        print(json.dumps(line), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
