#!/usr/bin/env python3
"""Throughput of the dense bf16 GEMM on GB300, as one JSON line.

Workload (one "step"): C = GELU_tanh(A @ B + bias) with M = N = K = 8192,
A row-major and B column-major bf16, Uniform(-1,1)/sqrt(K) from a seed, bias
fp32 N(0,1), fp32 accumulation, bf16 output; one call of the library's C ABI
(``gemm_batched``) on the current stream.  Metric: TFLOPS = 2MNK / time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--rows FILE] [--row NAME]

The line also carries ``rows``: the other workloads (bf16 256^3, SGEMM
4096^3, ragged 4097x3001x1000, split-K 256x256x65536, skinny 16x8192x8192,
batched 64x1024^3 with per-entry and broadcast B), each timed over cold-L2
launches with its roofline fraction and a clock sample (--no-rows skips them).
--impl reference times the CPU oracle (plain fp64 C, unchanged) on a bounded
slice of the same workload, split into row slices over one process per host
core: the deliberately slow baseline.  The line's cpu_baseline is the same
harness.  --rows FILE measures every library path (the rows above plus
stream-K and flat-K shapes) into FILE; --row NAME runs only that path
(--steps launches) and prints its JSON object.
Multi-GPU runs (torchrun) run one independent replica per GPU (weak scaling).
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS (2MNK/s), bf16 8192^3, and % of GB300 dense BF16 tensor peak"
UNIT = "TFLOPS"
M = N = K = 8192
WORKLOAD = ("bf16 GEMM M=N=K=8192, A row-major, B column-major, fused bias + GELU(tanh), "
            "fp32 accumulate, bf16 output")
WORKLOAD_ID = 3  # seeds 3001 (A), 3002 (B), 3004 (bias)
L2_NOTE = "inputs larger than L2: A + B = 256 MiB and C = 128 MiB vs a 126.5 MiB L2; no flush"
TC_SOURCES = ["tc_kernel.cuh", "tc_gemm.cu", "tc_gemm_fast.cu", "tc_gemm_general.cu", "ptx.cuh",
              "epilogue.cuh", "tile_order.h", "internal.h", "tc_gemm_ks2.cu", "debug_check.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rows", default=None, help="also measure the other paths into this file")
    ap.add_argument("--row", default=None, choices=ROW_NAMES,
                    help="run only this other path (--steps launches) and print its timing")
    ap.add_argument("--ablation", default=None,
                    help="interleaved GROUP_M / L2-hint / CTA-pair ablation of the headline "
                         "into this file (JSON)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="leave the other workloads out")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


class Replicas:
    """Host side of an N-process run: one independent replica of the workload per
    rank, one GPU each, and no collective on the data path (tiles are
    independent).  Barriers bracket the timed regions, a time is the maximum
    over ranks, and whole-job throughput counts every rank's work."""

    def __init__(self, backend, device=None, timeout_s=900.0):
        rank, world, local = env_rank()
        self.rank, self.world, self.local = rank, world, local
        self.dist = None
        self.device = device
        if world > 1:
            import datetime

            import torch.distributed as dist
            # a rank that dies makes the others' next barrier or reduction fail
            # after timeout_s instead of the backend's default half hour
            timeout = datetime.timedelta(seconds=timeout_s)
            if backend == "nccl":
                dist.init_process_group(backend, device_id=device, timeout=timeout)
            else:
                dist.init_process_group(backend, timeout=timeout)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x):
        """The maximum of x over the ranks."""
        if self.dist is None:
            return x
        import torch
        dev = self.device if self.dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def throughput(self, work_per_rank, ms):
        """Whole-job rate: every rank's work over the slowest rank's time."""
        return self.world * work_per_rank / (ms * 1e-3)

    def close(self):
        if self.dist is not None:
            self.dist.barrier()
            self.dist.destroy_process_group()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def tc_source_sha():
    h = hashlib.sha256()
    for name in TC_SOURCES:
        with open(os.path.join(ROOT, "dense_gemm_bf16_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "tc_gemm_bf16_8192_bias_gelu.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = traffic = None
    for line in text.splitlines():
        if line.startswith("kernel_source_sha256:"):
            sha = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if sha == tc_source_sha() else None


# ----------------------------------------------------------------------------- inputs

def c3_host_inputs():
    import numpy as np

    import datagen
    a = datagen.to_bf16_bits(datagen.uniform(datagen.seed_for(WORKLOAD_ID, datagen.ROLE_A),
                                             (M, K)) / math.sqrt(K))
    b = datagen.to_bf16_bits(datagen.uniform(datagen.seed_for(WORKLOAD_ID, datagen.ROLE_B),
                                             (K, N)) / math.sqrt(K))
    b_cm = np.ascontiguousarray(b.T)  # column-major storage: B(k, n) at n*K + k
    bias = datagen.to_f32(datagen.normal(datagen.seed_for(WORKLOAD_ID, datagen.ROLE_BIAS), (N,)))
    return a, b_cm, bias


class Gemm:
    """The C3 call through the C ABI, bound to fixed device buffers."""

    def __init__(self, dA, dB, dbias, dC, stream):
        import dense_gemm_bf16_gb300 as dg
        self.dg = dg
        self.args = [int(dg.DType.BF16), 1, M, N, K, dA.data_ptr(), K, 0, 0, dB.data_ptr(), K,
                     1, 0, dC.data_ptr(), N, 0, 0, int(dg.DType.BF16), 1.0, 0.0,
                     dbias.data_ptr(), int(dg.Epi.BIAS_GELU_TANH), 0]
        st, plan = dg.gemm_plan_query(*self.args, 0)
        if st != 0:
            raise RuntimeError(f"plan: {dg.gemm_status_string(st)}")
        self.plan = plan.as_dict()
        self.stream = stream

    def __call__(self):
        st = self.dg.gemm_batched(*self.args, None, 0, self.stream)
        if st != 0:
            raise RuntimeError(f"gemm_batched: {self.dg.gemm_status_string(st)}")


def e2e_pipelined(hA, hB, hbias, hC, device, steps, warmup, barrier=None):
    """End to end with host buffers, overlapped across steps: every step copies
    its inputs host -> device, runs the GEMM and copies its result back, on
    three streams with two device copies of each buffer, so that the inputs of
    step i + 1 go up and the result of step i - 1 comes down while step i
    computes.  Returns ms per step (CUDA events on the joining stream)."""
    import torch
    s_in, s_mm, s_out = (torch.cuda.Stream(device) for _ in range(3))
    bufs = []
    for _ in range(2):
        dA = torch.empty_like(hA, device=device)
        dB = torch.empty_like(hB, device=device)
        dbias = torch.empty_like(hbias, device=device)
        dC = torch.empty(hC.shape, dtype=hC.dtype, device=device)
        bufs.append((dA, dB, dbias, dC, Gemm(dA, dB, dbias, dC, s_mm.cuda_stream)))
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer j landed
    ev_mm = [torch.cuda.Event() for _ in range(2)]    # GEMM on buffer j done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # result of buffer j copied out
    main = torch.cuda.current_stream(device)

    def step(i):
        j = i & 1
        dA, dB, dbias, dC, gemm = bufs[j]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_mm[j])        # step i - 2 has read these inputs
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            dbias.copy_(hbias, non_blocking=True)
            ev_in[j].record(s_in)
        s_mm.wait_event(ev_in[j])
        if i >= 2:
            s_mm.wait_event(ev_out[j])           # step i - 2's result has been read out
        gemm()
        ev_mm[j].record(s_mm)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_mm[j])
            hC.copy_(dC, non_blocking=True)
            ev_out[j].record(s_out)

    def run(n):
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(main)
        for s_ in (s_in, s_mm, s_out):
            s_.wait_stream(main)
        for i in range(n):
            step(i)
        for s_ in (s_in, s_mm, s_out):
            main.wait_stream(s_)
        stop.record(main)
        torch.cuda.synchronize(device)
        return start.elapsed_time(stop)

    with nvtx("e2e warmup"):
        run(warmup)
    if barrier:
        barrier()
    with nvtx("e2e timed"):
        ms = run(steps)
    if barrier:
        barrier()
    return ms / steps


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index):
        import torch
        self.proc = None
        target = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            target = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"] + target, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- timing

@contextlib.contextmanager
def nvtx(name):
    """An NVTX range around a phase (warm-up, timed, e2e, one row), so that a
    profiler can select it (ncu --nvtx --nvtx-include "timed/")."""
    import torch
    try:
        torch.cuda.nvtx.range_push(name)
        pushed = True
    except Exception:
        pushed = False
    try:
        yield
    finally:
        if pushed:
            torch.cuda.nvtx.range_pop()


def time_steps(fn, steps, warmup, barrier=None):
    import torch
    with nvtx("warmup"):
        for _ in range(warmup):
            fn()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with nvtx("timed"):
        start.record()
        for _ in range(steps):
            fn()
        stop.record()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return start.elapsed_time(stop)  # ms for all steps


# ----------------------------------------------------------------------------- CPU oracle

def _oracle_problem(a_rows, b_cm_cols, bias_cols):
    """The workload restricted to some rows of A and columns of B (full K)."""
    import oracle
    return oracle.Problem(ab_dtype="bf16", M=a_rows.shape[0], N=b_cm_cols.shape[0], K=K,
                          A=a_rows.ravel(), lda=K, la="row", B=b_cm_cols.ravel(), ldb=K,
                          lb="col", c_dtype="bf16", bias=bias_cols, act="gelu_tanh")


def oracle_sample_seconds(a, b_cm, bias, rows, cols):
    """The oracle, as it stands, on the first `rows` x `cols` outputs of the
    workload (full K), in this process.  Returns (seconds, flops)."""
    import numpy as np

    import oracle
    p = _oracle_problem(a[:rows], np.ascontiguousarray(b_cm[:cols]), bias[:cols])
    t0 = time.perf_counter()
    oracle.gemm(p)
    return time.perf_counter() - t0, 2.0 * rows * cols * K


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


# worker side of OracleCores (a spawned process: module-level state only)
_W = {}


def _oracle_worker_init(names, shapes):
    import numpy as np
    from multiprocessing import shared_memory

    import oracle
    oracle.build()
    for key in ("a", "b", "bias"):
        shm = shared_memory.SharedMemory(name=names[key])
        dt = np.float32 if key == "bias" else np.uint16
        _W[key + "_shm"] = shm
        _W[key] = np.ndarray(shapes[key], dtype=dt, buffer=shm.buf)


def _oracle_worker_ready(_):
    return os.getpid()


def _oracle_worker_run(job):
    """Rows r0 .. r1 (of the first rows of A) x the first `cols` columns."""
    import numpy as np

    import oracle
    r0, r1, cols = job
    if r1 <= r0:
        return 0.0
    p = _oracle_problem(np.ascontiguousarray(_W["a"][r0:r1]),
                        np.ascontiguousarray(_W["b"][:cols]), _W["bias"][:cols])
    t0 = time.perf_counter()
    oracle.gemm(p)
    return time.perf_counter() - t0


class OracleCores:
    """The oracle (unchanged, single-threaded C) on every host core: one
    spawned process per core, each computing a slice of rows of the same
    sample from A and B in shared memory.  A sample's time is the wall time
    from handing out the slices to the last one's return."""

    def __init__(self, a, b_cm, bias, max_rows):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        self.cores = _host_cores()
        arrays = {"a": a[:max_rows], "b": b_cm, "bias": bias}
        self.shm, names, shapes = {}, {}, {}
        for key, arr in arrays.items():
            shm = shared_memory.SharedMemory(create=True, size=max(arr.nbytes, 1))
            import numpy as np
            np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
            self.shm[key], names[key], shapes[key] = shm, shm.name, arr.shape
        self.max_rows = max_rows
        # spawn: the parent holds a CUDA context, which a forked child must not inherit
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_oracle_worker_init,
                                                 initargs=(names, shapes))
        # every worker started and initialised before anything is timed (a
        # worker that cannot start would be replaced forever: bounded wait)
        self._map(_oracle_worker_ready, range(4 * self.cores), 300)

    def _map(self, fn, jobs, timeout_s):
        try:
            return self.pool.map_async(fn, jobs, chunksize=1).get(timeout_s)
        except BaseException:
            self.pool.terminate()
            raise

    def run(self, rows, cols):
        """Wall seconds for rows x cols outputs split over the cores."""
        rows = min(rows, self.max_rows)
        bounds = [rows * i // self.cores for i in range(self.cores + 1)]
        jobs = [(bounds[i], bounds[i + 1], cols) for i in range(self.cores)]
        t0 = time.perf_counter()
        self._map(_oracle_worker_run, jobs, 1800)
        return time.perf_counter() - t0, 2.0 * rows * cols * K

    def close(self):
        self.pool.close()
        self.pool.join()
        for shm in self.shm.values():
            shm.close()
            shm.unlink()


def _rows_for(seconds, per_out, cores):
    """Rows of the full-width sample that take about `seconds` on `cores`."""
    return max(cores, int(seconds * cores / max(per_out, 1e-9)) // N)


def cpu_baseline(a, b_cm, bias, target_s=8.0):
    """The oracle on every host core, on a sample of whole rows of the
    workload sized for about target_s seconds (calibrated on one core)."""
    dt, _ = oracle_sample_seconds(a, b_cm, bias, 1, 512)
    cores = _host_cores()
    rows = min(_rows_for(target_s, dt / 512, cores), M)
    pool = OracleCores(a, b_cm, bias, rows)
    try:
        t, fl = pool.run(rows, N)
    finally:
        pool.close()
    return {"value": fl / t / 1e12, "unit": UNIT, "cores": pool.cores, "kind": "oracle",
            "sample": f"first {rows} rows x {N} columns of C (full K = {K}), split into row "
                      f"slices over {pool.cores} processes (one per host core), {t:.1f} s "
                      "wall; fp64 oracle, unchanged, one thread per process"}


def reference_arm(args):
    """Times the oracle on this host's cores: one bounded sample of whole rows
    per step, split over one process per core."""
    a, b_cm, bias = c3_host_inputs()
    dt, _ = oracle_sample_seconds(a, b_cm, bias, 1, 256)
    cores = _host_cores()
    budget = 150.0 / (args.steps + args.warmup)  # whole run within a few minutes
    rows = min(_rows_for(budget, dt / 256, cores), M)
    pool = OracleCores(a, b_cm, bias, rows)
    try:
        for _ in range(args.warmup):
            pool.run(rows, N)
        tot_t, tot_f = 0.0, 0.0
        for _ in range(args.steps):
            t, f = pool.run(rows, N)
            tot_t += t
            tot_f += f
    finally:
        pool.close()
    value = tot_f / tot_t / 1e12
    sample = (f"per step: the first {rows} rows x {N} columns of C (full K = {K}), split into "
              f"row slices over {pool.cores} processes (one per host core); fp64 oracle, "
              f"unchanged, one thread per process; {args.steps} steps")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main arm

def main():
    args = parse_args()
    rank, world, local = env_rank()
    if args.impl == "reference":
        if rank != 0:
            return
        reference_arm(args)
        return

    import numpy as np
    import torch

    import dense_gemm_bf16_gb300 as dg

    torch.cuda.set_device(local if world > 1 else 0)
    device = torch.device("cuda", local if world > 1 else 0)
    reps = Replicas("nccl", device)
    dg.build()
    dg.lib()
    if args.row:
        print(json.dumps(measure_rows([args.row], device, reps=args.steps)[0]), flush=True)
        return
    if args.ablation:
        run_ablation(args, device)
        return

    a, b_cm, bias = c3_host_inputs()
    hA = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    hB = torch.from_numpy(b_cm.view(np.int16)).view(torch.bfloat16).pin_memory()
    hbias = torch.from_numpy(bias).pin_memory()
    dA = hA.to(device)
    dB = hB.to(device)
    dbias = hbias.to(device)
    dC = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    hC = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream(device).cuda_stream
    gemm = Gemm(dA, dB, dbias, dC, stream)

    barrier = reps.barrier
    max_over_ranks = reps.max

    # device-resident throughput (clocks sampled during the timed region)
    sampler = ClockSampler(device.index)
    time.sleep(0.3)
    ms_total = time_steps(gemm, args.steps, args.warmup, barrier)
    clocks = sampler.stop()
    ms_total = max_over_ranks(ms_total)
    ms_step = ms_total / args.steps
    flops = 2.0 * M * N * K
    value = reps.throughput(flops, ms_step) / 1e12

    # end to end through the C ABI with host buffers: every step H2D inputs, GEMM,
    # D2H result.  Reported: the copies overlapped across steps (three streams);
    # beside it, the same step with everything serial on one stream.
    e2e = None
    if not args.no_e2e:
        def e2e_step():
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            dbias.copy_(hbias, non_blocking=True)
            gemm()
            hC.copy_(dC, non_blocking=True)
        e2e_steps = max(5, min(args.steps, 50))
        ms_serial = max_over_ranks(time_steps(e2e_step, e2e_steps, 3, barrier)) / e2e_steps
        ms_e2e = max_over_ranks(e2e_pipelined(hA, hB, hbias, hC, device, e2e_steps, 3, barrier))
        h2d = hA.numel() * 2 + hB.numel() * 2 + hbias.numel() * 4
        e2e = {"value": reps.throughput(flops, ms_e2e) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hC.numel() * 2,
               "ms_per_step": ms_e2e,
               "overlap": "inputs of step i+1 up and result of step i-1 down while step i "
                          "computes (three streams, two device copies of each buffer)",
               "serial_value": reps.throughput(flops, ms_serial) / 1e12,
               "serial_ms_per_step": ms_serial}

    peaks, peak_src = measured_peaks()
    achieved = flops / (ms_step * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": profiled_traffic(), "peak_source": peak_src + " (bf16 burst)",
                "frac_vs_sustained_peak": achieved / peaks.get("bf16_tflops_sustained",
                                                               peaks["bf16_tflops"]),
                "kernel": "tc_gemm_kernel<256, 2, 1, 2>"}

    if args.rows and rank == 0:
        with open(args.rows, "w") as f:
            json.dump(measure_rows(ROW_NAMES, device), f, indent=1)

    # the other workloads, one GPU at a time (a single-GPU run only)
    rows = None
    if not args.no_rows and world == 1:
        rows = line_rows(device)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(a, b_cm, bias)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K,
                           "layout": "A row-major, B column-major, C row-major",
                           "epilogue": "bias + GELU(tanh)", "l2": L2_NOTE,
                           "parallelism": "replicas" if world > 1 else "single GPU",
                           "plan": gemm.plan},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps * gemm.plan["launches"],
                "clocks": clocks, "rows": rows}
        print(json.dumps(line), flush=True)
    reps.close()


# ----------------------------------------------------------------------------- ablation

ABLATION = [  # (label, GEMM options)
    ("group_m=8 (default)", {}),
    ("group_m=1 (row-major tile order)", {"GROUP_M": 1}),
    ("group_m=4", {"GROUP_M": 4}),
    ("group_m=16", {"GROUP_M": 16}),
    ("group_m=32", {"GROUP_M": 32}),
    ("L2 hints: A evict-first, B evict-last", {"L2_HINTS": 1}),
    ("L2 hints: A evict-last, B evict-first", {"L2_HINTS": 2}),
    ("single-CTA tiles (no CTA pairs)", {"CTA_PAIR": 1}),
    ("256 x 512 pair tiles (one accumulator)", {"WIDE_TILE": 2}),
    ("one K block per TMA load", {"DOUBLE_K": 1}),
]


def run_ablation(args, device, reps=None, launches=20):
    """Headline workload under each setting.  Every repetition runs all
    settings back to back, and the order rotates by one each repetition (a
    Latin square): each setting takes each position once, so the power-cap
    ramp within a repetition hits all settings alike."""
    import numpy as np
    import torch

    import dense_gemm_bf16_gb300 as dg
    a, b_cm, bias = c3_host_inputs()
    dA = torch.from_numpy(a.view(np.int16)).to(device)
    dB = torch.from_numpy(b_cm.view(np.int16)).to(device)
    dbias = torch.from_numpy(bias).to(device)
    dC = torch.empty((M, N), dtype=torch.int16, device=device)
    gemm = Gemm(dA, dB, dbias, dC, torch.cuda.current_stream(device).cuda_stream)
    defaults = {name: dg.gemm_get_option(dg.Option[name])
                for name in ("GROUP_M", "L2_HINTS", "CTA_PAIR", "WIDE_TILE")}
    times = {label: [] for label, _ in ABLATION}
    reps = reps or len(ABLATION)
    sampler = ClockSampler(device.index)
    for r in range(reps):
        order = ABLATION[r % len(ABLATION):] + ABLATION[:r % len(ABLATION)]
        for label, opts in order:
            for name, val in defaults.items():
                dg.gemm_set_option(dg.Option[name], opts.get(name, val))
            ms = time_steps(gemm, launches, 3)
            times[label].append(ms / launches)
    clocks = sampler.stop()
    for name, val in defaults.items():
        dg.gemm_set_option(dg.Option[name], val)
    flops = 2.0 * M * N * K
    out = {"workload": WORKLOAD, "reps": reps, "launches_per_rep": launches, "clocks": clocks,
           "results": [{"setting": label, "ms_median": statistics.median(times[label]),
                        "ms_all": times[label],
                        "tflops": flops / (statistics.median(times[label]) * 1e-3) / 1e12}
                       for label, _ in ABLATION]}
    with open(args.ablation, "w") as f:
        json.dump(out, f, indent=1)
    for r in out["results"]:
        print(f"{r['setting']:40s} {r['ms_median'] * 1000:8.1f} us {r['tflops']:8.1f} TFLOPS")


# ----------------------------------------------------------------------------- other paths

ROW_NAMES = ("small_256", "sgemm_4096", "ragged_4097x3001x1000", "splitk_256x256x65536",
             "skinny_16x8192x8192", "batched_64x1024", "batched_64x1024_bcast",
             "streamk_2560x2560x16384", "streamk_off_2560x2560x16384",
             "flat_4096x4096x16", "flat_4096x4096x16_f32")
# library options a row runs under (restored afterwards)
ROW_OPTIONS = {"streamk_off_2560x2560x16384": {"STREAM_K": 1}}


def build_row(name, device):
    """Inputs and one call of a non-headline path.  Returns
    (fn, flops, algorithmic_bytes, bound, plan, keepalive)."""
    import numpy as np
    import torch

    import datagen
    import dense_gemm_bf16_gb300 as dg
    peaks, _ = measured_peaks()
    stream = torch.cuda.current_stream(device).cuda_stream

    def dev(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    def bf16(seed, shape):
        return dev(datagen.to_bf16_bits(datagen.uniform(seed, shape)).view(np.int16))

    def call16(batch, m, n, k, A, lda, sa, B, ldb, sb, C, ldc, sc, cdt, alpha, beta):
        args_ = [0, batch, m, n, k, A.data_ptr(), lda, 0, sa, B.data_ptr(), ldb, 0, sb,
                 C.data_ptr(), ldc, 0, sc, cdt, alpha, beta, None, 0, 0]
        st, plan = dg.gemm_plan_query(*args_, 1 << 62)
        if st != 0:
            raise RuntimeError(dg.gemm_status_string(st))
        wst = torch.empty(max(int(plan.workspace_bytes), 256), dtype=torch.uint8, device=device)

        def fn():
            s_ = dg.gemm_batched(*args_, wst.data_ptr(), wst.numel(), stream)
            if s_ != 0:
                raise RuntimeError(dg.gemm_status_string(s_))
        return fn, plan.as_dict(), wst

    if name == "small_256":
        # bf16 256^3, row-major A and B, bf16 out, no epilogue: launch-latency bound
        n = 256
        A = dev(datagen.to_bf16_bits(datagen.uniform(datagen.seed_for(1, datagen.ROLE_A),
                                                     (n, n))).view(np.int16))
        B = dev(datagen.to_bf16_bits(datagen.uniform(datagen.seed_for(1, datagen.ROLE_B),
                                                     (n, n))).view(np.int16))
        C = torch.empty((n, n), dtype=torch.int16, device=device)
        fn, plan, wst = call16(1, n, n, n, A, n, 0, B, n, 0, C, n, 0, 0, 1.0, 0.0)
        return fn, 2.0 * n ** 3, 4 * n * n * 2, "hbm", plan, (A, B, C, wst)
    if name == "sgemm_4096":
        n = 4096
        A = dev(datagen.to_f32(datagen.uniform(2001, (n, n))))
        B = dev(datagen.to_f32(datagen.uniform(2002, (n, n))))
        C = dev(datagen.to_f32(datagen.uniform(2003, (n, n))))

        def fn():
            s_ = dg.sgemm_f32(n, n, n, A.data_ptr(), n, 0, B.data_ptr(), n, 0, C.data_ptr(), n, 0,
                              1.5, 0.5, None, 0, stream)
            if s_ != 0:
                raise RuntimeError(dg.gemm_status_string(s_))
        return fn, 2.0 * n ** 3, 4 * n * n * 4, "alu", {"kernel": 2}, (A, B, C)
    if name in ("ragged_4097x3001x1000", "splitk_256x256x65536", "skinny_16x8192x8192"):
        m_, n_, k_ = {"ragged_4097x3001x1000": (4097, 3001, 1000),
                      "splitk_256x256x65536": (256, 256, 65536),
                      "skinny_16x8192x8192": (16, 8192, 8192)}[name]
        seed = {"ragged_4097x3001x1000": 4001, "splitk_256x256x65536": 4011,
                "skinny_16x8192x8192": 4021}[name]
        A = bf16(seed, (m_, k_))
        B = bf16(seed + 1, (k_, n_))
        C = torch.empty((m_, n_), dtype=torch.float32, device=device)
        fn, plan, wst = call16(1, m_, n_, k_, A, k_, 0, B, n_, 0, C, n_, 0, 2, 1.0, 0.0)
        nbytes = (m_ * k_ + k_ * n_) * 2 + m_ * n_ * 4
        flops = 2.0 * m_ * n_ * k_
        bound = "tensor" if name.startswith("ragged") else "hbm"
        return fn, flops, nbytes, bound, plan, (A, B, C, wst)
    if name in ("batched_64x1024", "batched_64x1024_bcast"):
        bt, s_ = 64, 1024
        A = bf16(5001, (bt, s_, s_))
        B = bf16(5002, (bt, s_, s_))
        C = dev(datagen.to_bf16_bits(datagen.normal(5003, (bt, s_, s_))).view(np.int16))
        sb = 0 if name.endswith("bcast") else s_ * s_
        fn, plan, wst = call16(bt, s_, s_, s_, A, s_, s_ * s_, B, s_, sb, C, s_, s_ * s_, 0, 0.5,
                               1.0)
        nbytes = (bt * s_ * s_ + (bt if sb else 1) * s_ * s_ + 2 * bt * s_ * s_) * 2
        flops = 2.0 * bt * s_ ** 3
        t_comp = flops / (peaks["bf16_tflops"] * 1e12)
        t_mem = nbytes / (peaks["hbm_gbs"] * 1e9)
        return fn, flops, nbytes, "hbm" if t_mem > t_comp else "tensor", plan, (A, B, C, wst)
    if name in ("streamk_2560x2560x16384", "streamk_off_2560x2560x16384"):
        # 10 x 10 tiles of 256 x 256: one whole wave on the GPU's CTA pairs and a
        # partial one, which stream-K cuts along K
        m_ = n_ = 2560
        k_ = 16384
        A = bf16(6001, (m_, k_))
        B = bf16(6002, (k_, n_))
        C = torch.empty((m_, n_), dtype=torch.int16, device=device)
        fn, plan, wst = call16(1, m_, n_, k_, A, k_, 0, B, n_, 0, C, n_, 0, 0, 1.0, 0.0)
        nbytes = (m_ * k_ + k_ * n_ + m_ * n_) * 2
        return fn, 2.0 * m_ * n_ * k_, nbytes, "tensor", plan, (A, B, C, wst)
    if name in ("flat_4096x4096x16", "flat_4096x4096x16_f32"):
        # flat product ("2 . La GEMM, de zero a cuBLAS", small-K exercise): the
        # output write is nearly all of the traffic
        m_ = n_ = 4096
        k_ = 16
        f32 = name.endswith("f32")
        A = bf16(7001, (m_, k_))
        B = bf16(7002, (k_, n_))
        C = torch.empty((m_, n_), dtype=torch.float32 if f32 else torch.int16, device=device)
        fn, plan, wst = call16(1, m_, n_, k_, A, k_, 0, B, n_, 0, C, n_, 0, 2 if f32 else 0, 1.0,
                               0.0)
        nbytes = (m_ * k_ + k_ * n_) * 2 + m_ * n_ * (4 if f32 else 2)
        return fn, 2.0 * m_ * n_ * k_, nbytes, "hbm", plan, (A, B, C, wst)
    raise ValueError(f"unknown row {name!r}")


# the workloads besides the headline that the default line reports
LINE_ROWS = ("small_256", "sgemm_4096", "ragged_4097x3001x1000", "splitk_256x256x65536",
             "skinny_16x8192x8192", "batched_64x1024", "batched_64x1024_bcast")
PLAN_KEYS = ("block_n", "block_k", "cta_pair", "split_k", "stream_k", "fast_epilogue",
             "swap_ab", "pack_a", "pack_b", "grid", "launches")


def line_rows(device, reps=20):
    """The other workloads for the default line: per row the median time of
    `reps` cold-L2 launches, throughput, roofline fraction and plan, plus one
    clock sample over all of them."""
    sampler = ClockSampler(device.index)
    out = measure_rows(LINE_ROWS, device, reps=reps)
    clocks = sampler.stop()
    rows = {}
    for r in out:
        plan = r["plan"]
        rows[r["path"]] = {
            "us_median": r["ms_median"] * 1e3, "us_min": r["ms_min"] * 1e3,
            "tflops": r["tflops"], "gbs": r["gbs"], "bound": r["bound"], "peak": r["peak"],
            "frac": r["frac"], "flops": r["flops"], "algorithmic_bytes": r["algorithmic_bytes"],
            "plan": {k: plan[k] for k in PLAN_KEYS if k in plan} if "block_n" in plan else plan}
        if "peak_source" in r:
            rows[r["path"]]["peak_source"] = r["peak_source"]
    return {"timing": f"median of {reps} launches, each after a read of a 256 MiB buffer "
                      "(cold L2), CUDA events on the launching stream",
            "clocks": clocks, "results": rows}


def fp32_peak_tflops(device):
    """FP32 CUDA-core peak from unit counts and the clock: SMs x 128 FMA lanes x
    2 FLOP x the maximum SM clock (nvidia-smi), in TFLOP/s; None if unknown."""
    import subprocess

    import torch
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(torch.cuda.current_device()),
                              "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits"],
                             capture_output=True, text=True, timeout=20).stdout
        mhz = float(out.strip().splitlines()[0])
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        return None, None
    return sms * 128 * 2 * mhz * 1e6 / 1e12, mhz


def measure_rows(names, device, reps=20):
    """Times each named path with its roofline fraction: `reps` launches after
    3 warm-ups, each preceded by a read of a buffer twice the size of L2 (so
    every launch starts with a cold L2 that holds only clean lines: after a
    write instead, a memory-bound launch would also pay for writing the
    flush's dirty lines back to HBM) and bracketed by CUDA events on the
    launching stream.  All launches are queued before the first is waited
    for, so the host's time to issue a call (about 6 us) stays outside the
    events; the median per-launch time is reported."""
    import torch
    import dense_gemm_bf16_gb300 as dg
    peaks, _ = measured_peaks()
    flush = torch.zeros(64 << 20, dtype=torch.float32, device=device)  # 256 MiB
    out = []
    for name in names:
        saved = {k: dg.gemm_get_option(dg.Option[k]) for k in ROW_OPTIONS.get(name, {})}
        for k, v in ROW_OPTIONS.get(name, {}).items():
            dg.gemm_set_option(dg.Option[k], v)
        fn, flops, nbytes, bound, plan, keep = build_row(name, device)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        evs = []
        with nvtx(f"row {name}"):
            for _ in range(reps):
                flush.sum()
                s_ = torch.cuda.Event(enable_timing=True)
                e_ = torch.cuda.Event(enable_timing=True)
                s_.record()
                fn()
                e_.record()
                evs.append((s_, e_))
        torch.cuda.synchronize()
        ts = [s_.elapsed_time(e_) for s_, e_ in evs]
        med, mn = statistics.median(ts), min(ts)
        r = {"path": name, "ms_median": med, "ms_min": mn, "tflops": flops / (med * 1e-3) / 1e12,
             "gbs": nbytes / (med * 1e-3) / 1e9, "algorithmic_bytes": nbytes, "flops": flops,
             "bound": bound, "plan": plan}
        if bound == "hbm":
            r["peak"], r["frac"] = peaks["hbm_gbs"], r["gbs"] / peaks["hbm_gbs"]
        elif bound == "tensor":
            r["peak"], r["frac"] = peaks["bf16_tflops"], r["tflops"] / peaks["bf16_tflops"]
        else:
            # fp32 FMA pipe: SM count x 128 lanes x 2 FLOP x the maximum SM clock
            pk, mhz = fp32_peak_tflops(device)
            r["peak"] = pk
            r["peak_source"] = f"derived: SMs x 128 FMA lanes x 2 x {mhz} MHz" if pk else None
            r["frac"] = r["tflops"] / pk if pk else None
        out.append(r)
        del keep
        for k, v in saved.items():
            dg.gemm_set_option(dg.Option[k], v)
    return out


if __name__ == "__main__":
    main()
