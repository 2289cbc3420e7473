#!/usr/bin/env python
"""Throughput of the block-scaled FP4 quantisation path and of the NVFP4 GEMM
on one B300 (or N, one process per GPU, each with its own copy of the work).

Step (the unit the timed loop repeats): the activation-like 8192 x 4096 BF16
tensor (Student-t nu = 3 times a per-column lognormal scale) quantised three
ways -- E2M1/NVFP4 without the RHT, E2M1/NVFP4 with the 16-point RHT, uniform
E1M2/UFP4 with the RHT -- 16-element blocks, RTNE, row-wise, statistics fused;
then the UFP4 copy dequantised with the inverse RHT back to BF16 (UFP4 has no
tensor-core format: a consumer dequantises it). Each quantisation is the two
passes of the method through the C ABI -- fp4q_amax (the tensor amax), then
fp4q_quantize with FP4Q_AMAX_READY (block scales, codes, statistics) -- which
is exactly what fp4q_quantize launches at this size, split so that each pass
is timed on its own.

  value   algorithmic bytes of the step / step time, GB/s (whole job: all ranks)
  e2e     the same bytes / the time of the same step through the Python binding
          with the input in pinned host memory and every output copied back
  gemm    quantise-then-GEMM at 8192^3 (A, B N(0, 1/8192) BF16 -> NVFP4 with the
          RHT along K -> tcgen05 block-scaled GEMM -> BF16 Y), GEMM TFLOP/s
  roofline   of the kernel that takes most of the step's time
  cpu_baseline  the CPU oracle, as it stands, on a bounded sample of the step

L2: the 64 MiB input fits the 126 MB L2, so a 256 MiB buffer is written between
timed steps (outside the timed events); the GEMM leg's BF16 inputs (128 MiB
each) exceed L2.

--impl reference times the CPU oracle on the same step (a bounded sample per
step) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import re
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

METRIC = "quantize GB/s & % HBM peak; NVFP4 GEMM TFLOPS & % FP4 peak (1×B300)"
ROWS, COLS = 8192, 4096
SEED = 1234
# (format, rht) of the three quantisations of the step
WAYS = [("nvfp4", False), ("nvfp4", True), ("ufp4", True)]
GEMM_N = 8192
FP4_OVER_BF16 = 13.5 / 2.25        # nominal dense FP4 / BF16 tensor rate
L2_FLUSH_BYTES = 256 << 20

# algorithmic bytes per element (BF16 input): the amax pass reads 2; the
# quantisation pass reads 2 and writes 0.5 of codes + 1/16 of E4M3 scales; the
# dequantise pass reads 0.5 + 1/16 and writes 2.
B_AMAX = 2.0
B_QUANT = 2.0 + 0.5 + 1.0 / 16
B_DEQ = 0.5 + 1.0 / 16 + 2.0
STEP_BYTES_PER_EL = len(WAYS) * (B_AMAX + B_QUANT) + B_DEQ


def step_bytes(rows: int, cols: int) -> float:
    return STEP_BYTES_PER_EL * rows * cols


def workload_config(extra=None) -> dict:
    cfg = {"workload": "activation 8192x4096 BF16 (Student-t nu=3 x per-column lognormal), "
                       "quantised E2M1 / E2M1+RHT16 / UFP4+RHT16, 16-element blocks, RTNE, "
                       "row-wise, fused stats; UFP4 copy dequantised (inverse RHT) to BF16",
           "shape": [ROWS, COLS], "input_dtype": "bf16", "seed": SEED,
           "l2": "256 MiB buffer written between timed steps (input 64 MiB < L2)",
           "parallelism": "replicas (one independent workload per GPU)"}
    if extra:
        cfg.update(extra)
    return cfg


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true",
                   help="skip the CPU oracle leg (profiling runs)")
    p.add_argument("--no-gemm", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--sweep", action="store_true",
                   help="instead of the step: the size sweep (R x 4096 BF16 N(0,1), R = 2^8..2^18), "
                        "MXFP4 vs NVFP4 quantisation GB/s per size, one JSON line per size")
    p.add_argument("--sweep-max-rows", type=int, default=1 << 18)
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    if a.steps < 1:
        p.error("--steps must be >= 1")
    return a


# --------------------------------------------------------------------------- #
# distributed plumbing (barrier + max over ranks; no data-path collective)     #
# --------------------------------------------------------------------------- #

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float, device) -> float:
    """Max of a scalar over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def whole_job(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job throughput: the units every rank processed / the slowest rank's time."""
    return units_per_rank * world / seconds_max if seconds_max > 0 else float("nan")


# --------------------------------------------------------------------------- #
# clocks during the timed region                                              #
# --------------------------------------------------------------------------- #

_REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi samples (200 ms) of the SM clock and throttle reasons of one GPU."""

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.err = None
        if gpu_id is None:
            self.err = "no GPU id"
            return
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.err = f"nvidia-smi unavailable: {e}"

    def stop(self) -> dict | None:
        if self.proc is None:
            return {"error": self.err}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_lines(out.splitlines())


def parse_clock_lines(lines) -> dict:
    sm, smax, power = [], [], []
    seen = set()
    for ln in lines:
        f = [x.strip() for x in ln.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            smax.append(float(f[2]))
            power.append(float(f[3]))
        except ValueError:
            continue
        for name, val in zip(_REASONS, f[5:9]):
            if val.lower() == "active":
                seen.add(name)
    if not sm:
        return {"error": "no samples"}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
            "power_w_max": max(power), "reasons": sorted(seen)}


def gpu_uuid(device) -> str | None:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[device.index] if vis else str(device.index)


# --------------------------------------------------------------------------- #
# peaks, traffic counters                                                      #
# --------------------------------------------------------------------------- #

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", 0.0)),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


#: the source file that defines each kernel; its digest also covers the shared headers
KERNEL_SOURCES = {
    "amax_rows_kernel": "fp4q_rows.cu", "quant_rows_kernel": "fp4q_rows.cu", "dequant_rows_kernel": "fp4q_rows.cu",
    "amax_tiles_kernel": "fp4q_rows.cu", "quant_tiles_kernel": "fp4q_rows.cu",
    "quant_cols_outer_kernel": "fp4q_rows.cu", "gemm_nvf4_kernel": "fp4q_gemm.cu",
    "gemm_nvf4_pair_kernel": "fp4q_gemm.cu", "gemm_dq_kernel": "fp4q_gemm_dq.cu",
    "gemm_dq_kernel<3>": "fp4q_gemm_dq.cu",
    "gemm_outer_kernel": "fp4q_gemm_outer.cu", "code_hist_kernel": "fp4q_hist.cu",
}


def source_digest(kernel: str) -> str:
    """Digest of the source a kernel is built from: its .cu file and every
    header it includes, directly or through other headers (quoted includes,
    resolved beside the including file). ncu counters apply only to the build
    they came from."""
    csrc = os.path.join(ROOT, "fp4_block_scaled_05_b300", "csrc")
    src = KERNEL_SOURCES.get(kernel)
    if not src:
        return ""
    files, todo = {}, [os.path.normpath(os.path.join(csrc, src))]
    while todo:
        path = todo.pop()
        if path in files:
            continue
        if not os.path.isfile(path):
            return ""
        with open(path, "rb") as f:
            files[path] = f.read()
        for inc in re.findall(rb'#include "([^"]+)"', files[path]):
            todo.append(os.path.normpath(os.path.join(os.path.dirname(path), inc.decode())))
    h = hashlib.sha1()
    for path in sorted(files):
        h.update(os.path.relpath(path, csrc).encode() + b"\0" + files[path])
    return h.hexdigest()[:12]


def ncu_traffic(kernel: str, units: float) -> float | None:
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    summary, scaled by the elements (or FLOP) a launch processes here; None if
    the counters were taken on other sources of that kernel."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    k = t.get("kernels", {}).get(kernel)
    if not k or k.get("source_digest") != source_digest(kernel):
        return None
    return float(k["dram_bytes"]) * units / float(k["units"])


# --------------------------------------------------------------------------- #
# the CPU oracle leg                                                           #
# --------------------------------------------------------------------------- #

def oracle_step(bits, seed: int = SEED) -> dict:
    """One step of the path on the CPU oracle, one thread (test infrastructure;
    used only for the baseline timing)."""
    from oracle import fp4q_oracle as o
    out = {}
    for fmt, rht in WAYS:
        out[(fmt, rht)] = o.quantize(bits, fmt, rht=rht, seed=seed)["row"]
    u = out[("ufp4", True)]
    o.dequantize(u["codes"], u["scales"], u["tensor_scale"], "ufp4", True, seed)
    return out


# ---- the oracle on every host core: a process pool over row ranges -------------
# Each worker holds the whole input; a step runs, per way, pass 1 (the copy's
# amax) over row ranges in parallel, then pass 2 (scales, codes, statistics;
# for the UFP4 way also the dequantisation of those rows) over the same ranges
# with the tensor amax of pass 1. The arithmetic is the oracle's, unchanged.

_POOL_M32 = None
_POOL_SHM = None


def _pool_init(shm_name, shape):
    import os as _os
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        _os.environ[var] = "1"
    import numpy as np
    from multiprocessing import shared_memory
    global _POOL_M32, _POOL_SHM
    _POOL_SHM = shared_memory.SharedMemory(name=shm_name)
    _POOL_M32 = np.ndarray(shape, dtype=np.float32, buffer=_POOL_SHM.buf)


def _pool_amax(task):
    from oracle import fp4q_oracle as o
    fmt, rht, seed, r0, r1 = task
    return float(o.copy_amax(_POOL_M32[r0:r1], fmt, rht, seed))


def _pool_quant(task):
    import numpy as np
    from oracle import fp4q_oracle as o
    fmt, rht, seed, r0, r1, amax, dequant = task
    q = o.quantize_copy(_POOL_M32, fmt, rht, "rtne", seed, 0, rows_subset=np.arange(r0, r1),
                        amax=np.float32(amax))
    if dequant:
        o.dequantize(q["codes"], q["scales"], q["tensor_scale"], fmt, True, seed)
    st = q["stats"]
    return st["shrink_bias"] * st["n"], st["sum_sig2"], st["sum_err2"]


def _row_ranges(rows: int, parts: int):
    step = max(16, -(-rows // parts) // 16 * 16)
    return [(r0, min(rows, r0 + step)) for r0 in range(0, rows, step)]


def oracle_step_parallel(pool, rows: int, parts: int, seed: int = SEED) -> None:
    ranges = _row_ranges(rows, parts)
    for fmt, rht in WAYS:
        amax = max(pool.map(_pool_amax, [(fmt, rht, seed, r0, r1) for r0, r1 in ranges]))
        pool.map(_pool_quant, [(fmt, rht, seed, r0, r1, amax, fmt == "ufp4") for r0, r1 in ranges])


def host_description() -> dict:
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


class OraclePool:
    """A spawn-started pool of one worker per host core (up to 256). The first
    `rows` rows of the activation tensor, widened to FP32 once by the oracle,
    sit in shared memory that every worker maps."""

    def __init__(self, rows: int):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        import numpy as np
        import synth
        from oracle import fp4q_oracle as o
        m32 = o._as_f32_matrix(synth.bf16_bits(synth.activation(ROWS, COLS)[:rows]))
        self.shm = shared_memory.SharedMemory(create=True, size=m32.nbytes)
        np.ndarray(m32.shape, dtype=np.float32, buffer=self.shm.buf)[...] = m32
        self.n = min(os.cpu_count() or 1, 256)
        self.pool = mp.get_context("spawn").Pool(self.n, initializer=_pool_init,
                                                 initargs=(self.shm.name, m32.shape))

    def close(self):
        self.pool.close()
        self.pool.join()
        self.shm.close()
        self.shm.unlink()


def time_oracle(rows: int, reps: int = 1) -> dict:
    """CPU seconds and wall seconds of `reps` one-thread oracle steps on the
    first `rows` rows of the activation tensor."""
    import synth
    x = synth.activation(ROWS, COLS)[:rows]
    bits = synth.bf16_bits(x)
    oracle_step(bits[:16])                       # imports, first-touch
    c0, w0 = time.process_time(), time.perf_counter()
    for _ in range(reps):
        oracle_step(bits)
    wall = time.perf_counter() - w0
    cpu = time.process_time() - c0
    return {"wall": wall, "cpu": cpu, "cores": max(1, round(cpu / wall)) if wall > 0 else 1}


def cpu_baseline(single_rows: int = 2048) -> dict:
    """The oracle on the host: one thread on the first `single_rows` rows, and
    every core (a spawn-started process pool over row ranges) on the whole
    8192 x 4096 step. `value` is the all-cores figure."""
    t1 = time_oracle(single_rows)
    one = step_bytes(single_rows, COLS) / t1["wall"] / 1e9
    op = OraclePool(ROWS)
    n = op.n
    try:
        oracle_step_parallel(op.pool, 64, n)         # workers started, imports done
        w0 = time.perf_counter()
        oracle_step_parallel(op.pool, ROWS, n)
        wall = time.perf_counter() - w0
    finally:
        op.close()
    allc = step_bytes(ROWS, COLS) / wall / 1e9
    return {"value": allc, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"one whole step (8192 x 4096, three ways + UFP4 dequantisation) on {n} worker "
                      f"processes over row ranges (pass 1 amax, then pass 2 with the tensor amax), "
                      f"{wall:.2f} s wall, numpy",
            "single_core": {"value": one, "unit": "GB/s", "cores": 1,
                            "sample": f"one step on the first {single_rows} of {ROWS} rows "
                                      f"(tensor amax over the sample), {t1['wall']:.2f} s wall"},
            "host": host_description()}


def reference_arm(args) -> int:
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # each step is a bounded sample of rows on every host core, sized so the
    # whole run stays near two minutes
    op = OraclePool(ROWS)
    n, pool = op.n, op.pool
    try:
        oracle_step_parallel(pool, 64, n)
        w0 = time.perf_counter()
        oracle_step_parallel(pool, min(ROWS, 16 * n), n)
        per_row = (time.perf_counter() - w0) / min(ROWS, 16 * n)
        budget = 120.0 / (args.steps + args.warmup)
        rows = int(max(16, min(ROWS, budget / per_row)) // 16 * 16)
        for _ in range(args.warmup):
            oracle_step_parallel(pool, rows, n)
        w0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_step_parallel(pool, rows, n)
        wall = time.perf_counter() - w0
    finally:
        op.close()
    value = step_bytes(rows, COLS) * args.steps / wall / 1e9
    sample = (f"each step on the first {rows} of {ROWS} rows ({rows * COLS} elements; tensor amax over "
              f"the sample), {n} worker processes over row ranges, numpy")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config({"sample_rows": rows}),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle",
                             "sample": sample, "host": host_description()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- #
# the GPU legs                                                                 #
# --------------------------------------------------------------------------- #

class RawCalls:
    """Pre-marshalled C-ABI calls for the timed loop (the same entry points the
    binding wraps, without per-call Python bookkeeping)."""

    def __init__(self, fq, x, outs, deq_out, ws, stream: int):
        import ctypes
        self.fq = fq
        self.lib = fq._lib
        self.ws = ws
        self.stream = stream
        self.x = x
        rows, cols = x.shape
        self.calls = []
        for (fmt, rht), q in zip(WAYS, outs):
            s = q.c_struct()
            self.calls.append((
                (x.data_ptr(), 0, rows, cols, fq.FORMATS[fmt], fq.BLOCKS[fmt], int(rht), SEED, 1,
                 ws.data_ptr(), ws.numel(), stream),
                (x.data_ptr(), 0, rows, cols, fq.FORMATS[fmt], fq.BLOCKS[fmt], int(rht), 0, SEED,
                 1 | 4, ctypes.byref(s), None, ws.data_ptr(), ws.numel(), stream),
                s))
        u = outs[-1]
        self.deq_struct = u.c_struct()
        self.deq_args = (ctypes.byref(self.deq_struct), rows, cols, fq.FORMATS["ufp4"], 16, 1, SEED,
                         deq_out.data_ptr(), 0, stream)

    def amax(self, i):
        rc = self.lib.fp4q_amax(*self.calls[i][0])
        if rc:
            raise self.fq.FP4QError("fp4q_amax", rc)

    def quant(self, i):
        rc = self.lib.fp4q_quantize(*self.calls[i][1])
        if rc:
            raise self.fq.FP4QError("fp4q_quantize", rc)

    def deq(self):
        rc = self.lib.fp4q_dequantize(*self.deq_args)
        if rc:
            raise self.fq.FP4QError("fp4q_dequantize", rc)


def run_main_leg(fq, torch, device, steps, warmup):
    import synth
    x = synth.activation(ROWS, COLS).to(device)
    outs = [fq.alloc_copy(ROWS, COLS, fmt, "linear", device) for fmt, _ in WAYS]
    deq_out = torch.empty(ROWS, COLS, dtype=torch.bfloat16, device=device)
    ws = fq.workspace(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    raw = RawCalls(fq, x, outs, deq_out, ws, stream.cuda_stream)
    x_ref = x.clone()

    def one_step(ev):
        # ev: [start, end] for a throughput step, or one event after every
        # launch for the per-kernel breakdown
        ev[0].record(stream)
        per_kernel = len(ev) > 2
        for i in range(len(WAYS)):
            raw.amax(i)
            if per_kernel:
                ev[2 * i + 1].record(stream)
            raw.quant(i)
            if per_kernel:
                ev[2 * i + 2].record(stream)
        raw.deq()
        ev[-1].record(stream)

    nev = 2 * len(WAYS) + 2
    for _ in range(warmup):
        flush.zero_()
        one_step([torch.cuda.Event(enable_timing=True) for _ in range(nev)])
        flush.zero_()
        one_step([torch.cuda.Event(enable_timing=True) for _ in range(2)])
    torch.cuda.synchronize(device)
    if fq.fp4q_status(ws) != 0:
        raise RuntimeError("device status set during warm-up")

    # Throughput: K steps with events only at the step boundaries, so that each
    # launch's prologue may overlap the previous launch's tail (programmatic
    # dependent launch), as in a user's back-to-back calls.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(device)
    torch.cuda.synchronize(device)
    w0 = time.perf_counter()
    for k in range(steps):
        flush.zero_()                    # L2 flush, outside the step's events
        one_step(evs[k])
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - w0
    barrier(device)
    step_ms = [ev[0].elapsed_time(ev[1]) for ev in evs]

    # Per-kernel breakdown: the same K steps with an event after every launch.
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(steps)]
    barrier(device)
    torch.cuda.synchronize(device)
    for k in range(steps):
        flush.zero_()
        one_step(kev[k])
    torch.cuda.synchronize(device)
    barrier(device)
    amax_ms, quant_ms, deq_ms, kstep_ms = [], [], [], []
    for ev in kev:
        kstep_ms.append(ev[0].elapsed_time(ev[nev - 1]))
        for i in range(len(WAYS)):
            amax_ms.append(ev[2 * i].elapsed_time(ev[2 * i + 1]))
            quant_ms.append(ev[2 * i + 1].elapsed_time(ev[2 * i + 2]))
        deq_ms.append(ev[nev - 2].elapsed_time(ev[nev - 1]))
    status = fq.fp4q_status(ws)
    # self-checks outside the timed region: the input is intact, and the
    # statistics of a repeated quantisation are identical (no state leaks
    # from one call into the next)
    checks = {"input_unchanged": bool(torch.equal(x, x_ref))}
    stats, repeat_same = {}, True
    for (fmt, rht), q in zip(WAYS, outs):
        seen = []
        for _ in range(2):
            fq.fp4q_quantize(x, fmt=fmt, rht=rht, seed=SEED, axis="row", ws=ws, row_out=q)
            rs, _ = fq.fp4q_stats(ws)
            seen.append((rs["shrink_bias"], rs["snr_db"]))
        repeat_same &= seen[0] == seen[1]
        stats[f"{fmt}{'+rht' if rht else ''}"] = {"shrink_bias": seen[0][0], "snr_db": seen[0][1]}
    checks["stats_repeatable"] = bool(repeat_same)
    return {"step_ms_total": sum(step_ms), "wall_s": wall, "amax_ms": amax_ms,
            "quant_ms": quant_ms, "deq_ms": deq_ms, "instrumented_step_ms": statistics.mean(kstep_ms),
            "status": status, "stats": stats, "checks": checks, "launches_per_step": 2 * len(WAYS) + 1}


def run_e2e_leg(fq, torch, device, steps, warmup):
    """The step through the public binding with host buffers: pinned BF16 input
    copied in, every output (codes, scales, tensor scales, statistics, the
    dequantised tensor) copied back, inside the timed region."""
    import synth
    x_host = synth.activation(ROWS, COLS).pin_memory()
    x = torch.empty(ROWS, COLS, dtype=torch.bfloat16, device=device)
    outs = [fq.alloc_copy(ROWS, COLS, fmt, "linear", device) for fmt, _ in WAYS]
    hosts = [(torch.empty_like(q.codes, device="cpu").pin_memory(),
              torch.empty_like(q.scales, device="cpu").pin_memory(),
              torch.empty_like(q.tensor_scale, device="cpu").pin_memory()) for q in outs]
    deq = torch.empty(ROWS, COLS, dtype=torch.bfloat16, device=device)
    deq_host = torch.empty(ROWS, COLS, dtype=torch.bfloat16).pin_memory()
    ws = fq.workspace(device)
    stream = torch.cuda.current_stream(device)
    h2d = x_host.numel() * 2
    d2h = sum(c.numel() + s.numel() + 4 for c, s, _ in hosts) + deq_host.numel() * 2
    stats_bytes = len(WAYS) * (2 * 5 * 8 + 4)     # fp4q_stats reads the sums + copy mask
    d2h += stats_bytes

    def one_step():
        x.copy_(x_host, non_blocking=True)
        for (fmt, rht), q, (hc, hs, ht) in zip(WAYS, outs, hosts):
            fq.fp4q_quantize(x, fmt=fmt, rht=rht, seed=SEED, axis="row", ws=ws, row_out=q)
            fq.fp4q_stats(ws)
            hc.copy_(q.codes, non_blocking=True)
            hs.copy_(q.scales, non_blocking=True)
            ht.copy_(q.tensor_scale, non_blocking=True)
        fq.fp4q_dequantize(outs[-1], inverse_rht=True, seed=SEED, out=deq)
        deq_host.copy_(deq, non_blocking=True)

    for _ in range(warmup):
        one_step()
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(steps):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    return {"ms": e0.elapsed_time(e1), "h2d": h2d, "d2h": d2h}


def run_gemm_leg(fq, torch, device, steps, warmup):
    """Quantise-then-GEMM at 8192^3: A, B N(0, 1/8192) BF16 -> NVFP4 (RHT along
    K, tensor-core scale layout) -> Y = A B^T in BF16."""
    import synth
    n = GEMM_N
    a = synth.gemm_operand("a", n, n).to(device)
    b = synth.gemm_operand("b", n, n).to(device)
    qa = fq.alloc_copy(n, n, "nvfp4", "mma", device)
    qb = fq.alloc_copy(n, n, "nvfp4", "mma", device)
    y = torch.empty(n, n, dtype=torch.bfloat16, device=device)
    ws = fq.workspace(device)
    stream = torch.cuda.current_stream(device)

    def one(ev):
        ev[0].record(stream)
        for src, q in ((a, qa), (b, qb)):
            fq.fp4q_quantize(src, fmt="nvfp4", rht=True, seed=SEED, axis="row", layout="mma",
                             ws=ws, row_out=q)
        ev[1].record(stream)
        fq.fp4q_gemm(qa, qb, out=y, ws=ws)
        ev[2].record(stream)

    for _ in range(warmup):
        one([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize(device)
    if fq.fp4q_status(ws) != 0:
        raise RuntimeError("device status set during the GEMM warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(device)
    torch.cuda.synchronize(device)
    for k in range(steps):
        one(evs[k])
    torch.cuda.synchronize(device)
    barrier(device)
    q_ms = [e[0].elapsed_time(e[1]) for e in evs]
    g_ms = [e[1].elapsed_time(e[2]) for e in evs]
    status = fq.fp4q_status(ws)
    # SNR of Y against the BF16-input product on a sample of rows (FP64 on the device)
    rows = torch.arange(0, n, 64, device=device)
    ref = a[rows].double() @ b.double().T
    got = y[rows].double()
    snr = 10 * math.log10(float((ref * ref).sum()) / float(((got - ref) ** 2).sum()))
    return {"quant_ms": q_ms, "gemm_ms": g_ms, "status": status, "snr_db_vs_bf16": snr}


def run_gemm_ufp4_leg(fq, torch, device, steps, warmup, peaks, fmt="ufp4"):
    """UFP4 on the contraction at 8192^3 (the pages' proposal: the uniform grid
    with the RHT on every GEMM): A, B N(0, 1/8192) BF16 -> UFP4 + RHT16 along
    K, then fp4q_gemm, which runs UFP4 on the 16-bit tensor-core MMA: converter
    warps form the exact FP16 block values level * s_b in shared memory, the
    tensor cores accumulate in FP32, the epilogue applies g_A g_B. Time per
    GEMM call; the roofline is the dense FP16/BF16 tensor peak. fmt="hif4"
    runs HiF4 operands the same way (exact BF16 block values, a scale per
    4-element micro-block)."""
    import synth
    n = GEMM_N
    a = synth.gemm_operand("a", n, n).to(device)
    b = synth.gemm_operand("b", n, n).to(device)
    layout = "linear" if fmt == "hif4" else "mma"
    qa, _ = fq.fp4q_quantize(a, fmt=fmt, rht=True, seed=SEED, layout=layout)
    qb, _ = fq.fp4q_quantize(b, fmt=fmt, rht=True, seed=SEED, layout=layout)
    y = torch.empty(n, n, dtype=torch.bfloat16, device=device)
    ws = fq.workspace(device)
    stream = torch.cuda.current_stream(device)
    evs = []
    for k in range(warmup + steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fq.fp4q_gemm(qa, qb, out=y, ws=ws)
        e1.record(stream)
        if k >= warmup:
            evs.append((e0, e1))
    torch.cuda.synchronize(device)
    us = statistics.fmean(x.elapsed_time(z) for x, z in evs) * 1e3
    status = fq.fp4q_status(ws)
    flop = 2.0 * n ** 3
    rows = torch.arange(0, n, 64, device=device)
    ref = a[rows].double() @ b.double().T
    got = y[rows].double()
    snr = 10 * math.log10(float((ref * ref).sum()) / float(((got - ref) ** 2).sum()))
    tflops = flop / (us * 1e-6) / 1e12
    peak = peaks["bf16_tflops"]
    kind = "FP16" if fmt == "ufp4" else "BF16"
    return {"workload": f"A, B 8192x8192 BF16 N(0,1/8192) -> {fmt.upper()} + RHT16 along K -> fp4q_gemm: exact "
                        f"{kind} block values formed in shared memory, tcgen05 kind::f16 MMA (FP32 accumulate) x "
                        "g_A g_B, BF16 Y = A B^T",
            "us": us, "tflops": tflops, "launches": len(evs), "device_status": status,
            "snr_db_vs_bf16_product": snr,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak,
                         "peak_source": f"{peaks['source']} bf16 burst (the dense FP16 rate is the same)",
                         "traffic": ncu_traffic("gemm_dq_kernel" if fmt == "ufp4" else "gemm_dq_kernel<3>", flop)}}


def sweep_point(fq, torch, device, x, steps, warmup, peaks, ws, flush) -> dict:
    """One size of the sweep: MXFP4 (32-element E8M0 blocks, one pass) and
    NVFP4 (16-element E4M3 blocks, amax pass + quantisation pass) on the R x
    4096 tensor x, RTNE, no RHT, row-wise: median time per call and GB/s of
    algorithmic bytes, L2 flushed before each call. NVFP4 is timed as the
    two-call split (fp4q_amax, then fp4q_quantize with the amax ready) and as
    one fp4q_quantize call."""
    stream = torch.cuda.current_stream(device)
    rows, cols = x.shape
    n = rows * cols
    out = {}
    for fmt in ("mxfp4", "nvfp4"):
        q = fq.alloc_copy(rows, cols, fmt, "linear", device)
        times = {"amax": [], "quant": [], "one": []}
        for k in range(warmup + steps):
            flush.zero_()
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            fq.fp4q_amax(x, fmt=fmt, ws=ws)
            e1.record(stream)
            fq.fp4q_quantize(x, fmt=fmt, ws=ws, row_out=q, amax_ready=True)
            e2.record(stream)
            flush.zero_()
            e3, e4 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            e3.record(stream)
            fq.fp4q_quantize(x, fmt=fmt, ws=ws, row_out=q)
            e4.record(stream)
            if k >= warmup:
                times["amax"].append((e0, e1))
                times["quant"].append((e1, e2))
                times["one"].append((e3, e4))
        torch.cuda.synchronize(device)
        t_one = statistics.median(a.elapsed_time(b) for a, b in times["one"])
        t_a = statistics.median(a.elapsed_time(b) for a, b in times["amax"]) if fmt == "nvfp4" else 0.0
        t_q = statistics.median(a.elapsed_time(b) for a, b in times["quant"])
        b_q = (2.0 + 0.5 + (1.0 / 16 if fmt == "nvfp4" else 1.0 / 32)) * n
        b_a = 2.0 * n if fmt == "nvfp4" else 0.0
        out[fmt] = {"call_us": (t_a + t_q) * 1e3, "call_GB/s": (b_a + b_q) / ((t_a + t_q) / 1e3) / 1e9,
                    "quant_us": t_q * 1e3, "quant_GB/s": b_q / (t_q / 1e3) / 1e9,
                    "quant_frac_hbm": b_q / (t_q / 1e3) / 1e9 / peaks["hbm_gbs"],
                    "quant_bytes_per_element": b_q / n}
        if fmt == "nvfp4":
            out[fmt].update({"amax_us": t_a * 1e3, "amax_GB/s": b_a / (t_a / 1e3) / 1e9,
                             "amax_frac_hbm": b_a / (t_a / 1e3) / 1e9 / peaks["hbm_gbs"],
                             "one_launch_us": t_one * 1e3,
                             "one_launch_GB/s": (b_a + b_q) / (t_one / 1e3) / 1e9,
                             "call_frac_hbm": (b_a + b_q) / ((t_a + t_q) / 1e3) / 1e9 / peaks["hbm_gbs"]})
        else:
            out[fmt]["launches"] = 3 * (warmup + steps)
        del q
    return out


def run_sweep(fq, torch, device, args, peaks) -> None:
    """The size sweep: R x 4096 N(0,1) BF16, R = 2^8 .. 2^18, one JSON line
    per size (sweep_point)."""
    import synth
    cols = 4096
    ws = fq.workspace(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    rows_list = [r for r in synth.sweep_rows() if r <= args.sweep_max_rows]
    x_full = synth.sweep(max(rows_list), cols).to(device)
    for rows in rows_list:
        out = sweep_point(fq, torch, device, x_full[:rows], args.steps, args.warmup, peaks, ws, flush)
        print(json.dumps({"sweep": "R x 4096 BF16 N(0,1), RTNE, no RHT, row-wise", "rows": rows,
                          "elements": rows * cols, **out}), flush=True)
    assert fq.fp4q_status(ws) == 0


def run_sweep_largest_leg(fq, torch, device, steps, warmup, peaks) -> dict:
    """The sweep's largest point (262144 x 4096 = 2^30 elements, 2 GiB of BF16:
    far above L2), as the default run's keyed entry, with a roofline for each
    pass."""
    import synth
    rows = synth.sweep_rows()[-1]
    x = synth.sweep(rows, 4096).to(device)
    ws = fq.workspace(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    out = sweep_point(fq, torch, device, x, steps, warmup, peaks, ws, flush)
    status = fq.fp4q_status(ws)
    del x
    torch.cuda.empty_cache()
    n = rows * 4096
    peak = peaks["hbm_gbs"]

    def roof(gbs, ncu_name):
        return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                "peak_source": f"{peaks['source']} (copy bandwidth)", "traffic": ncu_traffic(ncu_name, n)}

    return {"workload": f"size sweep, largest point: {rows} x 4096 BF16 N(0,1) ({n} elements), RTNE, no RHT, "
                        "row-wise; MXFP4 (32-element E8M0, one pass) vs NVFP4 (16-element E4M3, amax pass + "
                        "quantisation pass); median per call, L2 flushed before each",
            **out, "device_status": status,
            "roofline": {"mxfp4_quantize": roof(out["mxfp4"]["quant_GB/s"], "quant_rows_kernel"),
                         "nvfp4_amax": roof(out["nvfp4"]["amax_GB/s"], "amax_rows_kernel"),
                         "nvfp4_quantize": roof(out["nvfp4"]["quant_GB/s"], "quant_rows_kernel")}}


def run_grad_leg(fq, torch, device, steps, warmup):
    """The gradient-like workload: 4096 x 14336 and 14336 x 4096 BF16, N(0, 1e-6)
    with 0.1% x100 outliers, NVFP4 with the 16-point RHT and Philox stochastic
    rounding (seed 1234), row-wise and column-wise (transposed) copies from one
    read: time per fp4q_quantize call."""
    import synth
    out = {}
    for which in ("a", "b"):
        x = synth.gradient(which).to(device)
        rows, cols = x.shape
        r = fq.alloc_copy(rows, cols, "nvfp4", "linear", device)
        c = fq.alloc_copy(cols, rows, "nvfp4", "linear", device)
        ws = fq.workspace(device)
        stream = torch.cuda.current_stream(device)
        evs = []
        for k in range(warmup + steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fq.fp4q_quantize(x, fmt="nvfp4", rht=True, rounding="sr", seed=SEED, axis="both", ws=ws,
                             row_out=r, col_out=c)
            e1.record(stream)
            if k >= warmup:
                evs.append((e0, e1))
        torch.cuda.synchronize(device)
        us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
        n = rows * cols
        byts = (B_AMAX + 2.0 + 2 * (0.5 + 1.0 / 16)) * n
        out[f"{rows}x{cols}"] = {"us": us, "GB/s": byts / (us * 1e-6) / 1e9,
                                 "status": fq.fp4q_status(ws)}
    return out


def run_two_level_leg(fq, torch, device, steps, warmup, peaks):
    """Two-level NVFP4 (double-block scale: FP32 scale per 128-element outer
    block, E4M3 per 16-element inner block; one pass, no tensor amax) on the
    activation tensor with the 16-point RHT, RTNE, row-wise, against the
    two-pass NVFP4 + RHT call on the same tensor: time per fp4q_quantize call
    (L2 flushed before each)."""
    import synth
    x = synth.activation(ROWS, COLS).to(device)
    ws = fq.workspace(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    n = ROWS * COLS
    out = {}
    for fmt, byts in (("nvfp4_2l", (2.0 + 0.5 + 1.0 / 16 + 4.0 / 128) * n), ("nvfp4", (B_AMAX + B_QUANT) * n)):
        q = fq.alloc_copy(ROWS, COLS, fmt, "linear", device)
        evs = []
        for k in range(warmup + steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fq.fp4q_quantize(x, fmt=fmt, rht=True, seed=SEED, ws=ws, row_out=q)
            e1.record(stream)
            if k >= warmup:
                evs.append((e0, e1))
        torch.cuda.synchronize(device)
        us = statistics.fmean(a.elapsed_time(b) for a, b in evs) * 1e3
        gbs = byts / (us * 1e-6) / 1e9
        out[fmt + "+rht"] = {"us": us, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
                             "bytes_per_element": byts / n, "launches": len(evs) * (1 if fmt == "nvfp4_2l" else 2),
                             "status": fq.fp4q_status(ws)}
    return out


def run_mx_leg(fq, torch, device, steps, warmup, peaks):
    """The E8M0 formats of the MXFP4 page (Resume technique §2, §2A-§2B) on the
    activation tensor, RTNE, no RHT, row-wise: MXFP4 on 32- and on 16-element
    blocks, the overflow-aware rule (OAS), the static macro-block scale (MBS),
    and HiF4 from the HiFloat page (E6M2 per 64, halving bits per 8 and 4),
    beside NVFP4: time per fp4q_quantize call (L2 flushed before each) and the
    SNR of each copy. Then the block-scaled GEMM at 8192^3 on the tensor cores
    with E8M0 scales (MXFP4 32-element blocks, OAS on 16-element blocks) and
    with per-128 FP32 scales along K (two-level NVFP4, MBS: a TMEM product per
    128-element chunk, scaled in the epilogue), operands quantised with the
    RHT along K."""
    import synth
    x = synth.activation(ROWS, COLS).to(device)
    ws = fq.workspace(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    n = ROWS * COLS
    quant = {}
    for fmt, bpe, launches in (("mxfp4", 2.5 + 1.0 / 32, 1), ("mxfp4_b16", 2.5 + 1.0 / 16, 1),
                               ("mxfp4_oas", 2.5 + 1.0 / 16, 1), ("mxfp4_mbs", 2.5 + 1.0 / 16 + 4.0 / 128, 1),
                               ("hif4", 2.5 + 4.0 / 64, 1), ("nvfp4", B_AMAX + B_QUANT, 2)):
        q = fq.alloc_copy(ROWS, COLS, fmt, "linear", device)
        fq.fp4q_quantize(x, fmt=fmt, ws=ws, row_out=q)
        st, _ = fq.fp4q_stats(ws)
        evs = []
        for k in range(warmup + steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fq.fp4q_quantize(x, fmt=fmt, ws=ws, row_out=q)
            e1.record(stream)
            if k >= warmup:
                evs.append((e0, e1))
        torch.cuda.synchronize(device)
        us = statistics.fmean(a.elapsed_time(b) for a, b in evs) * 1e3
        gbs = bpe * n / (us * 1e-6) / 1e9
        quant[fmt] = {"us": us, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "bytes_per_element": bpe,
                      "snr_db": st["snr_db"], "shrink_bias": st["shrink_bias"], "launches": len(evs) * launches,
                      "status": fq.fp4q_status(ws)}
    gemm = {}
    m = GEMM_N
    a = synth.gemm_operand("a", m, m).to(device)
    b = synth.gemm_operand("b", m, m).to(device)
    y = torch.empty(m, m, dtype=torch.bfloat16, device=device)
    rows = torch.arange(0, m, 64, device=device)
    ref = a[rows].double() @ b.double().T
    for fmt in ("mxfp4", "mxfp4_oas", "nvfp4_2l", "mxfp4_mbs"):
        qa, _ = fq.fp4q_quantize(a, fmt=fmt, rht=True, seed=SEED, layout="mma", ws=ws)
        qb, _ = fq.fp4q_quantize(b, fmt=fmt, rht=True, seed=SEED, layout="mma", ws=ws)
        evs = []
        for k in range(warmup + min(steps, 100)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fq.fp4q_gemm(qa, qb, out=y, ws=ws)
            e1.record(stream)
            if k >= warmup:
                evs.append((e0, e1))
        torch.cuda.synchronize(device)
        us = statistics.fmean(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3
        tflops = 2.0 * m ** 3 / (us * 1e-6) / 1e12
        got = y[rows].double()
        snr = 10 * math.log10(float((ref * ref).sum()) / float(((got - ref) ** 2).sum()))
        gemm[fmt] = {"us": us, "tflops": tflops, "frac_of_fp4_peak": tflops / (peaks["bf16_tflops"] * FP4_OVER_BF16),
                     "snr_db_vs_bf16_product": snr, "launches": len(evs), "status": fq.fp4q_status(ws)}
    return {"quantize": quant, "gemm_8192": gemm}


def run_histogram_leg(fq, torch, device, steps, warmup, peaks):
    """Code utilisation of the activation's three quantised copies ([UFP4]
    Resultados: the RHT raises the effective bucket ratio): the histogram
    kernel's time over the E2M1 + RHT copy (0.5 B/element read) and the
    effective bucket ratio of each way."""
    import synth
    x = synth.activation(ROWS, COLS).to(device)
    ws = fq.workspace(device)
    stream = torch.cuda.current_stream(device)
    ratios, copies = {}, {}
    for fmt, rht in WAYS:
        q = fq.alloc_copy(ROWS, COLS, fmt, "linear", device)
        fq.fp4q_quantize(x, fmt=fmt, rht=rht, seed=SEED, ws=ws, row_out=q)
        name = f"{fmt}{'+rht' if rht else ''}"
        ratios[name] = fq.fp4q_effective_bucket_ratio(fq.fp4q_code_histogram(q))
        copies[name] = q
    q = copies["nvfp4+rht"]
    counts = torch.empty(16, dtype=torch.int64, device=device)
    evs = []
    for k in range(warmup + steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fq.fp4q_code_histogram(q, out=counts)
        e1.record(stream)
        if k >= warmup:
            evs.append((e0, e1))
    torch.cuda.synchronize(device)
    us = statistics.fmean(a.elapsed_time(b) for a, b in evs) * 1e3
    gbs = 0.5 * ROWS * COLS / (us * 1e-6) / 1e9
    return {"us": us, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "launches": len(evs),
            "effective_bucket_ratio": ratios}


def main(argv=None) -> int:
    args = parse_args(argv)
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    import fp4_block_scaled_05_b300 as fq     # fails loudly when libfp4q.so is missing

    peaks = load_peaks()
    if args.sweep:
        run_sweep(fq, torch, device, args, peaks)
        return 0
    sampler = ClockSampler(gpu_uuid(device))
    main_r = run_main_leg(fq, torch, device, args.steps, args.warmup)
    gemm_r = None if args.no_gemm else run_gemm_leg(fq, torch, device, args.steps, args.warmup)
    gemm_u = None if args.no_gemm else run_gemm_ufp4_leg(fq, torch, device, min(args.steps, 50), args.warmup,
                                                         peaks)
    gemm_h = None if args.no_gemm else run_gemm_ufp4_leg(fq, torch, device, min(args.steps, 50), args.warmup,
                                                         peaks, fmt="hif4")
    grad_r = run_grad_leg(fq, torch, device, min(args.steps, 50), args.warmup)
    tl_r = run_two_level_leg(fq, torch, device, min(args.steps, 200), args.warmup, peaks)
    hist_r = run_histogram_leg(fq, torch, device, min(args.steps, 200), args.warmup, peaks)
    mx_r = run_mx_leg(fq, torch, device, min(args.steps, 200), args.warmup, peaks)
    sweep_r = run_sweep_largest_leg(fq, torch, device, min(args.steps, 20), args.warmup, peaks)
    e2e_steps = min(args.steps, 100)
    e2e_r = None if args.no_e2e else run_e2e_leg(fq, torch, device, e2e_steps, args.warmup)
    clocks = sampler.stop()

    n_el = ROWS * COLS
    t_step = reduce_max(main_r["step_ms_total"] / 1e3, device)
    value = whole_job(step_bytes(ROWS, COLS) * args.steps, t_step, world) / 1e9
    ms_per_step = t_step / args.steps * 1e3

    # per-kernel averages over the instrumented pass of the timed steps
    kern = {
        "amax": {"ms": statistics.fmean(main_r["amax_ms"]), "bytes": B_AMAX * n_el,
                 "launches": len(main_r["amax_ms"]), "ncu_name": "amax_rows_kernel"},
        "quantize": {"ms": statistics.fmean(main_r["quant_ms"]), "bytes": B_QUANT * n_el,
                     "launches": len(main_r["quant_ms"]), "ncu_name": "quant_rows_kernel"},
        "dequantize": {"ms": statistics.fmean(main_r["deq_ms"]), "bytes": B_DEQ * n_el,
                       "launches": len(main_r["deq_ms"]), "ncu_name": "dequant_rows_kernel"},
    }
    for k in kern.values():
        k["gbs"] = k["bytes"] / (k["ms"] / 1e3) / 1e9
        k["frac"] = k["gbs"] / peaks["hbm_gbs"]
        k["total_ms"] = k["ms"] * k["launches"]
    dom_name = max(kern, key=lambda n: kern[n]["total_ms"])
    dom = kern[dom_name]
    roofline = {"kernel": dom_name, "bound": "hbm", "achieved": dom["gbs"],
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": dom["frac"],
                "peak_source": f"{peaks['source']} (copy bandwidth)",
                "traffic": ncu_traffic(dom["ncu_name"], n_el),
                "algorithmic_bytes_per_launch": dom["bytes"]}

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(),
            "roofline": roofline,
            "kernels": {n: {"avg_us": k["ms"] * 1e3, "GB/s": k["gbs"], "frac_hbm": k["frac"],
                            "launches": k["launches"]} for n, k in kern.items()},
            "kernel_timing": "value and ms_per_step: K steps with events at step boundaries only; per-kernel "
                             "avg_us (and the roofline): the same K steps again with an event after every "
                             "launch, whose step takes instrumented_ms_per_step",
            "instrumented_ms_per_step": main_r["instrumented_step_ms"],
            "gpu_launches": main_r["launches_per_step"] * args.steps,
            "stats": main_r["stats"], "device_status": main_r["status"],
            "self_check": main_r["checks"],
            "wall_s_timed_region": main_r["wall_s"]}

    if e2e_r is not None:
        t_e2e = reduce_max(e2e_r["ms"] / 1e3, device)
        line["e2e"] = {"value": whole_job(step_bytes(ROWS, COLS) * e2e_steps, t_e2e, world) / 1e9,
                       "unit": "GB/s", "h2d_bytes_per_step": e2e_r["h2d"],
                       "d2h_bytes_per_step": e2e_r["d2h"], "steps": e2e_steps}
    if gemm_r is not None:
        flop = 2.0 * GEMM_N ** 3
        g_avg = statistics.fmean(gemm_r["gemm_ms"])
        g_max = reduce_max(sum(gemm_r["gemm_ms"]) / 1e3, device)
        tflops = flop / (g_avg / 1e3) / 1e12
        fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
        q_avg = statistics.fmean(gemm_r["quant_ms"])
        line["gemm"] = {
            "workload": "A, B 8192x8192 BF16 N(0,1/8192) -> NVFP4 + RHT16 along K (E4M3 block "
                        "scales, FP32 tensor scale) -> tcgen05 block-scaled GEMM, FP32 "
                        "accumulate, BF16 Y = A B^T",
            "tflops": tflops, "whole_job_tflops": whole_job(flop * args.steps, g_max, world) / 1e12,
            "avg_us": g_avg * 1e3, "launches": len(gemm_r["gemm_ms"]),
            "quantize_A_and_B_us": q_avg * 1e3,
            "quantize_A_and_B_GB/s": 2 * (B_AMAX + B_QUANT) * GEMM_N * GEMM_N / (q_avg / 1e3) / 1e9,
            "pipeline_tflops": flop / ((g_avg + q_avg) / 1e3) / 1e12,
            "snr_db_vs_bf16_product": gemm_r["snr_db_vs_bf16"],
            "device_status": gemm_r["status"],
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": fp4_peak,
                         "unit": "TFLOP/s", "frac": tflops / fp4_peak,
                         "peak_source": f"{peaks['source']} bf16 burst x {FP4_OVER_BF16:g} "
                                        "(nominal dense FP4/BF16 ratio)",
                         "traffic": ncu_traffic("gemm_nvf4_pair_kernel", flop)},
        }
        line["gpu_launches_gemm_leg"] = 3 * args.steps
        line["gemm_ufp4"] = gemm_u
        line["gemm_hif4"] = gemm_h
    line["gradient_leg"] = {
        "workload": "4096x14336 and 14336x4096 BF16 N(0,1e-6) with 0.1% x100, NVFP4 + RHT16 + Philox "
                    "SR (seed 1234), row-wise and column-wise copies from one read",
        "bytes_per_element": B_AMAX + 2.0 + 2 * (0.5 + 1.0 / 16), **grad_r}
    line["two_level_leg"] = {
        "workload": "activation 8192x4096 BF16, RHT16, RTNE, row-wise: two-level NVFP4 (FP32 scale per "
                    "128-element outer block, E4M3 per 16; one pass) vs NVFP4 with a tensor scale (amax "
                    "pass + quantisation pass), time per fp4q_quantize call, L2 flushed before each",
        **tl_r}
    line["code_histogram"] = {
        "workload": "16-code histogram of the activation's E2M1 + RHT copy (16.8 MB of codes); effective "
                    "bucket ratio exp(H)/8 of each way's copy", **hist_r}
    line["mx_formats_leg"] = {
        "workload": "activation 8192x4096 BF16, RTNE, no RHT, row-wise: MXFP4 (32-element E8M0 blocks), MXFP4 "
                    "on 16-element blocks, OAS (16, E8M0), MBS-static (16, E8M0, 8-bit-mantissa scale per "
                    "128), HiF4 (E6M2 per 64, halving bits per 8 and per 4, levels 0..7), NVFP4; time per "
                    "fp4q_quantize call, L2 flushed before each, and each copy's SNR. "
                    "GEMM 8192^3 on the tensor cores with E8M0 scales (MXFP4, OAS) and with per-128 FP32 "
                    "scales along K (two-level NVFP4, MBS); operands + RHT16 along K",
        **mx_r}
    line["sweep_largest"] = sweep_r
    line["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
