#!/usr/bin/env python
"""Benchmark of the fp16 -> fp32 product Out = A @ B.T on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one call of the library on one synthetic problem (the whole hot
path: TMA staging, tcgen05 MMAs into TMEM, epilogue to HBM).  The default
workload is the 8192^3 product (fp16 normal(0,1), seed 2).  Rank 0 prints one
JSON line.

  value      TFLOP/s with A, B resident in HBM, CUDA events on the launching
             stream, max over ranks, whole-job aggregate (N replicas: weak scaling)
  e2e        the same metric through gemm_nt_f16_f32_from_host: pinned host
             A, B -> device, product, Out -> pinned host, every step
  roofline   the dominant kernel against the measured peak (MEASURED_PEAKS.json)
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload
  hot        (workloads that fit in L2) the same steps back to back, no flush
  context_cublas  cuBLAS (torch.mm / torch.bmm, fp32 Out where torch offers it)
             on the same operands, timed the same way after the timed region
  --impl reference  times that oracle alone (the reference arm of this bench)

Inputs of the default workload (512 MiB touched per step) exceed the 129 MB L2,
so no L2 flush is needed between steps.  Workloads of 16 MiB to 2x L2 rotate
over enough copies of their operands and Out (more than 3x L2 in all) that each
copy has left L2 before it is used again, and run back to back; smaller ones
flush L2 by writing a 256 MiB buffer between timed steps (the flush's dirty
lines then drain to DRAM during the next step, which the rotation avoids).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "TFLOP/s fp16→fp32 Out=A·Bᵀ at 8192³; % of dense fp16 peak / HBM roofline"
L2_BYTES = 129 * 1024 * 1024
# element widths of the 6- and 4-bit floats, stored packed along K
PACKED_BITS = {"e2m3": 6, "e3m2": 6, "e2m1": 4}

# DRAM traffic per launch of the dominant kernel from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload, with the
# sha256 of the kernel source it was taken on; reported as null once the kernel
# source no longer matches.
TRAFFIC = {
    "square_8192": (1074521600 + 248043520, "dfb399817f9f0705"),
    "square_4096": (91492352 + 34789888, "dfb399817f9f0705"),
    "ragged_batch16_3001x2047x1000": (162286592 + 332889344, "dfb399817f9f0705"),
    "skinny_64x16384x8192": (269563136 + 2948352, "1c2d3c01ce774de5"),
    # block-scaled E4M3 and E2M1 inputs (--ab-dtype e4m3 / e2m1 --mx), packed E2M1 (--ab-dtype e2m1)
    "square_8192/mx-e4m3": (358762240 + 234705152, "dfb399817f9f0705"),
    "square_8192/mx-e2m1": (171194624 + 217513216, "dfb399817f9f0705"),
    "square_8192/e2m1": (156736768 + 216092416, "dfb399817f9f0705"),
    # the weight-stationary shape on the skinny product (--path TC05_WS)
    "skinny_64x16384x8192/TC05_WS": (278262528 + 5557504, "0de165ee5081595b"),
}


_PAIR_SRC = ["tc05_pair.cu", "tc05_common.cuh", "ptx.cuh", "ptx_mx.cuh"]
_ONE_SRC = ["tc05_gemm.cu", "tc05_kernel.cuh", "tc05_common.cuh", "ptx.cuh", "ptx_mx.cuh"]
_SMALL_SRC = ["tc05_small.cu", "tc05_kernel.cuh", "tc05_common.cuh", "ptx.cuh", "ptx_mx.cuh"]
KERNEL_SOURCES = {
    "square_8192": _PAIR_SRC,
    "square_4096": _PAIR_SRC,
    "ragged_batch16_3001x2047x1000": _PAIR_SRC,
    "skinny_64x16384x8192": _ONE_SRC,
    "tile_128x64x64": _ONE_SRC,
}


def traffic_key(workload, ab="f16", out="f32", mx=False, path="AUTO"):
    """TRAFFIC key of a run: the workload, then its element types when not
    fp16 -> fp32 (with "mx-" for block scales), then an explicit path."""
    key = workload
    if mx:
        key += "/mx-" + ab
    elif ab != "f16" or out != "f32":
        key += "/" + ab + ("" if out == "f32" else "->" + out)
    if mx and out != "f32":
        key += "->" + out
    return key + ("" if path == "AUTO" else "/" + path)


def kernel_source_sha(workload, path="AUTO"):
    """sha256 prefix of the sources of the kernel that dominates `workload`
    (on an explicit path of the other instruction shapes, that kernel's)."""
    h = hashlib.sha256()
    for name in (_SMALL_SRC if path in ("TC05_M64", "TC05_WS") else KERNEL_SOURCES[workload]):
        with open(os.path.join(ROOT, "dense_fp16_tensor_gemm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "tflops": d["bf16_tflops"],
                "tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "tflops": 1900.0, "tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle samples every 100 ms while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = bus_id
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.bus_id:
            cmd += ["--id=" + self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file if ln.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 7:
                continue
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, r[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        top = max(sm)
        loaded = [s for s in sm if s >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x, world, device="cpu"):
    """Largest value of x over all ranks (the job is as slow as its slowest rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank, world, ms_per_step):
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def oracle_cpu_sample(w, A, B, target_s, dtype="f16", scales=None):
    """Time the CPU oracle on whole rows of the workload (batch 0), sized to
    about target_s seconds; `scales` (SA, SB) selects the block-scaled oracle.
    Returns (tflops, seconds, rows, threads)."""
    import oracle
    A0 = A if A.ndim == 2 else A[0]
    B0 = B if B.ndim == 2 else B[0]
    if scales is None:
        def run(rows):
            oracle.gemm_nt(A0[:rows], B0, dtype=dtype)
    else:
        SA0 = scales[0] if scales[0].ndim == 2 else scales[0][0]
        SB0 = scales[1] if scales[1].ndim == 2 else scales[1][0]

        def run(rows):
            oracle.gemm_nt_mx(A0[:rows], SA0[:rows], B0, SB0, dtype=dtype)
    probe = min(8, A0.shape[0])
    run(1)  # thread pool start-up
    t0 = time.perf_counter()
    run(probe)
    per_row = max(time.perf_counter() - t0, 1e-4) / probe
    rows = int(max(1, min(A0.shape[0], target_s / per_row)))
    t0 = time.perf_counter()
    run(rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * B0.shape[0] * A0.shape[1]
    return flops / dt / 1e12, dt, rows, oracle.max_threads()


def run_reference(args, w):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    world, rank, _ = dist_init()
    if rank != 0:
        return 0
    A, B = workloads.workload_inputs(w.name, args.ab_dtype)
    scales = workloads.workload_mx_scales(w.name) if args.mx else None
    per_step = max(1.0, args.cpu_seconds / 5)
    vals = []
    rows_used = None
    for i in range(args.warmup + args.steps):
        tf, dt, rows, threads = oracle_cpu_sample(w, A, B, per_step, args.ab_dtype, scales)
        if i >= args.warmup:
            vals.append((tf, dt))
            rows_used = rows
    tf = statistics.median(v[0] for v in vals)
    ms = statistics.median(v[1] for v in vals) * 1e3
    sample = ("%d full rows of batch 0 (%d x %d outputs, K=%d) per step"
              % (rows_used, rows_used, w.N, w.K))
    line = {
        "impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, None, args.ab_dtype, args.out_dtype, mx=args.mx),
        "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_policy(alg_bytes):
    """(rotate, flush, n_sets) for a workload of alg_bytes per step: inputs larger
    than 2 x L2 run back to back; 16 MiB to 2 x L2 rotate over copies that fill
    more than 3 x L2; smaller ones flush L2 between timed steps."""
    import math
    rotate = 16 * 2 ** 20 <= alg_bytes <= 2 * L2_BYTES
    flush = alg_bytes <= 2 * L2_BYTES and not rotate
    n_sets = 1 + int(math.ceil(3 * L2_BYTES / alg_bytes)) if rotate else 1
    return rotate, flush, n_sets


def roofline_of(flops, alg_bytes, kernel_ms, peaks):
    """The bound (tensor or HBM) by arithmetic intensity against the measured
    peaks, and the achieved fraction of it."""
    tensor_bound = flops / alg_bytes * peaks["hbm_gbs"] * 1e9 > peaks["tflops"] * 1e12
    if tensor_bound:
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peaks["tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["tflops"]}
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"]}


def time_workload(gnt, torch, w, steps, warmup, stream, bus, peaks):
    """Device time of one fp16 -> fp32 workload on the automatic path, as the
    headline line times its own (inputs resident in HBM, the same L2 policy,
    CUDA events on the launching stream, clocks sampled meanwhile)."""
    A, B = workloads.workload_inputs(w.name)
    a = torch.from_numpy(A.view("int16")).view(torch.float16).cuda()
    b = torch.from_numpy(B.view("int16")).view(torch.float16).cuda()
    batched = A.ndim == 3
    out = torch.empty((w.batch, w.M, w.N) if batched else (w.M, w.N), dtype=torch.float32, device="cuda")
    nb = w.batch if batched else 1
    sA, sB, sO = (w.M * w.K, w.N * w.K, w.M * w.N) if batched else (0, 0, 0)
    rotate, flush, n_sets = l2_policy(w.bytes)
    sets = [(a, b, out)] + [(a.clone(), b.clone(), torch.empty_like(out)) for _ in range(n_sets - 1)]
    sh = stream.cuda_stream
    cur = [0]

    def step():
        x, y, o = sets[cur[0]]
        cur[0] = (cur[0] + 1) % n_sets
        gnt.gemm_nt_f16_f32_batched_path(x.data_ptr(), y.data_ptr(), o.data_ptr(), w.M, w.N, w.K, w.K, w.K, w.N,
                                         sA, sB, sO, nb, gnt.Path.AUTO, sh)

    scratch = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device="cuda") if flush else None
    sampler = ClockSampler(bus)
    sampler.start()
    # warm-up right before the timed region, so that it starts on a busy GPU
    for _ in range(warmup):
        step()
    gnt.gemm_nt_check(sh)
    n_ev = steps if flush else 1
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
    torch.cuda.synchronize()
    if flush:
        for i in range(steps):
            scratch.fill_(float(i))
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
    else:
        ev[0][0].record(stream)
        for _ in range(steps):
            step()
        ev[0][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    gnt.gemm_nt_check(sh)
    ms = sum(s.elapsed_time(e) for s, e in ev) / steps
    roof = roofline_of(w.flops, w.bytes, ms, peaks)
    # DRAM bytes per launch from an ncu capture, while the kernel's sources match it
    tr = TRAFFIC.get(traffic_key(w.name))
    roof["traffic"] = tr[0] if tr and w.name in KERNEL_SOURCES and tr[1] == kernel_source_sha(w.name) else None
    rec = {"value": w.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
           "roofline": roof, "gbs_algorithmic": w.bytes / (ms * 1e-3) / 1e9, "clocks": clocks,
           "gpu_launches": steps, "path": gnt.gemm_nt_select_path(a.data_ptr(), b.data_ptr(), out.data_ptr(), w.M,
                                                                   w.N, w.K, w.K, w.K, w.N, sA, sB, sO, nb).name,
           "l2": workload_config(w, flush, n_sets=n_sets)["l2"]}
    if w.name == "skinny_64x16384x8192":
        rec["hbm_frac_of_8tbs"] = rec["gbs_algorithmic"] / 8000.0
    if w.name == "tile_128x64x64":
        rec["note"] = "one 128x64x64 tile: launch-bound, time reported"
    del sets, a, b, out, scratch
    torch.cuda.empty_cache()
    return rec


def steady_state(gnt, torch, step, flops, seconds, ms_hint, stream, bus, peaks):
    """The same step back to back for about `seconds` (long enough for the board
    to reach its power cap): TFLOP/s over the whole run, against the measured
    sustained peak."""
    n = max(10, int(seconds * 1e3 / max(ms_hint, 1e-3)))
    sampler = ClockSampler(bus)
    sampler.start()
    for _ in range(3):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    gnt.gemm_nt_check(stream.cuda_stream)
    ms = e0.elapsed_time(e1) / n
    value = flops / (ms * 1e-3) / 1e12
    peak = peaks.get("tflops_sustained") or peaks["tflops"]
    return {"value": value, "unit": "TFLOP/s", "ms_per_step": ms, "steps": n, "seconds": ms * n * 1e-3,
            "frac_of_sustained_peak": value / peak, "sustained_peak": peak, "frac_of_burst_peak": value / peaks["tflops"],
            "clocks": clocks, "gpu_launches": n, "l2": "inputs larger than L2, steps back to back"}


def workload_config(w, flush, ab="f16", out="f32", alg_bytes=None, a_major="K", b_major="K", mx=False, n_sets=1):
    cfg = {"workload": "%s: %s; Out = A @ B.T, A (%s%d,%d) and B (%s%d,%d) %s row-major, "
                       "fp32 accumulate, %s Out" % (
                           w.name, w.description, "%d," % w.batch if w.batch > 1 else "", w.M, w.K,
                           "%d," % w.batch if w.batch > 1 else "", w.N, w.K, ab, out),
           "batch": w.batch, "M": w.M, "N": w.N, "K": w.K, "seed": w.seed, "ab_dtype": ab,
           "out_dtype": out}
    if a_major != "K" or b_major != "K":
        cfg["a_major"], cfg["b_major"] = a_major, b_major
        cfg["workload"] += "; A stored %s, B stored %s" % (
            "(K,M) row-major" if a_major == "MN" else "(M,K) row-major",
            "(K,N) row-major" if b_major == "MN" else "(N,K) row-major")
    alg_bytes = alg_bytes or w.bytes
    if flush is not None:
        if n_sets > 1:
            cfg["l2"] = ("operands and Out rotate over %d copies (%.0f MiB each, %.0f MiB in all > 3 x 129 MB L2): "
                         "each copy has left L2 before its next use; steps back to back, no flush"
                         % (n_sets, alg_bytes / 2 ** 20, n_sets * alg_bytes / 2 ** 20))
        else:
            cfg["l2"] = ("inputs larger than L2 (%.0f MiB per step > 129 MB L2), no flush" % (alg_bytes / 2 ** 20)
                         if not flush else "L2 flushed between timed steps (256 MiB write)")
    if mx:
        cfg["block_scales"] = ("one E8M0 scale per 32 K elements of each row of A and B, uniform 2^-7..2^7 "
                               "(seed + 7), packed into the atom layout once before timing")
    return cfg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="square_8192", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--path", default="AUTO")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0)
    ap.add_argument("--no-cublas", action="store_true", help="skip the cuBLAS context timing")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other four workloads (the default 8192^3 run times them too)")
    ap.add_argument("--steady-seconds", type=float, default=3.0,
                    help="back-to-back run of the default workload after the timed region, for the "
                         "power-capped figure (0: skip)")
    ap.add_argument("--a-major", default="K", choices=["K", "MN"],
                    help="MN: A handed to the library as its transpose, (K, M) row-major")
    ap.add_argument("--b-major", default="K", choices=["K", "MN"],
                    help="MN: B handed to the library as its transpose, (K, N) row-major (the NN product)")
    ap.add_argument("--ab-dtype", default="f16", choices=["f16", "bf16", "e4m3", "e5m2", "e2m3", "e3m2", "e2m1"],
                    help="element type of A and B (bf16, e4m3, e5m2: the same draws rounded to that type; "
                         "e2m3, e3m2, e2m1: rounded to that grid and stored packed along K)")
    ap.add_argument("--out-dtype", default="f32", choices=["f32", "f16", "bf16"],
                    help="element type of Out (16-bit: fp32 accumulator rounded to nearest even)")
    ap.add_argument("--mx", action="store_true",
                    help="block-scaled 8-bit product (needs --ab-dtype e4m3 or e5m2): one E8M0 scale per 32 K "
                         "elements of each row, drawn uniformly from 2^-7..2^7 and packed once before timing")
    args = ap.parse_args()
    if args.mx and args.ab_dtype not in ("e4m3", "e5m2", "e2m3", "e3m2", "e2m1"):
        ap.error("--mx needs an 8-, 6- or 4-bit --ab-dtype")
    if args.ab_dtype in PACKED_BITS and (args.a_major != "K" or args.b_major != "K"):
        ap.error("packed 6- and 4-bit operands are K-major")
    if args.mx and (args.a_major != "K" or args.b_major != "K"):
        ap.error("--mx takes K-major operands only")
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    import numpy as np
    import torch
    import torch.distributed as dist

    import dense_fp16_tensor_gemm_gb300 as gnt

    world, rank, local = dist_init()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    gnt.load()
    path = gnt.Path[args.path]
    default_types = args.ab_dtype == "f16" and args.out_dtype == "f32"
    a_mn, b_mn = args.a_major == "MN", args.b_major == "MN"
    default_layout = not a_mn and not b_mn
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
           "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
    codes = {"f16": gnt.DType.F16, "bf16": gnt.DType.BF16, "f32": gnt.DType.F32,
             "e4m3": gnt.DType.E4M3, "e5m2": gnt.DType.E5M2, "e2m3": gnt.DType.E2M3,
             "e3m2": gnt.DType.E3M2, "e2m1": gnt.DType.E2M1}
    packed = args.ab_dtype in PACKED_BITS
    # the 8-bit MMA kind (8-, 6- and 4-bit elements)
    f8 = args.ab_dtype in ("e4m3", "e5m2") or packed
    ab_es = PACKED_BITS[args.ab_dtype] / 8 if packed else (1 if f8 else 2)
    raw = np.uint8 if f8 else np.int16
    A, B = workloads.workload_inputs(w.name, args.ab_dtype)
    batched = A.ndim == 3
    # stored operands: an MN-major one is its transpose, row-major; 6- and
    # 4-bit ones packed along K
    As = np.ascontiguousarray(np.swapaxes(A, -1, -2)) if a_mn else A
    Bs = np.ascontiguousarray(np.swapaxes(B, -1, -2)) if b_mn else B
    lda, ldb = As.shape[-1], Bs.shape[-1]
    if packed:
        As, Bs = workloads.pack_subbyte(As, args.ab_dtype), workloads.pack_subbyte(Bs, args.ab_dtype)
        a, b = torch.from_numpy(As).cuda(), torch.from_numpy(Bs).cuda()
    else:
        a = torch.from_numpy(As.view(raw)).view(tdt[args.ab_dtype]).cuda()
        b = torch.from_numpy(Bs.view(raw)).view(tdt[args.ab_dtype]).cuda()
    out = torch.empty((w.batch, w.M, w.N) if batched else (w.M, w.N), dtype=tdt[args.out_dtype],
                      device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    nb = w.batch if batched else 1
    sA, sB, sO = (w.M * w.K, w.N * w.K, w.M * w.N) if batched else (0, 0, 0)
    majors = {"K": gnt.Major.K, "MN": gnt.Major.MN}

    scales = workloads.workload_mx_scales(w.name) if args.mx else None
    if args.mx:
        sa_plain = torch.from_numpy(scales[0]).cuda()
        sb_plain = torch.from_numpy(scales[1]).cuda()
        sa_packed = gnt.pack_mx_scales(sa_plain, w.K)
        sb_packed = gnt.pack_mx_scales(sb_plain, w.K)

    # algorithmic bytes: A and B (and their block scales) read once, Out written once
    alg_bytes = float(w.batch) * (ab_es * w.M * w.K + ab_es * w.N * w.K + out.element_size() * w.M * w.N)
    if args.mx:
        alg_bytes += float(w.batch) * (w.M + w.N) * ((w.K + 31) // 32)
    # cold-L2 timing: rotate over copies, or flush (see the module docstring)
    rotate = 16 * 2 ** 20 <= alg_bytes <= 2 * L2_BYTES
    flush = alg_bytes <= 2 * L2_BYTES and not rotate
    n_sets = 1 + int(np.ceil(3 * L2_BYTES / alg_bytes)) if rotate else 1
    sets = [(a, b, out, sa_packed if args.mx else None, sb_packed if args.mx else None)]
    for _ in range(n_sets - 1):
        sets.append((a.clone(), b.clone(), torch.empty_like(out), sa_packed.clone() if args.mx else None,
                     sb_packed.clone() if args.mx else None))
    cur = [0]

    def step(fixed=False):
        i = 0 if fixed else cur[0]
        if not fixed:
            cur[0] = (cur[0] + 1) % n_sets
        a, b, out, sa_packed, sb_packed = sets[i]
        if args.mx:
            gnt.gemm_nt_mx(a.data_ptr(), sa_packed.data_ptr(), b.data_ptr(), sb_packed.data_ptr(), out.data_ptr(),
                           codes[args.ab_dtype], codes[args.out_dtype], w.M, w.N, w.K, w.K, w.K, w.N, sA, sB,
                           sO, nb, path, sh)
        elif not default_layout:
            gnt.gemm_nt_batched_major(a.data_ptr(), majors[args.a_major], b.data_ptr(), majors[args.b_major],
                                      out.data_ptr(), codes[args.ab_dtype], codes[args.out_dtype], w.M, w.N, w.K,
                                      lda, ldb, w.N, sA, sB, sO, nb, path, sh)
        elif default_types:
            gnt.gemm_nt_f16_f32_batched_path(a.data_ptr(), b.data_ptr(), out.data_ptr(), w.M, w.N, w.K,
                                             w.K, w.K, w.N, sA, sB, sO, nb, path, sh)
        else:
            gnt.gemm_nt_batched_ex(a.data_ptr(), b.data_ptr(), out.data_ptr(), codes[args.ab_dtype],
                                   codes[args.out_dtype], w.M, w.N, w.K, w.K, w.K, w.N, sA, sB, sO, nb,
                                   path, sh)

    scratch = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device="cuda") if flush else None

    bus = None
    try:
        bus = torch.cuda.get_device_properties(local).pci_bus_id
    except AttributeError:
        pass
    sampler = ClockSampler(bus if isinstance(bus, str) else None)
    sampler.start()
    # warm-up right before the timed region, so that it starts on a busy GPU
    for _ in range(args.warmup):
        step()
    gnt.gemm_nt_check(sh)
    # With inputs larger than L2 the steps run back to back between one pair of
    # events (one launch of the library's kernel per step, so the mean launch
    # duration is the total over K).  Smaller inputs need an L2 flush between
    # steps, and each step is bracketed by its own events so the flush is not
    # timed.
    n_ev = args.steps if flush else 1
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    barrier()
    torch.cuda.synchronize()
    t_host = time.perf_counter()
    if flush:
        for i in range(args.steps):
            scratch.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
    else:
        starts[0].record(stream)
        for i in range(args.steps):
            step()
        ends[0].record(stream)
    host_us = (time.perf_counter() - t_host) / args.steps * 1e6
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    gnt.gemm_nt_check(sh)
    per_launch = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(per_launch)
    ms_step = max_over_ranks(total_ms / args.steps, world, "cuda")
    value = job_tflops(w.flops, world, ms_step)
    kernel_ms = total_ms / args.steps
    step_ms_median = statistics.median(per_launch) if flush else None

    def timed(fn, n):
        """Mean ms per call of fn over n calls, CUDA events on the stream;
        L2 flushed before each call when the workload fits in L2."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        if flush:
            for i in range(n):
                scratch.fill_(float(i))
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record(stream)
                fn()
                s1.record(stream)
                ts.append((s0, s1))
        else:
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(n):
                fn()
            s1.record(stream)
            ts.append((s0, s1))
        torch.cuda.synchronize()
        return sum(x.elapsed_time(y) for x, y in ts) / n

    # ---- hot-L2 figure for workloads that fit in L2 (one set of operands back to back)
    hot = None
    if flush or rotate:
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        h0.record(stream)
        for _ in range(args.steps):
            step(fixed=True)
        h1.record(stream)
        torch.cuda.synchronize()
        hot_ms = h0.elapsed_time(h1) / args.steps
        hot = {"value": w.flops / (hot_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": hot_ms,
               "l2": "inputs resident in L2 from the previous step (no flush)"}

    # ---- context: cuBLAS on the same operands, timed the same way
    cublas = None
    if not args.no_cublas:
        # the logical operands of each set: A (M, K) and B^T (K, N), views of the stored ones
        def operands(i):
            sa_, sb_ = sets[i][0], sets[i][1]
            al_ = sa_.transpose(-1, -2) if a_mn else sa_
            bt_ = sb_ if b_mn else sb_.transpose(-1, -2)
            if packed:
                # cuBLAS's 4-bit floats: two per byte, its float4_e2m1fn_x2 type (no 6-bit type)
                fp4 = getattr(torch, "float4_e2m1fn_x2", None)
                ok4 = fp4 is not None and args.ab_dtype == "e2m1"
                al_, bt_ = (al_.view(fp4), bt_.view(fp4)) if ok4 else (None, None)
            return al_, bt_
        ops = [operands(i) for i in range(n_sets)]
        al, bt = ops[0]
        ccur = [0]

        def nxt():
            i = ccur[0]
            ccur[0] = (i + 1) % n_sets
            return i
        mm = torch.bmm if batched else torch.mm
        cub_fn = None
        if packed and not (args.mx and al is not None):
            cub_fn = None  # no unscaled 6- or 4-bit product in cuBLAS
        elif args.mx:
            # cuBLAS's block-scaled path: its 128 x 4 blocked scale layout is
            # the library's atom layout
            if not batched:
                try:
                    e8 = torch.float8_e8m0fnu
                    scs = [(st[3].view(e8), st[4].view(e8)) for st in sets]
                    torch._scaled_mm(al, bt, scale_a=scs[0][0], scale_b=scs[0][1], out_dtype=torch.float32)

                    def cub_mx():
                        i = nxt()
                        return torch._scaled_mm(ops[i][0], ops[i][1], scale_a=scs[i][0], scale_b=scs[i][1],
                                                out_dtype=torch.float32)
                    cub_fn, cub_out = cub_mx, "f32"
                except (TypeError, RuntimeError, NotImplementedError, AttributeError):
                    cub_fn = None
        elif f8:
            # cuBLAS's 8-bit path: scaled matmul with unit scales (2-D only;
            # it wants the second operand column-major, which B^T of a
            # row-major B is)
            one = torch.ones((), dtype=torch.float32, device="cuda")
            if not batched and not a_mn and not b_mn:
                try:
                    torch._scaled_mm(al, bt, scale_a=one, scale_b=one, out_dtype=torch.float32)

                    def cub_f8():
                        i = nxt()
                        return torch._scaled_mm(ops[i][0], ops[i][1], scale_a=one, scale_b=one,
                                                out_dtype=torch.float32)
                    cub_fn, cub_out = cub_f8, "f32"
                except (TypeError, RuntimeError, NotImplementedError):
                    cub_fn = None
        else:
            def cub_mm32():
                i = nxt()
                return mm(ops[i][0], ops[i][1], out_dtype=torch.float32)

            def cub_mm():
                i = nxt()
                return mm(ops[i][0], ops[i][1])
            try:
                mm(al, bt, out_dtype=torch.float32)
                cub_fn, cub_out = cub_mm32, "f32"
            except (TypeError, RuntimeError, NotImplementedError):
                cub_fn, cub_out = cub_mm, args.ab_dtype
        if cub_fn is not None:
            cub_ms = timed(cub_fn, max(3, args.steps))
            cublas = {"value": w.flops / (cub_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": cub_ms,
                      "call": ("torch._scaled_mm(A, B^T, E8M0 block scales) -> f32 Out" +
                               (" (A, B float4_e2m1fn_x2)" if packed else "") if args.mx else
                               "torch._scaled_mm(A, B^T, unit scales) -> f32 Out" if f8 else
                               "torch.%s(A, B^T%s) -> %s Out" % ("bmm" if batched else "mm",
                                                                ", out_dtype=float32" if cub_out == "f32" else "",
                                                                cub_out)),
                      "ratio": (w.flops / (kernel_ms * 1e-3) / 1e12) / (w.flops / (cub_ms * 1e-3) / 1e12)}

    # ---- end to end through the host-buffer entry point
    e2e_steps = args.e2e_steps or max(3, args.steps // 4)
    if packed:
        ha, hb = torch.from_numpy(As).pin_memory(), torch.from_numpy(Bs).pin_memory()
    else:
        ha = torch.from_numpy(As.view(raw)).view(tdt[args.ab_dtype]).pin_memory()
        hb = torch.from_numpy(Bs.view(raw)).view(tdt[args.ab_dtype]).pin_memory()
    ho = torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory()

    if args.mx:
        hsa = torch.from_numpy(scales[0]).pin_memory()
        hsb = torch.from_numpy(scales[1]).pin_memory()

    def e2e_step():
        if args.mx:
            # the call a user with host data makes: plain scales in, packed on the device
            a.copy_(ha, non_blocking=True)
            b.copy_(hb, non_blocking=True)
            sa_plain.copy_(hsa, non_blocking=True)
            sb_plain.copy_(hsb, non_blocking=True)
            if packed:
                gnt.gemm_nt_packed(a, b, w.K, codes[args.ab_dtype], sa_plain, sb_plain, out=out, path=path,
                                   stream=stream)
            else:
                gnt.gemm_nt_mx_tensors(a, sa_plain, b, sb_plain, out=out, path=path, stream=stream)
            ho.copy_(out, non_blocking=True)
        elif default_types and default_layout:
            gnt.gemm_nt_f16_f32_from_host(ha.data_ptr(), hb.data_ptr(), ho.data_ptr(), a.data_ptr(),
                                          b.data_ptr(), out.data_ptr(), w.M, w.N, w.K, w.batch, sh)
        else:
            # no pipelined host entry for these types: whole copies on the stream
            a.copy_(ha, non_blocking=True)
            b.copy_(hb, non_blocking=True)
            step()
            ho.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    gnt.gemm_nt_check(sh)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, "cuda")
    e2e_val = job_tflops(w.flops, world, e2e_ms)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks = measured_peaks()
    headline = (w.name == "square_8192" and default_types and default_layout and not args.mx
                and args.path == "AUTO")
    bus_id = bus if isinstance(bus, str) else None
    # ---- the other four workloads, each timed like the headline (1 GPU)
    others = None
    if headline and world == 1 and not args.no_workloads:
        others = {}
        n_other = max(200, args.steps)
        for name in ("tile_128x64x64", "square_4096", "skinny_64x16384x8192", "ragged_batch16_3001x2047x1000"):
            others[name] = time_workload(gnt, torch, workloads.WORKLOADS[name], n_other, args.warmup, stream,
                                         bus_id, peaks)
    # ---- the headline back to back for seconds: the power-capped figure
    steady = None
    if headline and args.steady_seconds > 0:
        steady = steady_state(gnt, torch, step, w.flops, args.steady_seconds, kernel_ms, stream, bus_id, peaks)
    ai = w.flops / alg_bytes
    # the 8-bit MMA runs at twice the 16-bit rate: its peak is the measured
    # bf16 one times that nominal ratio (4.5 / 2.25 PFLOP/s dense)
    tpeak = peaks["tflops"] * (2.0 if f8 else 1.0)
    tensor_bound = ai * peaks["hbm_gbs"] * 1e9 > tpeak * 1e12
    tr = TRAFFIC.get(traffic_key(w.name, args.ab_dtype, args.out_dtype, args.mx, args.path))
    traffic = (tr[0] if default_layout and tr and tr[1] == kernel_source_sha(w.name, args.path)
               else None)
    if tensor_bound:
        achieved = w.flops / (kernel_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                "frac": achieved / tpeak, "traffic": traffic,
                "peak_source": ("%s bf16 dense burst x 2 (the nominal fp8 / bf16 ratio%s)" % (
                                    peaks["source"], "; kind::f8f6f4 runs 6- and 4-bit elements at the "
                                    "8-bit rate" if packed else "")
                                if f8 else
                                "%s bf16 dense burst (kind::f16 runs fp16 at the bf16 rate)" % peaks["source"])}
    else:
        achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": "%s HBM copy bandwidth" % peaks["source"]}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        tf, dt, rows, threads = oracle_cpu_sample(w, A, B, args.cpu_seconds, args.ab_dtype, scales)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": "%d full rows of batch 0 (%d x %d outputs, K=%d), %.1f s" % (
                   rows, rows, w.N, w.K, dt)}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.ab_dtype, "data": "synthetic",
        "config": workload_config(w, flush, args.ab_dtype, args.out_dtype, alg_bytes, args.a_major, args.b_major,
                                  args.mx, n_sets),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(As.nbytes + Bs.nbytes + (scales[0].nbytes + scales[1].nbytes
                                                                  if args.mx else 0)),
                "d2h_bytes_per_step": int(out.numel() * out.element_size())},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "block_scaled": bool(args.mx),
        "host_us_per_step": host_us,
        "path": args.path,
        "ms_per_step_median": step_ms_median,
        "hot": hot,
        "context_cublas": cublas,
        "workloads": others,
        "steady_state": steady,
        "device": {"name": torch.cuda.get_device_name(local),
                   "sms": torch.cuda.get_device_properties(local).multi_processor_count},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
