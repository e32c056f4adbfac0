#!/usr/bin/env python3
"""Benchmark of the FP32 GEMM C = A x B on GB300, one JSON line on rank 0.

Workload: M = N = K = 4096, row-major FP32, A and B uniform on [-1, 1) from the
seeds 1004 / 2004 (the compute-bound headline shape). One step = one call of
the product kernel over the whole product. Inputs are resident in HBM when the
timed region starts; the L2 cache (129 MB) is flushed by writing a 256 MB buffer
before every timed step, outside the timed interval; each step is timed with CUDA
events on the stream the kernel is launched on.

`--impl reference` times the CPU oracle (the deliberately plain C triple loop) on
a bounded row sample of the same workload on the host cores instead.

Under torchrun (WORLD_SIZE > 1) every rank runs an independent replica of the
workload on its own GPU (no collective on the data path); the time is the max
over ranks and the value counts the work of all ranks ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "FP32 GEMM TFLOP/s at 1024³/4096³ and % of GB300 FP32 roofline (1 GPU)"
UNIT = "TFLOP/s"
WORKLOAD = dict(M=4096, N=4096, K=4096, config_no=4)
L2_FLUSH_BYTES = 256 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FFMA_PROFILE = os.path.join(ROOT, "profiles", "sgemm_ffma_4096.md")
FFMA_1024_PROFILE = os.path.join(ROOT, "profiles", "sgemm_ffma_1024.md")
TF32X3_PROFILE = os.path.join(ROOT, "profiles", "gemm_tf32x3_4096.md")
BF16_PROFILE = os.path.join(ROOT, "profiles", "gemm_bf16_4096.md")
F16_PROFILE = os.path.join(ROOT, "profiles", "gemm_f16_4096.md")
F64_PROFILE = os.path.join(ROOT, "profiles", "dgemm_f64_2048.md")
# Codes of t2s_gemm_f32_plan.
PLAN_HUGE_TAIL = 5
# Tiles as BM x BN x BK (the K-block depth) of a launch over all of K: every tile but the 4-warp
# 128 x 128 and 128 x 64 ones then takes 64-deep K blocks (256 x 128 on the TMA path only).
PLAN_NAMES = {0: "128x128x32 tiles", 1: "128x128x32 tiles, compact k loop", 2: "128x64x32 tiles",
              3: "64x64x64 tiles", 4: "256x128x64 tiles",
              5: "256x128x64 tiles in whole rounds over the SMs, the rest as 64x64x64 tiles "
                 "in a second launch", 6: "128x128x64 tiles of 8 warps",
              7: "128x64x64 tiles of 8 warps", 8: "128x128x32 tiles on a persistent grid",
              9: "56x128x64 tiles of 8 warps", 10: "32x32x64 tiles",
              11: "256x128x32 tiles on a persistent grid with TMA stores of C"}

KERNEL_SOURCES = {
    "ffma": ["sgemm_ffma.cu", "t2s_device.cuh"],
    "tf32x3": ["gemm_tf32x3.cu", "tc_gemm.cuh", "t2s_device.cuh"],
    "bf16": ["gemm_16bit.cu", "tc_gemm.cuh", "t2s_device.cuh"],
    "f64": ["gemm_f64.cu"],
}


# --------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def code_only(text: str) -> str:
    """CUDA/C++ source with comments removed and whitespace collapsed: what the compiler sees,
    so that a change of comments alone keeps a profile's recorded hash valid. String and
    character literals are kept as they are (a "//" inside one is not a comment)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_hash(kind: str) -> str:
    """First 16 hex digits of the SHA-256 of the kernel's sources, comments removed."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "roofline_driven_tiling_gb300", "csrc", name),
                  encoding="utf-8") as f:
            h.update(code_only(f.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def profile_traffic(path: str, kind: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source (the summary records the source hash); else None."""
    if not os.path.exists(path):
        return None
    text = open(path, encoding="utf-8").read()
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_hash(kind):
        return None
    return float(m_bytes.group(1))


def measured_peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


# --------------------------------------------------------------------------- CPU leg
def cpu_oracle_rate(A, B, target_s: float):
    """Times the oracle on a bounded row sample of C = A x B; returns (TFLOP/s, info).

    The oracle splits rows over its OpenMP threads, so the sample is a whole number of
    rows per thread, sized from a one-row-per-thread calibration to take about target_s.
    """
    import oracle  # test infrastructure, used here only as the CPU baseline
    M, K = A.shape
    N = B.shape[1]
    nt = max(1, oracle.num_threads())
    t0 = time.perf_counter()
    oracle.sgemm_rows(A, B, 0, min(nt, M), oracle.MUL_ADD)
    per_round = max(time.perf_counter() - t0, 1e-4)
    rows = int(min(M, nt * max(1, round(target_s / per_round))))
    t0 = time.perf_counter()
    oracle.sgemm_rows(A, B, 0, rows, oracle.MUL_ADD)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    info = {"cores": nt, "rows": rows, "seconds": dt,
            "sample": "rows 0..%d of the %dx%dx%d product (%d outputs, each a %d-term FP32 "
                      "dot product, two roundings per term)" % (rows - 1, M, N, K, rows * N, K)}
    return flops / dt / 1e12, info


def cpu_oracle_configs(budget_s: float = 4.0):
    """Times the oracle (two roundings per term, all host threads) on the workload of every
    configuration of the pages' measurements: the integer pattern at 256^3 and 1024^3, the
    constants 0.5 / 0.4 at 1024^3, the ragged 1000 x 1003 x 997, 4096^3 and the roofline sweep
    shapes, all uniform on [-1, 1) but the first three. A product whose estimate (from one row
    per thread) is within budget_s runs whole, three times up to 1024^3 and once above; a
    larger one runs once on a row sample of about budget_s. Returns one record per workload."""
    import oracle  # test infrastructure, used here only as the CPU baseline
    from roofline_driven_tiling_gb300 import inputs
    nt = max(1, oracle.num_threads())
    work = [(name, M, N, K, kind, no) for name, (M, N, K, kind, no) in inputs.CONFIGS.items()]
    work += [("c5_sweep_%dx%dx%d" % shape, *shape, "uniform", 5) for shape in inputs.SWEEP]
    records = []
    for name, M, N, K, kind, no in work:
        A, B = inputs.make(kind, M, N, K, no)
        t0 = time.perf_counter()
        oracle.sgemm_rows(A, B, 0, min(nt, M), oracle.MUL_ADD)
        per_round = max(time.perf_counter() - t0, 1e-5)
        if per_round * -(-M // nt) <= budget_s:
            rows, runs = M, (3 if M * N * K <= 1024 ** 3 else 1)
        else:
            rows, runs = int(min(M, nt * max(1, round(budget_s / per_round)))), 1
        secs = []
        for _ in range(runs):
            t0 = time.perf_counter()
            oracle.sgemm_rows(A, B, 0, rows, oracle.MUL_ADD)
            secs.append(time.perf_counter() - t0)
        med = statistics.median(secs)
        records.append({"config": name, "shape": [M, N, K], "inputs": kind, "rows": rows,
                        "whole_product": rows == M, "runs": runs,
                        "seconds_mean": sum(secs) / runs, "seconds_median": med,
                        "seconds_min": min(secs), "tflops": 2.0 * rows * N * K / med / 1e12,
                        "cores": nt})
    return records


def cpu_blocked_rate(A, B, target_s: float = 4.0):
    """Times the cache-blocked multi-core CPU GEMM (a stronger CPU baseline than the oracle;
    it checks nothing) on a row block of C = A x B sized to take about target_s; returns the
    bench-line entry."""
    import cpu_baseline
    M, K = A.shape
    N = B.shape[1]
    nt = cpu_baseline.num_threads()
    rows = min(M, 256)
    t0 = time.perf_counter()
    cpu_baseline.sgemm(A[:rows], B)
    per_row = max(time.perf_counter() - t0, 1e-4) / rows
    rows = int(min(M, max(rows, target_s / per_row)))
    t0 = time.perf_counter()
    cpu_baseline.sgemm(A[:rows], B)
    dt = time.perf_counter() - t0
    return {"value": 2.0 * rows * N * K / dt / 1e12, "unit": UNIT, "cores": nt,
            "kind": "cache-blocked multi-core C (fused multiply-adds in ascending k, bit-identical "
                    "to the oracle's FMA reading; a baseline, not a checker)",
            "sample": "rows 0..%d of the %dx%dx%d product" % (rows - 1, M, N, K), "seconds": dt}


def cpu_literal_loop_1024():
    """The literal i / j / k triple loop (the oracle's two-rounding reading, one thread) at
    1024^3, to set beside the CPU time the third page reports for the same loop and size."""
    import oracle
    from roofline_driven_tiling_gb300 import inputs
    A, B = inputs.constant(1024, 1024, 1024)  # the page's A = 0.5, B = 0.4
    nt = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        C = oracle.sgemm(A, B, oracle.MUL_ADD)
        dt = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(nt)
    return {"seconds": dt, "gflops": 2.0 * 1024 ** 3 / dt / 1e9, "cores": 1,
            "c00": float(C[0, 0]),
            "workload": "C = A x B, 1024^3, A = 0.5, B = 0.4, plain C triple loop (i, j, k), "
                        "one thread; the page's own figure for this loop is about 16-17 s on an "
                        "unstated CPU"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from roofline_driven_tiling_gb300 import inputs
    import oracle
    oracle.build()
    w = WORKLOAD
    A, B = inputs.uniform_pair(w["M"], w["N"], w["K"], w["config_no"])
    # About two minutes of CPU work for the whole run, at most 4 s a step.
    budget = min(4.0, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
    per_step = float(os.environ.get("T2S_REF_STEP_SECONDS", budget))
    for _ in range(args.warmup):
        cpu_oracle_rate(A, B, min(per_step, 1.0))
    rates, infos = [], []
    for _ in range(args.steps):
        r, info = cpu_oracle_rate(A, B, per_step)
        rates.append(r)
        infos.append(info)
    value = statistics.mean(rates)
    ms = statistics.mean(i["seconds"] for i in infos) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_block(),
        "kernel": "CPU oracle (plain C triple loop, OpenMP over rows)",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": infos[0]["cores"],
                         "kind": "oracle", "sample": infos[0]["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def config_block():
    w = WORKLOAD
    return {"workload": "sgemm %dx%dx%d fp32 row-major, A,B uniform[-1,1) seeds %d/%d"
                        % (w["M"], w["N"], w["K"], 1000 + w["config_no"], 2000 + w["config_no"]),
            "M": w["M"], "N": w["N"], "K": w["K"], "layout": "row-major dense",
            "l2": "flushed (256 MB write) before every timed step"}


# --------------------------------------------------------------------------- GPU leg
def time_steps(fn, steps, warmup, stream, flush_buf):
    """Runs fn() warmup times, then `steps` timed times with an L2 flush before each;
    returns per-step milliseconds measured by CUDA events on `stream`."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(stream):
        for s, e in ev:
            flush_buf.add_(1)  # 256 MB read + write: evicts A, B and C from L2
            s.record(stream)
            fn()
            e.record(stream)
    torch.cuda.synchronize()
    barrier()
    return [s.elapsed_time(e) for s, e in ev]


def measure_probes(lib, dev, stream):
    """Measured ceilings from the library's throughput probes (the best of 5 launches, each
    timed alone with CUDA events on `stream`): the FP32 FMA pipe at the product kernels' 8
    warps per SM, and the TF32 tensor pipe (tcgen05.mma kind::tf32, M 128, N 256)."""
    import torch
    from roofline_driven_tiling_gb300 import binding
    out = torch.empty(binding.t2s_probe_outputs(), dtype=torch.float32, device=dev)
    sp = stream.cuda_stream
    res = {}
    for kind, iters in (("fp32_fma", 1 << 17), ("tf32_mma", 1 << 14)):
        binding.probe(kind, iters, out.data_ptr(), sp)
        best = 0.0
        for _ in range(5):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            flops = binding.probe(kind, iters, out.data_ptr(), sp)
            e.record(stream)
            torch.cuda.synchronize()
            best = max(best, flops / (s.elapsed_time(e) * 1e-3) / 1e12)
        res[kind + "_tflops"] = best
    if binding.t2s_device_status(sp) != binding.T2S_OK:
        raise RuntimeError("device status reports a timed-out wait in a probe")
    return res


def extra_store_probe(dev, stream):
    """The store path's ceiling: t2s_probe_store_f32 writes a 16384 x 16384 FP32 matrix (the
    1.07 GB C of the 16384^2 x 32 product, above L2) with no arithmetic in the short-K product's
    store pattern, through TMA boxes (mode 0) and with 16-byte stores from registers (mode 1);
    the best of 5 launches each."""
    import torch
    from roofline_driven_tiling_gb300 import binding
    M = N = 16384
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    sp = stream.cuda_stream
    res = {"matrix": "%d x %d FP32 (%d MB)" % (M, N, 4 * M * N // 10**6), "call": "t2s_probe_store_f32",
           "unit": "GB/s"}
    for mode, key in ((0, "tma_boxes_gbs"), (1, "plain_stores_gbs")):
        binding.probe_store(M, N, C.data_ptr(), mode, 1.0, sp)
        best = 0.0
        for _ in range(5):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            nbytes = binding.probe_store(M, N, C.data_ptr(), mode, 1.0, sp)
            e.record(stream)
            torch.cuda.synchronize()
            best = max(best, nbytes / (s.elapsed_time(e) * 1e-3) / 1e9)
        res[key] = best
    del C
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from roofline_driven_tiling_gb300 import binding, inputs
    from roofline_driven_tiling_gb300 import roofline as rl

    w = WORKLOAD
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.uniform_pair(M, N, K, w["config_no"])
    dA = torch.from_numpy(A).to(dev)
    dB = torch.from_numpy(B).to(dev)
    dC = torch.empty((M, N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev).zero_()
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    lib = binding.lib()

    def step():
        rc = lib.t2s_gemm_f32(M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sp)
        if rc != 0:
            raise binding.T2SError(rc, "t2s_gemm_f32")

    flops = rl.gemm_flops(M, N, K)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    plan = binding.t2s_gemm_f32_plan(M, N, K, sms)
    launches_per_call = 2 if plan == PLAN_HUGE_TAIL else 1
    from roofline_driven_tiling_gb300.clocks import ClockSampler

    with ClockSampler(torch.cuda.current_device()) as clk:
        times = time_steps(step, args.steps, max(args.warmup, 3), stream, flush)
    clocks = clk.summary()
    if binding.t2s_device_status(sp) != binding.T2S_OK:
        raise RuntimeError("device status reports a timed-out wait")
    t_total = reduce_max(sum(times) / 1e3, device=dev if ws > 1 else None)
    ms_per_step = t_total / args.steps * 1e3
    value = flops * args.steps * ws / t_total / 1e12
    avg_launch_s = sum(times) / len(times) / 1e3

    peaks = measured_peaks()
    bw = float(peaks.get("hbm_gbs", 6800.0))
    fp32_peak = rl.fp32_peak_tflops()
    achieved = flops / avg_launch_s / 1e12
    roof = {"bound": "alu", "achieved": achieved, "peak": fp32_peak, "unit": UNIT,
            "frac": achieved / fp32_peak, "launches_per_call": launches_per_call,
            "traffic": profile_traffic(FFMA_PROFILE, "ffma"),
            "peak_basis": "152 SMs x 128 FP32 lanes x 2 FLOP x 2070 MHz (unit counts and max clock)",
            "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes_per_launch": rl.gemm_bytes(M, N, K),
            "ai_algorithmic": rl.gemm_ai(M, N, K),
            "ridge_ai": rl.ridge_ai(fp32_peak, bw / 1e3),
            "hbm_gbs_measured": bw}
    probes = measure_probes(lib, dev, stream)
    roof["peak_ffma_probe"] = probes["fp32_fma_tflops"]
    roof["frac_ffma_probe"] = achieved / probes["fp32_fma_tflops"]
    roof["peak_ffma_probe_basis"] = ("t2s_probe_fp32_fma: fma.rn.f32x2 chains only, 8 warps per "
                                     "SM, best of 5 launches (measured, burst)")
    if clocks and clocks.get("sm_mhz"):
        at_clock = rl.fp32_peak_tflops(mhz=clocks["sm_mhz"])
        roof["peak_at_observed_clock"] = at_clock
        roof["frac_at_observed_clock"] = achieved / at_clock

    # ---- end to end through the public host-memory entry point: pinned host buffers in,
    # copies overlapped with the product inside the call, result back in host memory.
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()

    def e2e_step():
        rc = lib.t2s_gemm_f32_host(M, N, K, hA.data_ptr(), hB.data_ptr(), hC.data_ptr(),
                                   dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sp)
        if rc != 0:
            raise binding.T2SError(rc, "t2s_gemm_f32_host")

    e2e_times = time_steps(e2e_step, max(1, min(args.steps, 10)), 2, stream, flush)
    e2e_t = reduce_max(sum(e2e_times) / 1e3, device=dev if ws > 1 else None)
    e2e_value = flops * len(e2e_times) * ws / e2e_t / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_block(),
        "kernel": "t2s_gemm_f32 (packed FP32 FMA, TMA + mbarrier ring; %s)" % PLAN_NAMES.get(plan, plan),
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 4 * (M * K + K * N),
                "d2h_bytes_per_step": 4 * M * N,
                "call": "t2s_gemm_f32_host (pinned host A, B, C; copies overlapped in the call)"},
        "gpu_launches": args.steps * launches_per_call,
        "clocks": clocks,
    }

    # ---- reported separately: 3xTF32 tensor-core kernel and the 1024^3 shape
    if not args.skip_extras:
        line["tf32x3"] = extra_tf32x3(lib, dA, dB, M, N, K, stream, flush, args, dev, ws,
                                      probes["tf32_mma_tflops"])
        line["bf16"] = extra_half(lib, M, N, K, stream, flush, args, dev, "bf16")
        line["f16"] = extra_half(lib, M, N, K, stream, flush, args, dev, "f16")
        line["f64"] = extra_f64(lib, stream, flush, args, dev)
        line["also_1024"] = extra_1024(lib, dev, stream, flush, args, ws)
        line["memory_roof"] = extra_vector_add(lib, dev, stream, flush, args)
        line["memory_roof"]["c_store_probe"] = extra_store_probe(dev, stream)

    if rank == 0 and ws == 1 and not args.skip_cpu:
        rate, info = cpu_oracle_rate(A, B, float(os.environ.get("T2S_CPU_SECONDS", "12")))
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": info["cores"],
                                "kind": "oracle", "sample": info["sample"]}
        line["cpu_baseline_blocked"] = cpu_blocked_rate(A, B)
        line["cpu_literal_loop_1024"] = cpu_literal_loop_1024()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def extra_tf32x3(lib, dA, dB, M, N, K, stream, flush, args, dev, ws, tf32_probe=None):
    import torch
    from roofline_driven_tiling_gb300 import binding
    from roofline_driven_tiling_gb300 import roofline as rl
    need = lib.t2s_gemm_f32_tf32x3_workspace_size(M, N, K)
    wsbuf = torch.empty(need, dtype=torch.uint8, device=dev)
    dC = torch.empty((M, N), dtype=torch.float32, device=dev)
    sp = stream.cuda_stream

    def step():
        rc = lib.t2s_gemm_f32_tf32x3(M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                                     wsbuf.data_ptr(), need, sp)
        if rc != 0:
            raise binding.T2SError(rc, "t2s_gemm_f32_tf32x3")

    try:
        times = time_steps(step, args.steps, max(args.warmup, 3), stream, flush)
    except binding.T2SError as e:
        return {"unavailable": str(e)}
    flops = rl.gemm_flops(M, N, K)
    t = sum(times) / len(times) / 1e3
    if tf32_probe:
        tf32_peak = tf32_probe
        basis = ("t2s_probe_tf32_mma: back-to-back tcgen05.mma kind::tf32 M128 N256 K8 on "
                 "shared-memory operands, one CTA per SM (measured, burst)")
    else:
        # Fallback: the measured bf16 burst figure x the nominal tf32 : bf16 ratio (1.1 : 2.25).
        tf32_peak = float(measured_peaks().get("bf16_tflops", 1898.5)) * 1.1 / 2.25
        basis = "measured bf16 burst x 1.1/2.25 (nominal tf32:bf16)"
    return {"value": flops / t / 1e12, "unit": UNIT, "ms_per_step": t * 1e3,
            "kernel": "t2s_gemm_f32_tf32x3 (split pre-pass + tcgen05 kind::tf32, 3 MMAs)",
            "roofline": {"bound": "tensor", "achieved_effective": flops / t / 1e12,
                         "tensor_flops_per_launch": 3 * flops,
                         "achieved_tensor": 3 * flops / t / 1e12, "peak": tf32_peak,
                         "frac": 3 * flops / t / 1e12 / tf32_peak, "unit": UNIT,
                         "peak_basis": basis,
                         "traffic": profile_traffic(TF32X3_PROFILE, "tf32x3")}}


def extra_half(lib, M, N, K, stream, flush, args, dev, fmt="bf16"):
    """A 16-bit-operand product (FP32 accumulation) on the same shape, against the measured
    dense bf16 tensor peak (FP16 runs at the same nominal rate); `fmt` is "bf16" or "f16"."""
    import torch
    from roofline_driven_tiling_gb300 import binding, inputs
    from roofline_driven_tiling_gb300 import roofline as rl
    make = inputs.uniform_bf16 if fmt == "bf16" else inputs.uniform_f16
    Ab = make(M, K, inputs.SEED_A_BASE + WORKLOAD["config_no"])
    Bb = make(K, N, inputs.SEED_B_BASE + WORKLOAD["config_no"])
    dA = torch.from_numpy(Ab.view(np.int16)).to(dev)
    dB = torch.from_numpy(Bb.view(np.int16)).to(dev)
    dC = torch.empty((M, N), dtype=torch.float32, device=dev)
    name = "t2s_gemm_%s_f32" % fmt
    need = getattr(lib, name + "_workspace_size")(M, N, K)
    wsbuf = torch.empty(need, dtype=torch.uint8, device=dev)
    sp = stream.cuda_stream
    fn = getattr(lib, name)

    def step():
        rc = fn(M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), wsbuf.data_ptr(), need, sp)
        if rc != 0:
            raise binding.T2SError(rc, name)

    try:
        times = time_steps(step, args.steps, max(args.warmup, 3), stream, flush)
    except binding.T2SError as e:
        return {"unavailable": str(e)}
    flops = rl.gemm_flops(M, N, K)
    t = sum(times) / len(times) / 1e3
    peak = float(measured_peaks().get("bf16_tflops", 1898.5))
    label = "bfloat16" if fmt == "bf16" else "binary16"
    cut = "uniform values cut to bfloat16" if fmt == "bf16" else "uniform on the 2^-11 grid"
    return {"value": flops / t / 1e12, "unit": UNIT, "ms_per_step": t * 1e3,
            "workload": "%dx%dx%d, %s A and B (%s), FP32 C" % (M, N, K, label, cut),
            "kernel": "%s (B read in place, tcgen05 kind::f16 on SM pairs, FP32 acc.)" % name,
            "roofline": {"bound": "tensor", "achieved": flops / t / 1e12, "peak": peak,
                         "frac": flops / t / 1e12 / peak, "unit": UNIT,
                         "peak_basis": "measured cuBLAS bf16 burst (FP16 has the same nominal rate)",
                         "traffic": profile_traffic(BF16_PROFILE if fmt == "bf16" else F16_PROFILE,
                                                    "bf16")}}


def extra_f64(lib, stream, flush, args, dev):
    """The FP64 kernels at 2048^3 (uniform binary64 inputs) against the FP64 CUDA-core rate
    (DFMA units x 2 FLOP x SMs x clock; the units per SM are the measured probe figure)."""
    import torch
    from roofline_driven_tiling_gb300 import binding, inputs
    from roofline_driven_tiling_gb300 import roofline as rl
    n = 2048
    dA = torch.from_numpy(inputs.uniform_f64(n, n, 5001)).to(dev)
    dB = torch.from_numpy(inputs.uniform_f64(n, n, 5002)).to(dev)
    dC = torch.empty((n, n), dtype=torch.float64, device=dev)
    sp = stream.cuda_stream
    out = {"workload": "dgemm 2048^3 fp64, uniform on [-1, 1) (L2 flushed per step)",
           "peak_tflops": rl.fp64_peak_tflops(), "peak_basis": rl.FP64_PEAK_BASIS}
    for name in ("ffma", "smem32", "naive"):
        fn = getattr(lib, binding.KERNELS_F64[name])

        def step(fn=fn):
            rc = fn(n, n, n, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sp)
            if rc != 0:
                raise binding.T2SError(rc, binding.KERNELS_F64[name])

        times = time_steps(step, max(3, min(args.steps // 10, 10)), 3, stream, flush)
        t = sum(times) / len(times) / 1e3
        tf = rl.gemm_flops(n, n, n) / t / 1e12
        out[name] = {"ms": t * 1e3, "tflops": tf, "frac": tf / rl.fp64_peak_tflops()}
    out["ffma"]["traffic"] = profile_traffic(F64_PROFILE, "f64")
    return out


def extra_1024(lib, dev, stream, flush, args, ws):
    import torch
    from roofline_driven_tiling_gb300 import inputs
    from roofline_driven_tiling_gb300 import roofline as rl
    n = 1024
    A, B = inputs.integer_pattern(n, n, n)
    dA, dB = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    dC = torch.empty((n, n), dtype=torch.float32, device=dev)
    sp = stream.cuda_stream
    out = {"workload": "sgemm 1024^3 fp32, integer pattern (L2 flushed per step)"}
    need = lib.t2s_gemm_f32_splitk_workspace_size(n, n, n, 0)
    wsk = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    wss = torch.empty(max(lib.t2s_gemm_f32_streamk_workspace_size(n, n, n), 256),
                      dtype=torch.uint8, device=dev)

    def splitk(M, N, K, a, b, c, s):
        return lib.t2s_gemm_f32_splitk(M, N, K, a, b, c, 0, wsk.data_ptr(), wsk.numel(), s)

    def streamk(M, N, K, a, b, c, s):
        return lib.t2s_gemm_f32_streamk(M, N, K, a, b, c, wss.data_ptr(), wss.numel(), s)

    wst = torch.empty(max(lib.t2s_gemm_f32_tf32x3_workspace_size(n, n, n), 256),
                      dtype=torch.uint8, device=dev)

    def tf32x3(M, N, K, a, b, c, s):
        return lib.t2s_gemm_f32_tf32x3(M, N, K, a, b, c, wst.data_ptr(), wst.numel(), s)

    for name, fn in (("ffma", lib.t2s_gemm_f32), ("ffma_splitk_auto", splitk),
                     ("ffma_streamk", streamk), ("tf32x3", tf32x3),
                     ("naive", lib.t2s_gemm_f32_naive),
                     ("smem32", lib.t2s_gemm_f32_smem32)):
        times = time_steps(lambda: fn(n, n, n, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sp),
                           max(args.steps, 10), 3, stream, flush)
        t = sum(times) / len(times) / 1e3
        out[name] = {"ms": t * 1e3, "tflops": rl.gemm_flops(n, n, n) / t / 1e12,
                     "frac_fp32_peak": rl.gemm_flops(n, n, n) / t / 1e12 / rl.fp32_peak_tflops()}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out["ffma"]["tiling"] = PLAN_NAMES.get(lib.t2s_gemm_f32_plan(n, n, n, sms))
    out["ffma"]["traffic"] = profile_traffic(FFMA_1024_PROFILE, "ffma")
    return out


def extra_vector_add(lib, dev, stream, flush, args):
    """Vector add z = x + y over 2^28 floats (3 GB moved per call): the bandwidth slope of
    the roofline (AI = 1/12 FLOP/B), measured with the same timing rules."""
    import torch
    from roofline_driven_tiling_gb300 import binding
    from roofline_driven_tiling_gb300 import roofline as rl
    n = 1 << 28
    x = torch.empty(n, dtype=torch.float32, device=dev).uniform_(-1, 1)
    y = torch.empty(n, dtype=torch.float32, device=dev).uniform_(-1, 1)
    z = torch.empty(n, dtype=torch.float32, device=dev)
    sp = stream.cuda_stream

    def step():
        rc = lib.t2s_vector_add_f32(n, x.data_ptr(), y.data_ptr(), z.data_ptr(), sp)
        if rc != 0:
            raise binding.T2SError(rc, "t2s_vector_add_f32")

    times = time_steps(step, max(args.steps // 5, 5), 3, stream, flush)
    t = sum(times) / len(times) / 1e3
    nbytes = rl.vector_add_bytes(n)
    gbs = nbytes / t / 1e9
    peak = float(measured_peaks().get("hbm_gbs", 6792.4))
    return {"workload": "z = x + y, 2^28 fp32 elements (12 bytes moved per element)",
            "kernel": "t2s_vector_add_f32 (32-byte loads and stores)",
            "ms": t * 1e3, "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak,
            "bound": "hbm", "ai": rl.arithmetic_intensity(rl.vector_add_flops(n), nbytes),
            "tflops": n / t / 1e12}


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--skip-cpu", action="store_true", help="omit the CPU oracle baseline")
    p.add_argument("--skip-extras", action="store_true", help="omit tf32x3 and 1024^3 lines")
    p.add_argument("--cpu-configs", action="store_true",
                   help="only time the CPU oracle on every configuration's workload (host cores, "
                        "no GPU) and print one JSON line")
    args = p.parse_args(argv)
    if args.cpu_configs:
        print(json.dumps({"cpu_oracle_configs": cpu_oracle_configs(), "kind": "oracle"}), flush=True)
        return 0
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
