"""Roofline sweep: every FP32 entry point over the sweep shapes, placed on the GB300 roofline.

    python -m roofline_driven_tiling_gb300.sweep [--iters 50] [--no-flush] [--out FILE]
        [--shapes MxNxK,...] [--kernels ffma,...] [--splitk-chunks S] [--misalign]

The pages this library follows time a GEMM at one size and read the result against the
roofline (page "4주차: Roofline과 Tiling", sections "2. Roofline" and "실제 Kernel을 plot 해보면":
attainable = min(peak, bandwidth x AI); page "GEMM 커널 테스트 코드 작성 및 최적화 (1024^3 크기
실험)", section "결과 해석": GFLOP/s = FLOPs / time). This tool does the same for the square
shapes 128^3 .. 8192^3, the two low-AI shapes 16384 x 16384 x 32 and 8192 x 8192 x 64, and
the ragged 1000 x 1003 x 997, for the product and the other FP32 entry points.

* Inputs: uniform on [-1, 1) from the library's seeded generator (seeds 1005 / 2005).
* Timing: CUDA events on the launching stream around each call, after 5 untimed calls; by
  default an L2 flush (a 256 MB write) before every timed call, so that A and B come from
  HBM as the roofline's byte count assumes (--no-flush times back-to-back calls instead, as
  the pages do). Median, minimum and mean over the timed calls.
* Roof: min(P, BW x AI) with AI = 2MNK / 4(MK + KN + MN) (algorithmic bytes), P the FP32
  CUDA-core peak (SMs x 128 lanes x 2 x 2070 MHz) and BW the measured copy bandwidth
  (MEASURED_PEAKS.json beside the package when present, else 6800 GB/s). The 3xTF32 entry
  point runs on the tensor cores: its effective FLOP/s are reported against the same FP32
  roof, for comparison.
* Each result is compared with the product's: bit for bit for the naive and smem32 kernels
  (the same fused multiply-adds in the same order), within 1e-6 K max|a| max|b| for the
  others. A mismatch is reported in the line and fails the run.
* `cublas` is the vendor library's FP32 product (torch.mm with TF32 off), timed the same way
  as a comparison point; it is not part of this library.
* --shapes replaces the sweep's shapes (one small shape and one kernel make a short run that
  a profiler can capture), --splitk-chunks fixes the split-K chunk count (0: the automatic
  choice), and --misalign offsets A, B and C by one float so that every kernel takes its
  general (non-TMA) load path.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

SHAPES = [(n, n, n) for n in (128, 256, 512, 1024, 2048, 4096, 8192)] + [
    (16384, 16384, 32), (8192, 8192, 64), (1000, 1003, 997)]
KERNELS = ("ffma", "tf32x3", "splitk", "streamk", "smem32", "naive", "cublas")
SEED_A, SEED_B = 1005, 2005
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


def _hbm_gbs():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


def _calls(binding, lib, M, N, K, dA, dB, dC, ws, stream, chunks=0, shift=0, torch=None):
    """One closure per entry point (the workspace tensor is large enough for all), and the
    vendor library's product for comparison."""
    a, b, c, s = (dA.data_ptr() + 4 * shift, dB.data_ptr() + 4 * shift,
                  dC.data_ptr() + 4 * shift, stream)
    w, wn = ws.data_ptr(), ws.numel()

    def check(rc, name):
        if rc != binding.T2S_OK:
            raise binding.T2SError(rc, name)

    return {
        "ffma": lambda: check(lib.t2s_gemm_f32(M, N, K, a, b, c, s), "t2s_gemm_f32"),
        "tf32x3": lambda: check(lib.t2s_gemm_f32_tf32x3(M, N, K, a, b, c, w, wn, s),
                                "t2s_gemm_f32_tf32x3"),
        "splitk": lambda: check(lib.t2s_gemm_f32_splitk(M, N, K, a, b, c, chunks, w, wn, s),
                                "t2s_gemm_f32_splitk"),
        "streamk": lambda: check(lib.t2s_gemm_f32_streamk(M, N, K, a, b, c, w, wn, s),
                                 "t2s_gemm_f32_streamk"),
        "smem32": lambda: check(lib.t2s_gemm_f32_smem32(M, N, K, a, b, c, s),
                                "t2s_gemm_f32_smem32"),
        "naive": lambda: check(lib.t2s_gemm_f32_naive(M, N, K, a, b, c, s), "t2s_gemm_f32_naive"),
        "cublas": lambda: torch.mm(dA[shift:].view(M, K), dB[shift:].view(K, N),
                                   out=dC[shift:].view(M, N)),
    }


def _workspace_bytes(lib, M, N, K, chunks=0):
    return max(lib.t2s_gemm_f32_tf32x3_workspace_size(M, N, K),
               lib.t2s_gemm_f32_splitk_workspace_size(M, N, K, chunks),
               lib.t2s_gemm_f32_streamk_workspace_size(M, N, K), 256)


def _time(torch, fn, iters, stream, flush):
    for _ in range(5):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    with torch.cuda.stream(stream):
        for s, e in ev:
            if flush is not None:
                flush.add_(1)
            s.record(stream)
            fn()
            e.record(stream)
    torch.cuda.synchronize()
    ms = sorted(s.elapsed_time(e) for s, e in ev)
    return ms[len(ms) // 2], ms[0], sum(ms) / len(ms)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--iters", type=int, default=50, help="timed calls per point (at most)")
    ap.add_argument("--no-flush", action="store_true", help="time back-to-back calls")
    ap.add_argument("--kernels", default=",".join(KERNELS))
    ap.add_argument("--out", default=None, help="also write the JSON lines to this file")
    ap.add_argument("--shapes", default=None, help="MxNxK[,MxNxK...] instead of the sweep")
    ap.add_argument("--splitk-chunks", type=int, default=0, help="split-K chunks (0: automatic)")
    ap.add_argument("--misalign", action="store_true",
                    help="offset A, B and C by one float (the general load path)")
    args = ap.parse_args(argv)
    shapes = SHAPES if not args.shapes else [tuple(int(x) for x in t.split("x"))
                                             for t in args.shapes.split(",") if t]
    shift = 1 if args.misalign else 0

    import torch

    from . import binding, inputs, roofline as rl
    from .clocks import ClockSampler

    if not torch.cuda.is_available():
        raise SystemExit("the sweep needs a CUDA device")
    lib = binding.lib()
    dev = torch.device("cuda")
    stream = torch.cuda.Stream(dev)
    flush = None if args.no_flush else torch.zeros(FLUSH_BYTES // 4, device=dev)
    bw, bw_basis = _hbm_gbs()
    peak = rl.fp32_peak_tflops()
    kernels = [k for k in args.kernels.split(",") if k]
    if "cublas" in kernels:
        # The FP32 product, not TF32.
        torch.backends.cuda.matmul.allow_tf32 = False
        torch.set_float32_matmul_precision("highest")
    out = open(args.out, "w") if args.out else None
    rows, bad = [], 0
    clk = ClockSampler(torch.cuda.current_device())
    with clk:
        for (M, N, K) in shapes:
            A, B = inputs.uniform(M, K, SEED_A), inputs.uniform(K, N, SEED_B)
            dA = torch.zeros(M * K + shift, dtype=torch.float32, device=dev)
            dB = torch.zeros(K * N + shift, dtype=torch.float32, device=dev)
            dA[shift:] = torch.from_numpy(A.ravel()).to(dev)
            dB[shift:] = torch.from_numpy(B.ravel()).to(dev)
            dC_buf = torch.empty(M * N + shift, dtype=torch.float32, device=dev)
            dC = dC_buf[shift:].view(M, N)
            ws = torch.empty(_workspace_bytes(lib, M, N, K, args.splitk_chunks), dtype=torch.uint8,
                             device=dev)
            calls = _calls(binding, lib, M, N, K, dA, dB, dC_buf, ws, stream.cuda_stream,
                           args.splitk_chunks, shift, torch)
            flops = rl.gemm_flops(M, N, K)
            tol = 1e-6 * K * float(abs(A).max()) * float(abs(B).max())
            ref = None
            for name in kernels:
                fn = calls[name]
                with torch.cuda.stream(stream):
                    dC.fill_(float("nan"))
                    fn()
                torch.cuda.synchronize()
                if binding.t2s_device_status(stream.cuda_stream) != binding.T2S_OK:
                    raise SystemExit("device status reports a timed-out wait (%s)" % name)
                if name == "ffma":
                    ref = dC.clone()
                    check = "reference"
                elif ref is None:
                    check = "unchecked"
                else:
                    diff = float((dC - ref).abs().max())
                    exact = bool(torch.equal(dC.view(torch.int32), ref.view(torch.int32)))
                    if name in ("naive", "smem32"):
                        check = "bit-exact" if exact else "MISMATCH"
                    elif exact:
                        check = "bit-exact"
                    else:
                        check = "within tolerance" if diff <= tol else "MISMATCH"
                    bad += check == "MISMATCH"
                # Keep each point to about half a second of device time.
                est = flops / (1e12 * (5.0 if name in ("naive", "smem32") else 30.0))
                iters = max(3, min(args.iters, int(0.5 / max(est, 1e-6))))
                med, mn, mean = _time(torch, fn, iters, stream, flush)
                pt = rl.place(flops, med / 1e3, rl.gemm_bytes(M, N, K), peak, bw)
                rec = {"shape": [M, N, K], "kernel": name, "iters": iters, "ms_median": med,
                       "ms_min": mn, "ms_mean": mean, "tflops": pt["tflops"], "ai": pt["ai"],
                       "roof_tflops": pt["roof_tflops"], "frac_of_roof": pt["frac_of_roof"],
                       "region": pt["region"], "check": check, "l2_flush": flush is not None,
                       "bw_gbs": bw, "bw_basis": bw_basis}
                if name == "ffma":
                    rec["plan"] = binding.t2s_gemm_f32_plan(
                        M, N, K, torch.cuda.get_device_properties(dev).multi_processor_count)
                line = json.dumps(rec)
                print(line, flush=True)
                if out:
                    out.write(line + "\n")
                rows.append(rec)
            del dA, dB, dC, dC_buf, ws
            torch.cuda.empty_cache()
    if out:
        out.close()
    # Summary table: TFLOP/s (fraction of the roof) per shape and kernel.
    print("\n| shape | AI | roof | " + " | ".join(kernels) + " |")
    print("|---|---|---|" + "---|" * len(kernels))
    for (M, N, K) in shapes:
        pts = {r["kernel"]: r for r in rows if r["shape"] == [M, N, K]}
        first = next(iter(pts.values()))
        cells = ["%.1f (%.0f %%)" % (pts[k]["tflops"], 100 * pts[k]["frac_of_roof"]) if k in pts
                 else "—" for k in kernels]
        print("| %dx%dx%d | %.1f | %.1f | %s |" % (M, N, K, first["ai"], first["roof_tflops"],
                                                   " | ".join(cells)))
    c = clk.summary()
    if c:
        print("\nclocks during the sweep: median %.0f MHz (maximum %.0f), %d samples, throttle "
              "reasons: %s" % (c["sm_mhz"], c["sm_max_mhz"], c["samples"],
                               ", ".join(c["reasons"]) or "none"))
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main())
