#!/usr/bin/env python3
"""Benchmark of the FP32 matrix product C = A * B on GB300 (one JSON line).

Default workload: M = N = K = 4096, A and B i.i.d. uniform[-1, 1) from seed 1
(the pages' problem size, "GEMM from naive to tiled", section 二.1). A step
is one call of the C ABI on device-resident inputs; L2 is flushed (a 256 MiB
device write, then a 256 MiB read, so that no dirty lines remain) before
every step, outside the timed events. Reported:

  value      TFLOP/s = 2 M N K / mean device time of a step (CUDA events on
             the launching stream), summed over ranks (replicas);
  roofline   the bound of the kernel the step runs: "tensor" for the 3xTF32
             kernels (the dense TF32 tensor rate, SMs x 4096 ops/clk x the
             median SM clock sampled inside the timed region, divided by the
             3 products per fp32 product; the measured bf16 burst scaled to
             TF32 is given beside it as context), "hbm" for the vector shapes
             (algorithmic bytes against the measured copy bandwidth), "alu"
             for the FFMA kernels (SMs x 128 FMA/clk x 2 flop x the median SM
             clock sampled inside the timed region);
  ffma_kernel  the CUDA-core FFMA kernel on the same inputs, timed the same
             way with its own clock record, as a fraction of the FP32 FMA
             peak at that clock;
  e2e        the same metric through sgemm_host(): pinned host A, B in,
             host C out, copies inside the timed region;
  cpu_baseline  the CPU oracle timed on this host's cores on a bounded row
             sample of the same product.

``--impl reference`` times the CPU oracle (the reference of this build) on
the same workload instead. Under torchrun (N > 1) each rank runs its own
replica on its own GPU; only rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FMA_PER_CLK_PER_SM = 128   # FP32 FMA lanes per SM (4 SMSPs x 32)
L2_FLUSH_BYTES = 256 << 20
CPU_SAMPLE_SECONDS = 12.0
# Nominal dense tensor rates per GPU: TF32 1.1 PFLOP/s, BF16 2.25 PFLOP/s.
TF32_PER_BF16 = 1.1 / 2.25
BF16_FALLBACK_TFLOPS = 1900.0   # used only when no measured peak is present
HBM_FALLBACK_GBS = 6800.0
TF32X3_PRODUCTS = 3             # TF32 tensor products per fp32 product
# Dense TF32 tensor-core rate of one SM, ops per clock, as ncu reports it
# for this part (the peak_sustained of its TF32 tensor-op counter).
TF32_OPS_PER_CLK_PER_SM = 4096


def flops(M, N, K):
    return 2.0 * M * N * K


def algorithmic_bytes(M, N, K):
    return 4.0 * (M * K + K * N + M * N)


# Source files that define each kernel (its traffic record is valid only
# while these are unchanged).
KERNEL_SOURCES = {
    "k_tiled_tma": ["sgemm_tiled.cu", "ptx.cuh", "kernels.h"],
    "k_tf32x3": ["sgemm_tf32x3.cu", "tcgen05.cuh", "ptx.cuh", "kernels.h"],
    "k_tf32x3_pair": ["sgemm_tf32x3.cu", "tcgen05.cuh", "ptx.cuh",
                      "kernels.h"],
    "k_gemv_row_tma": ["sgemm_gemv.cu", "ptx.cuh", "kernels.h"],
    "k_gemv_col_tma": ["sgemm_gemv.cu", "ptx.cuh", "kernels.h"],
    "k_tiled_ldg": ["sgemm_tiled.cu", "ptx.cuh", "kernels.h"],
    "k_small": ["sgemm_small.cu", "ptx.cuh", "kernels.h"],
    "k_gemv_row": ["sgemm_small.cu", "ptx.cuh", "kernels.h"],
    "k_gemv_col": ["sgemm_small.cu", "ptx.cuh", "kernels.h"],
}


def source_digest(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp32_matrix_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(kernel, workload):
    """dram bytes per launch from the committed ncu record, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            recs = json.load(f)
    except (OSError, ValueError):
        return None
    if kernel not in KERNEL_SOURCES:
        return None
    digest = source_digest(kernel)
    for r in recs.get("records", []):
        if (r.get("kernel") == kernel and r.get("workload") == workload
                and r.get("source_sha256") == digest):
            return r.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running.

    Samples every 25 ms with nvidia-smi's own timestamps; ``window()`` marks
    the host-side start and end of the timed region (the end taken after
    the device synchronised), and the summary keeps the samples inside it,
    so the median is the clock under load, not the idle clock around it.
    """

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 25

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev),
                 "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms",
                 str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(
                text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "note": "nvidia-smi unavailable"}
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.lines:
            p = [x.strip() for x in line.split(",")]
            try:
                rows.append((self._stamp(p[0]), float(p[1]), float(p[2]),
                             float(p[3]), [n for n, v in zip(names, p[5:9])
                                           if v.lower() == "active"]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if r[0] is not None and self.t0 is not None
                  and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        basis = "samples inside the timed region"
        if not inside:
            # no stamp inside (a very short region): the upper half of all
            # samples, as the kernel keeps the SM clock up while it runs
            inside = sorted(rows, key=lambda r: r[1])[len(rows) // 2:]
            basis = "upper half of the samples around the timed region"
        sm = [r[1] for r in inside]
        reasons = sorted({n for r in inside for n in r[4]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in rows) if rows else None,
                "reasons": reasons, "samples": len(rows),
                "samples_in_region": len(sm), "basis": basis,
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max(r[3] for r in inside) if inside else None}


def measured_bf16_tflops():
    """(bf16 dense TFLOP/s burst, source) from MEASURED_PEAKS.json."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured"
    except (OSError, ValueError, KeyError):
        return BF16_FALLBACK_TFLOPS, "fallback"


def measured_hbm_gbs():
    """(HBM copy GB/s, source) from MEASURED_PEAKS.json."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, ValueError, KeyError):
        return HBM_FALLBACK_GBS, "fallback"


class L2Flush:
    """Evicts the step's inputs from L2 before each step: writes a buffer
    larger than L2, then reads another one, so that L2 is left holding clean
    lines and the timed step pays no write-back of the flush's dirty data."""

    def __init__(self):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32,
                             device="cuda")
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=(0,), out=self.sink)


def time_steps(step, flush, stream, n, warmup, sampler=None):
    """Per-step device times (ms) with an L2 flush before each step; the
    clock sampler (if any) is told where the timed region starts and ends."""
    import torch
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    if sampler is not None:
        sampler.start()
    for i in range(n):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.stop()
    return [a.elapsed_time(b) for a, b in ev]


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_oracle_rate(M, N, K, kind, seed, target_s=CPU_SAMPLE_SECONDS,
                    min_rows=None):
    """TFLOP/s of the CPU oracle on a row sample of the product, sized to run
    about target_s seconds. Returns (tflops, rows, seconds, threads)."""
    import numpy as np
    import matgen
    import oracle
    threads = oracle.num_threads()
    A = matgen.KINDS[kind](seed, matgen.MATRIX_A, M, K)
    B = matgen.KINDS[kind](seed, matgen.MATRIX_B, K, N)
    rows = max(threads, 1) if min_rows is None else min_rows
    while True:
        idx = np.arange(rows, dtype=np.int64) % M
        t0 = time.perf_counter()
        oracle.gemm_rows(A, B, idx)
        dt = time.perf_counter() - t0
        if dt >= target_s / 4 or rows >= M:
            break
        rows = min(M, rows * 2)
    if dt < target_s and rows < M:
        rows = int(min(M, max(rows, rows * target_s / max(dt, 1e-6))))
        idx = np.arange(rows, dtype=np.int64) % M
        t0 = time.perf_counter()
        oracle.gemm_rows(A, B, idx)
        dt = time.perf_counter() - t0
    return flops(rows, N, K) / dt / 1e12, rows, dt, threads


def reduce_max(x, world, device="cuda"):
    """Max over the ranks of a per-rank number (the slowest replica sets the
    whole-job time); the number itself for one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_rank, ms_max, world):
    """Whole-job throughput: every rank's flops over the slowest rank's time."""
    return flop_per_rank * world / (ms_max * 1e-3) / 1e12


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import matgen
    import oracle
    M, N, K = w["M"], w["N"], w["K"]
    threads = oracle.num_threads()
    A = matgen.KINDS[w["kind"]](w["seed"], matgen.MATRIX_A, M, K)
    B = matgen.KINDS[w["kind"]](w["seed"], matgen.MATRIX_B, K, N)
    # Size one step so that warmup + steps take about 90 s in total.
    probe_rows = max(threads, 1)
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, np.arange(probe_rows, dtype=np.int64))
    t_row = (time.perf_counter() - t0) / probe_rows
    budget = 90.0 / max(args.steps + args.warmup, 1)
    rows = int(max(threads, min(M, budget / max(t_row, 1e-9))))
    rows = max(1, min(M, rows))
    times = []
    for step in range(args.warmup + args.steps):
        start = (step * rows) % M
        idx = (start + np.arange(rows, dtype=np.int64)) % M
        t0 = time.perf_counter()
        oracle.gemm_rows(A, B, idx)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
    sec = sum(times) / len(times)
    value = flops(rows, N, K) / sec / 1e12
    sample = ("%d of %d rows of C per step (fp64 oracle, row order i-k-j)"
              % (rows, M))
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_of(w, extra={"sample": sample}),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = ("FP32 SGEMM TFLOP/s at M=N=K=4096 and % of GB300 FP32 FFMA peak "
          "(1 GPU)")


def config_of(w, extra=None):
    c = {"workload": w["name"], "M": w["M"], "N": w["N"], "K": w["K"],
         "layout": "row-major, dense leading dimensions",
         "inputs": "%s, seed %d" % (w["kind"], w["seed"])}
    if extra:
        c.update(extra)
    return c


def run_gpu(args, w):
    import numpy as np
    import torch
    import matgen
    import dense_fp32_matrix_gb300 as dfm
    from dense_fp32_matrix_gb300 import build

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    build.build()

    M, N, K = w["M"], w["N"], w["K"]
    A = torch.from_numpy(matgen.KINDS[w["kind"]](w["seed"], 0, M, K)).cuda()
    B = torch.from_numpy(matgen.KINDS[w["kind"]](w["seed"], 1, K, N)).cuda()
    C = torch.empty((M, N), device="cuda")
    # Layout of the timed product: dense by default; --pad adds floats to
    # every row of A, B and C (leading dimensions K + pad, N + pad) and
    # --offset shifts their bases by that many floats (misaligned for the
    # paths that need 16-byte rows). A, B, C keep dense copies for the e2e
    # leg and its check.
    # --ops: A and/or B stored transposed (A as K x M, B as N x K) and the
    # product run through sgemm_ex; the logical A, B stay for the e2e leg.
    op_a, op_b = args.ops[0], args.ops[1]
    As = A.t().contiguous() if op_a == "T" else A
    Bs = B.t().contiguous() if op_b == "T" else B
    lda = (M if op_a == "T" else K) + args.pad
    ldb = (K if op_b == "T" else N) + args.pad
    ldc = N + args.pad
    keep = []

    def placed(X, rows, cols, ld):
        buf = torch.zeros(args.offset + rows * ld + 4, device="cuda")
        buf[args.offset:args.offset + rows * ld].view(rows, ld)[:, :cols] = X
        keep.append(buf)
        view = buf[args.offset:args.offset + rows * ld].view(rows, ld)[:, :cols]
        return buf.data_ptr() + 4 * args.offset, view

    if args.pad or args.offset:
        pA, _ = placed(As, As.shape[0], As.shape[1], lda)
        pB, _ = placed(Bs, Bs.shape[0], Bs.shape[1], ldb)
        pC, C = placed(C, M, N, ldc)
    else:
        pA, pB, pC = As.data_ptr(), Bs.data_ptr(), C.data_ptr()
    flush = L2Flush()
    stream = torch.cuda.current_stream()
    path_name = args.path
    plan = dfm.sgemm_plan_ex(op_a, op_b, M, N, K, lda, ldb, ldc, pA, pB,
                             pC) if path_name == "auto" else path_name

    def step():
        if args.ops == "NN":
            dfm.sgemm_path(M, N, K, pA, lda, pB, ldb, pC, ldc, stream,
                           path_name)
        else:
            dfm.sgemm_ex(op_a, op_b, M, N, K, 1.0, pA, lda, pB, ldb, 0.0, pC,
                         ldc, stream, path_name)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    st, site = dfm.sgemm_watchdog_status()
    if st != 0:
        raise RuntimeError("watchdog fired during warm-up (site %d)" % site)

    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = dfm.sgemm_launch_count()
    with ClockSampler(dev) as clocks:
        clocks.start()
        for i in range(args.steps):
            flush()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        clocks.stop()
    launches = dfm.sgemm_launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    st, site = dfm.sgemm_watchdog_status()
    if st != 0:
        raise RuntimeError("watchdog fired during timing (site %d)" % site)
    ms = [a.elapsed_time(b) for a, b in ev]
    ms_step = reduce_max(sum(ms) / len(ms), world)
    tflops = flops(M, N, K) / (ms_step * 1e-3) / 1e12
    value = job_tflops(flops(M, N, K), ms_step, world)
    clk = clocks.summary()

    # e2e through the C ABI with host buffers: H2D inputs, compute, D2H C.
    hA = A.cpu().pin_memory()
    hB = B.cpu().pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    dA = torch.empty_like(A)
    dB = torch.empty_like(B)
    dC = torch.empty((M, N), device="cuda")
    e2e_steps = max(3, min(args.steps, 50))
    # sgemm_host takes sgemm's own path choice; with a forced CUDA-core path
    # the e2e leg runs in the CUDA-core math mode so that it computes with
    # the same arithmetic.
    prev_mode = dfm.sgemm_set_math_mode(
        "auto" if plan.startswith("tf32x3") else "ffma")
    e2e_plan = dfm.sgemm_plan(M, N, K, K, N, N, dA.data_ptr(),
                              dB.data_ptr(), dC.data_ptr())
    for _ in range(3):
        dfm.sgemm_host(M, N, K, hA, K, hB, N, hC, N, dA, dB, dC, stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        dfm.sgemm_host(M, N, K, hA, K, hB, N, hC, N, dA, dB, dC, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world)
    dfm.sgemm_set_math_mode(prev_mode)
    # sgemm_host pipelines large products in row blocks, each computed as
    # sgemm of that block, so it may differ from the one-piece product in
    # the last bits: check it against the device result within twice the
    # accuracy bound, with S_ij = sum_k |A_ik B_kj| bounded by
    # (sum_k |A_ik|) * max |B| (no extra matrix product needed).
    s_bound = A.abs().sum(dim=1, keepdim=True).cpu() * B.abs().max().item()
    if not bool(((hC - C.cpu()).abs() <= 2e-4 * s_bound + 2e-6).all()):
        raise RuntimeError("e2e result differs from the device-path result")

    def ffma_peak_at(mhz):
        return sms * FMA_PER_CLK_PER_SM * 2 * mhz * 1e6 / 1e12

    def ffma_basis(mhz, where):
        return ("%d SMs x %d FP32 FMA/clk x 2 flop x %.0f MHz (median SM "
                "clock of the samples inside %s)"
                % (sms, FMA_PER_CLK_PER_SM, mhz, where))

    # The clock of the timed region (its median under load).
    clock_mhz = clk["sm_mhz"] or (clk["sm_max_mhz"] or 2070.0)
    kernel = {"tiled_tma": "k_tiled_tma", "tiled_ldg": "k_tiled_ldg",
              "tf32x3": "k_tf32x3", "tf32x3_pair": "k_tf32x3_pair",
              "gemv_row": "k_gemv_row_tma", "gemv_col": "k_gemv_col_tma",
              "small": "k_small", "naive": "k_naive"}.get(plan, plan)
    # The vector paths take their TMA kernels only for 16-byte aligned
    # operands (the same test as the library's); else the plain ones.
    if plan == "gemv_row" and not (pB % 16 == 0 and ldb % 4 == 0
                                   and pA % 16 == 0):
        kernel = "k_gemv_row"
    if plan == "gemv_col" and not (pA % 16 == 0 and lda % 4 == 0
                                   and ldb == 1 and pB % 16 == 0):
        kernel = "k_gemv_col"
    if plan.startswith("tf32x3"):
        # Roofline of the tensor kernels: the dense TF32 rate of the tensor
        # cores at the SM clock of the timed region (ncu's per-clock rate of
        # the TF32 tensor-op counter), in fp32 work: each fp32 product is
        # 3 TF32 products. The measured bf16 burst scaled by the nominal
        # TF32/BF16 ratio is given beside it as context only: that burst
        # ran under the power cap at a much lower clock than these kernels
        # do, so it is not a ceiling for them.
        hw_peak = sms * TF32_OPS_PER_CLK_PER_SM * clock_mhz * 1e6 / 1e12
        eff_peak = hw_peak / TF32X3_PRODUCTS
        bf16, src = measured_bf16_tflops()
        tf32_from_bf16 = bf16 * TF32_PER_BF16
        roof = {"bound": "tensor", "achieved": tflops, "peak": eff_peak,
                "unit": "TFLOP/s", "frac": tflops / eff_peak,
                "traffic": recorded_traffic(kernel, w["name"]),
                "kernel": kernel,
                "peak_basis": ("dense TF32 tensor rate %d SMs x %d ops/clk "
                               "(ncu) x %.0f MHz (median SM clock inside the "
                               "timed region) = %.1f TFLOP/s of TF32; 3 TF32 "
                               "products per fp32 product -> %.1f TFLOP/s of "
                               "fp32 work" % (sms, TF32_OPS_PER_CLK_PER_SM,
                                              clock_mhz, hw_peak, eff_peak)),
                "tensor_tflops": TF32X3_PRODUCTS * tflops,
                "tensor_peak": hw_peak,
                "context_bf16_derived": {
                    "peak": tf32_from_bf16 / TF32X3_PRODUCTS,
                    "frac": tflops / (tf32_from_bf16 / TF32X3_PRODUCTS),
                    "basis": ("bf16 burst %.1f TFLOP/s (%s, "
                              "MEASURED_PEAKS.json, taken under the power "
                              "cap) x nominal TF32/BF16 ratio 1.1/2.25 / 3 "
                              "products; context, not a ceiling"
                              % (bf16, src))}}
    elif plan in ("gemv_row", "gemv_col"):
        # a stream over the matrix: bound by HBM bandwidth
        hbm, src = measured_hbm_gbs()
        gbs = 4 * (M * K + K * N + M * N) / (ms_step * 1e-3) / 1e9
        # Context: PyTorch's own reduction over the same matrix, timed the
        # same way (flush, events): another kernel that streams these bytes
        # once from a cold L2, launch and ramp included.
        X = A if M > 1 else B
        sink = torch.empty((), device="cuda")
        rms = time_steps(lambda: torch.sum(X, dim=(0, 1), out=sink), flush,
                         stream, max(5, min(args.steps, 100)), 3)
        r_ms = statistics.median(rms)
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                "frac": gbs / hbm,
                "traffic": recorded_traffic(kernel, w["name"]),
                "kernel": kernel,
                "peak_basis": "HBM copy bandwidth %.1f GB/s (%s, "
                              "MEASURED_PEAKS.json); algorithmic bytes "
                              "4(MK + KN + MN)" % (hbm, src),
                "context_torch_sum": {
                    "kernel": "torch.sum over the same %d x %d matrix"
                              % tuple(X.shape),
                    "ms_median": r_ms,
                    "gbs": 4 * X.numel() / (r_ms * 1e-3) / 1e9,
                    "gemv_ms_median": statistics.median(ms),
                    "basis": "same flush and event timing as the product; "
                             "a library reduction over the same bytes, "
                             "for comparison"}}
    else:
        roof = {"bound": "alu", "achieved": tflops,
                "peak": ffma_peak_at(clock_mhz), "unit": "TFLOP/s",
                "frac": tflops / ffma_peak_at(clock_mhz),
                "traffic": recorded_traffic(kernel, w["name"]),
                "kernel": kernel,
                "peak_basis": ffma_basis(clock_mhz, "the timed region")}

    # The CUDA-core FFMA kernel on the same inputs, timed the same way, with
    # its own clock record: its roofline is the FP32 FMA peak at the clock
    # seen while it ran.
    ffma = None
    if plan.startswith("tf32x3") and not args.no_ffma:
        prev = dfm.sgemm_set_math_mode("ffma")
        try:
            ffma_path = dfm.sgemm_plan_ex(op_a, op_b, M, N, K, lda, ldb, ldc,
                                          pA, pB, pC)
            with ClockSampler(dev) as fclocks:
                fms = time_steps(step, flush, stream,
                                 max(5, min(args.steps, 100)), args.warmup,
                                 fclocks)
        finally:
            dfm.sgemm_set_math_mode(prev)
        st, site = dfm.sgemm_watchdog_status()
        if st != 0:
            raise RuntimeError("watchdog fired in the FFMA leg (site %d)"
                               % site)
        fclk = fclocks.summary()
        f_mhz = fclk["sm_mhz"] or (fclk["sm_max_mhz"] or 2070.0)
        f_ms = reduce_max(sum(fms) / len(fms), world)
        f_tflops = flops(M, N, K) / (f_ms * 1e-3) / 1e12
        ffma = {"path": ffma_path, "kernel": "k_tiled_tma",
                "value": job_tflops(flops(M, N, K), f_ms, world),
                "unit": "TFLOP/s", "ms_per_step": f_ms,
                "ms_min": min(fms), "ms_median": statistics.median(fms),
                "steps": len(fms),
                "peak": ffma_peak_at(f_mhz),
                "frac_of_ffma_peak": f_tflops / ffma_peak_at(f_mhz),
                "peak_basis": ffma_basis(f_mhz, "this leg's timed region"),
                "cycles_per_step_M": f_ms * 1e-3 * f_mhz,
                "clocks": {"sm_mhz": fclk["sm_mhz"],
                           "sm_mhz_min": fclk.get("sm_mhz_min"),
                           "sm_max_mhz": fclk["sm_max_mhz"],
                           "reasons": fclk["reasons"],
                           "samples": fclk["samples"],
                           "samples_in_region": fclk.get("samples_in_region"),
                           "power_w_max": fclk.get("power_w_max")},
                "traffic": recorded_traffic("k_tiled_tma", w["name"])}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": config_of(w, extra={
            "path": plan, "sms": sms, "gpu": props.name,
            "arithmetic": ("3xTF32 tensor-core products (hi/lo split), fp32 "
                           "accumulation" if plan.startswith("tf32x3") else
                           "fp32 fused multiply-add on CUDA cores"),
            "l2": "flushed before every step (a 256 MiB device write, then "
                  "a 256 MiB read so no dirty lines remain; outside the timed "
                  "events)",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "layout": ("row-major, dense leading dimensions"
                       if not (args.pad or args.offset) else
                       "row-major, lda = K + %d, ldb = ldc = N + %d, bases "
                       "shifted by %d floats" % (args.pad, args.pad,
                                                 args.offset))
                      + ("" if args.ops == "NN" else
                         "; operands %s (A stored %s, B stored %s)"
                         % (args.ops, "K x M" if op_a == "T" else "M x K",
                            "N x K" if op_b == "T" else "K x N"))}),
        "roofline": roof,
        "ffma_kernel": ffma,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_mhz_min": clk.get("sm_mhz_min"),
                   "sm_max_mhz": clk["sm_max_mhz"],
                   "reasons": clk["reasons"], "samples": clk["samples"],
                   "samples_in_region": clk.get("samples_in_region"),
                   "basis": clk.get("basis"),
                   "power_w_max": clk.get("power_w_max")},
        "cycles_per_step_M": ms_step * 1e-3 * clock_mhz,
        "e2e": {"value": job_tflops(flops(M, N, K), e2e_ms, world),
                "unit": "TFLOP/s",
                "h2d_bytes_per_step": 4 * (M * K + K * N),
                "d2h_bytes_per_step": 4 * M * N,
                "api": "sgemm_host (pinned host buffers, 2-D async copies "
                       "on the stream)",
                "path": e2e_plan},
        "gpu_launches": launches,
        "gpu_launches_basis": {"per_step": launches / args.steps,
                               "how": "the library's own count of the kernel "
                                      "launches it issued (sgemm_launch_count) "
                                      "across the timed region"},
        "ms_min": min(ms), "ms_median": statistics.median(ms),
    }
    if plan in ("tiled_tma", "tiled_ldg"):
        line["pct_of_ffma_peak"] = 100.0 * roof["frac"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows, sec, threads = cpu_oracle_rate(M, N, K, w["kind"],
                                                   w["seed"])
        line["cpu_baseline"] = {
            "value": rate, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d of %d rows of C (fp64 oracle, %.1f s)" % (
                rows, M, sec)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None,
                   help="workload name (default: the 4096^3 headline)")
    p.add_argument("--shape", default=None,
                   help="MxNxK: an ad-hoc shape (uniform values, seed 3) "
                        "instead of a named workload")
    p.add_argument("--path", default="auto",
                   help="force a kernel path (auto, tiled_tma, tiled_ldg, ...)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--pad", type=int, default=0,
                   help="extra floats per row of A, B and C (leading "
                        "dimensions K + pad, N + pad)")
    p.add_argument("--offset", type=int, default=0,
                   help="shift the bases of A, B and C by this many floats")
    p.add_argument("--ops", default="NN", choices=["NN", "NT", "TN", "TT"],
                   help="A / B as stored (N) or stored transposed (T), run "
                        "through sgemm_ex")
    p.add_argument("--no-ffma", action="store_true",
                   help="skip timing the CUDA-core kernel beside the tensor one")
    args = p.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps
    from matgen import workloads
    if args.shape:
        M, N, K = (int(x) for x in args.shape.lower().split("x"))
        w = dict(name="shape_%dx%dx%d" % (M, N, K), M=M, N=N, K=K,
                 kind="uniform", seed=3)
    else:
        w = workloads.by_name(args.workload) if args.workload else dict(
            workloads.HEADLINE)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
