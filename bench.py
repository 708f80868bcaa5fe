"""Benchmark of the dense row-major GEMM hot path on GB300.

One step is one pass of the whole hot path over the 4096^3 workloads: the
FP32 SIMT SGEMM (A, B uniform[-1,1], seed 2) and the FP16 tcgen05 GEMM
(A, B normal(0,1)/sqrt(K) cast to FP16, seed 3), both M = N = K = 4096,
called through the library's C ABI.  Throughput is 2*M*N*K per GEMM over
CUDA-event time on the launching stream; L2 is flushed (a 512 MiB write)
before each GEMM, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--alpha a --beta b]

--alpha/--beta time the scaled form C := alpha * A.B + beta * C through the
*_ex entry points instead (the fused epilogue; beta != 0 reads the old C).

--impl reference times the CPU oracle (plain FP64 triple loop) on a bounded
row sample of the same workloads.  Under torchrun (N > 1) every rank runs
an independent replica on its own GPU (the path has no exchange step).
"""
from __future__ import annotations

import argparse
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

import numpy as np
import torch

import workloads

METRIC = "TFLOP/s (2MNK/t) and % of FP32-FFMA / dense FP16 tensor peak at 4096³"
UNIT = "TFLOP/s"
STEP_WORKLOADS = ("f32_4096", "f16_4096")
SMS_NOMINAL = 152
FP32_LANES_PER_SM = 128          # FFMA lanes per SM (4 SM sub-partitions x 32)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}


# ------------------------------------------------------------ environment

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        busy = [s for s in sm if smax is None or s >= 0.3 * smax] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ multi-rank

def max_over_ranks(value: float, ws: int, device) -> float:
    """The largest `value` over all ranks (every rank gets it); the value
    itself with one rank.  The replicas' step time is the slowest rank's."""
    if ws <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(step_flops: float, step_ms: float, ws: int) -> float:
    """Whole-job throughput: every one of the ws replicas does step_flops per
    step, and a step of the job takes the slowest rank's step_ms."""
    return ws * step_flops / (step_ms * 1e-3) / 1e12


# ------------------------------------------------------------ measured peaks and extra legs

def ffma_probe(dg, dev, stream, sms, seconds=0.15):
    """Measured FP32 FFMA throughput (the SGEMM roofline's denominator):
    the library's register-only fma.rn.f32x2 probe on every SM, timed with
    CUDA events on the launching stream, with the SM clock sampled while it
    runs.  Returns TFLOP/s, the median clock and TFLOP/s per GHz."""
    blocks = 4 * sms
    out = torch.empty(blocks * dg.gemm_probe_ffma_threads(), dtype=torch.float32, device=dev)
    iters = 20000
    st, fl = dg.gemm_probe_ffma(blocks, iters, out.data_ptr(), stream.cuda_stream)
    if st != dg.GEMM_OK:
        raise RuntimeError(f"ffma probe: {dg.status_string(st)}")
    torch.cuda.synchronize(dev)
    # Size one launch to ~seconds / 5 from a first timing.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        dg.gemm_probe_ffma(blocks, iters, out.data_ptr(), stream.cuda_stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    iters = max(iters, int(iters * (seconds / 5) / max(e0.elapsed_time(e1) * 1e-3, 1e-6)))
    sampler = ClockSampler(dev.index)
    sampler.start()
    times = []
    with torch.cuda.stream(stream):
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            st, fl = dg.gemm_probe_ffma(blocks, iters, out.data_ptr(), stream.cuda_stream)
            e1.record(stream)
            times.append((e0, e1))
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = statistics.median(a.elapsed_time(b) for a, b in times)
    tf = fl / (ms * 1e-3) / 1e12
    mhz = clocks["sm_mhz"] if clocks else None
    return {"tflops": round(tf, 2), "ms_per_launch": round(ms, 3), "flops_per_launch": fl,
            "launch": f"{blocks} CTAs x {dg.gemm_probe_ffma_threads()} threads, 16 independent "
                      f"fma.rn.f32x2 chains x {iters} iterations per thread",
            "sm_mhz": mhz, "tflops_per_ghz": round(tf / (mhz / 1000.0), 3) if mhz else None,
            "clocks": clocks}


# The scope's configurations (the seeded workloads), with the oracle rows
# checked per configuration: all rows where the oracle is quick, else a
# deterministic sample (first and last rows, both sides of tile edges,
# random rows).
CONFIG_ROWS = {"f32_256": None, "f32_256_int": None, "f32_2048": 128, "f32_4096": 128,
               "f16_4096": 128, "bf16_8192": 96, "f32_edge": None, "bf16_edge": 256}
TOLERANCE = {"f32": 1e-5, "f16": 2e-3, "bf16": 1e-2}


def run_configs(dg, dev, stream, sms, ffma_peak, ffma_measured, tensor_peak, peaks_src,
                reps=15, check=True):
    """Every configuration: CUDA-event time per call (L2 flushed before
    each, median of `reps` after 3 warm-ups), TFLOP/s, the fraction of its
    roofline, and the oracle comparison on sampled rows (bit-exact for the
    integer-valued copy)."""
    import oracle
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    out = {}
    for name in CONFIG_ROWS:
        w = workloads.WORKLOADS[name]
        A_cpu, B_cpu = workloads.make(w)
        A, B = A_cpu.to(dev), B_cpu.to(dev)
        C = torch.full((w.M, w.N), float("nan"), dtype=A.dtype, device=dev)
        times = []
        with torch.cuda.stream(stream):
            for i in range(reps + 3):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                st = dg.gemm(w.dtype, w.M, w.N, w.K, A.data_ptr(), w.K, B.data_ptr(), w.N,
                             C.data_ptr(), w.N, stream.cuda_stream)
                e1.record(stream)
                if st != dg.GEMM_OK:
                    raise RuntimeError(f"{name}: {dg.status_string(st)}")
                if i >= 3:
                    times.append((e0, e1))
        st, bits = dg.gemm_device_check(stream.cuda_stream)
        if st != dg.GEMM_OK:
            raise RuntimeError(f"{name}: device check {dg.status_string(st)} ({bits:#x})")
        ms = statistics.median(a.elapsed_time(b) for a, b in times)
        tf = w.flops / (ms * 1e-3) / 1e12
        _, plan = dg.gemm_plan(w.dtype, w.M, w.N, w.K, A.data_ptr(), w.K, B.data_ptr(), w.N,
                               C.data_ptr(), w.N, sms)
        entry = {"shape": [w.M, w.N, w.K], "dtype": w.dtype, "inputs": f"{w.dist} seed {w.seed}",
                 "ms_median": round(ms, 4), "tflops": round(tf, 2)}
        if w.dtype == "f32":
            entry.update({"peak_tflops": round(ffma_peak, 1), "frac_of_peak": round(tf / ffma_peak, 4),
                          "peak_kind": "FFMA, derived: SMs x 128 lanes x 2 x max SM clock"})
            if ffma_measured:
                entry["frac_of_measured_ffma"] = round(tf / ffma_measured, 4)
        else:
            entry.update({"peak_tflops": round(tensor_peak, 1), "frac_of_peak": round(tf / tensor_peak, 4),
                          "peak_kind": f"dense BF16/FP16 tensor, {peaks_src} burst"})
        entry["plan"] = {"path": plan.path, "ctas": plan.ctas, "cluster_ctas": plan.cluster_ctas,
                         "split_tiles": plan.split_tiles, "stream_k": plan.split_in_k,
                         "splitk_slices": plan.splitk_slices}
        if check:
            nrows = CONFIG_ROWS[name]
            rows = None if nrows is None else workloads.sample_rows(w.M, nrows, seed=w.seed)
            ref, S = oracle.gemm(w.dtype, workloads.to_numpy_bits(A_cpu),
                                 workloads.to_numpy_bits(B_cpu), rows=rows)
            got = C.float().cpu().numpy().astype(np.float64)
            if rows is not None:
                got = got[rows]
            if w.dist == "int":
                exact = bool(np.array_equal(got, ref))
                entry["parity_on_sample"] = {"rows": int(got.shape[0]), "bit_exact": exact,
                                             "pass": exact}
            else:
                err, idx, bad = oracle.normalized_error(got, ref, S)
                entry["parity_on_sample"] = {"rows": int(got.shape[0]),
                                             "max_normalised_error": err,
                                             "tolerance": TOLERANCE[w.dtype],
                                             "pass": bool(err <= TOLERANCE[w.dtype] and bad == 0)}
        out[name] = entry
        del A, B, C
    return out


def run_sustained(dg, cases, dev, stream, seconds=1.0):
    """Each GEMM of the step back to back for about `seconds` (no L2 flush
    in between), timed with CUDA events around the whole run, with the SM
    clock sampled throughout: TFLOP/s at the clock the power cap settles at,
    and TFLOP/s per GHz, which compares runs taken at different clocks."""
    out = {}
    for c in cases:
        w = c["w"]

        def call():
            st = dg.gemm(w.dtype, w.M, w.N, w.K, c["A"].data_ptr(), w.K, c["B"].data_ptr(),
                         w.N, c["C"].data_ptr(), w.N, stream.cuda_stream)
            if st != dg.GEMM_OK:
                raise RuntimeError(f"{w.name}: {dg.status_string(st)}")
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(5):
                call()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        n = max(10, int(seconds / max(e0.elapsed_time(e1) * 1e-3 / 5, 1e-6)))
        sampler = ClockSampler(dev.index)
        sampler.start()
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                call()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        clocks = sampler.stop()
        st, bits = dg.gemm_device_check(stream.cuda_stream)
        if st != dg.GEMM_OK:
            raise RuntimeError(f"{w.name}: device check {dg.status_string(st)} ({bits:#x})")
        ms = e0.elapsed_time(e1)
        tf = n * w.flops / (ms * 1e-3) / 1e12
        mhz = clocks["sm_mhz"] if clocks else None
        out[w.name] = {"calls": n, "seconds": round(ms / 1000, 3), "tflops": round(tf, 2),
                       "sm_mhz": mhz,
                       "tflops_per_ghz": round(tf / (mhz / 1000.0), 2) if mhz else None,
                       "clocks": clocks}
    return out


# ------------------------------------------------------------ our arm

def run_ours(args, ws, rank, local):
    import dense_gemm_major_gb300 as dg
    dg.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    peaks, peaks_src = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count

    # Inputs, resident in HBM before timing.
    cases = []
    for name in args.workloads:
        w = workloads.WORKLOADS[name]
        A, B = workloads.make(w)
        # The old C (read only when beta != 0): uniform[-1, 1], seed 7.
        C_cpu = (torch.rand((w.M, w.N), generator=torch.Generator().manual_seed(7)) * 2 - 1
                 ).to(A.dtype)
        cases.append({"w": w, "A_cpu": A, "B_cpu": B, "C_cpu": C_cpu, "A": A.to(dev),
                      "B": B.to(dev), "C": C_cpu.to(dev)})
    scaled = args.alpha != 1.0 or args.beta != 0.0
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    # This library's kernel launches per step: one per GEMM, plus the
    # re-pitch launch of an FP32 GEMM with an operand TMA cannot address
    # (the step's operands are row-major: both copies are one launch) and
    # the reduction launch of a split-K GEMM (none when an FP32 tile's
    # k-slices combine within a cluster).
    launches_per_step = 0
    for c in cases:
        w = c["w"]
        _, plan = dg.gemm_plan_ex(w.dtype, w.M, w.N, w.K, args.alpha, c["A"].data_ptr(), w.K,
                                  c["B"].data_ptr(), w.N, args.beta, c["C"].data_ptr(), w.N,
                                  sms)
        if plan.path == dg.PATH_NOOP:
            continue
        reduce = plan.splitk_slices > 1 and not (w.dtype == "f32" and plan.cluster_ctas > 1)
        launches_per_step += 1 + (1 if reduce else 0) + (1 if plan.pack else 0)

    def launch(c, s=sptr):
        w = c["w"]
        if scaled:
            st = dg.gemm_ex(w.dtype, w.M, w.N, w.K, args.alpha, c["A"].data_ptr(), w.K,
                            c["B"].data_ptr(), w.N, args.beta, c["C"].data_ptr(), w.N, s)
        else:
            st = dg.gemm(w.dtype, w.M, w.N, w.K, c["A"].data_ptr(), w.K, c["B"].data_ptr(),
                         w.N, c["C"].data_ptr(), w.N, s)
        if st != dg.GEMM_OK:
            raise RuntimeError(f"{w.name}: {dg.status_string(st)}")

    # Warm-up, then a device fault check.
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for c in cases:
                flush.zero_()
                launch(c)
    st, bits = dg.gemm_device_check(sptr)
    if st != dg.GEMM_OK:
        raise RuntimeError(f"device check after warm-up: {dg.status_string(st)} ({bits:#x})")

    # Timed region: K steps; events around each GEMM on the launching stream.
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in cases] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            for i, c in enumerate(cases):
                flush.zero_()
                ev[k][i][0].record(stream)
                launch(c)
                ev[k][i][1].record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    st, bits = dg.gemm_device_check(sptr)
    if st != dg.GEMM_OK:
        raise RuntimeError(f"device check after timing: {dg.status_string(st)} ({bits:#x})")

    per_ms = [[ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps)]
              for i in range(len(cases))]
    step_ms = max_over_ranks(sum(sum(x) for x in per_ms) / args.steps, ws, dev)
    step_flops = sum(c["w"].flops for c in cases)
    value = job_tflops(step_flops, step_ms, ws)

    # Per-kernel figures and rooflines.
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    ffma_peak = sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    tensor_peak = float(peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]))   # FP16 rate = BF16 rate
    per_kernel = {}
    for i, c in enumerate(cases):
        w = c["w"]
        avg = sum(per_ms[i]) / len(per_ms[i])
        tf = w.flops / (avg * 1e-3) / 1e12
        peak = ffma_peak if w.dtype == "f32" else tensor_peak
        per_kernel[w.name] = {
            "shape": [w.M, w.N, w.K], "ms_avg": round(avg, 4), "ms_median": round(statistics.median(per_ms[i]), 4),
            "tflops": round(tf, 2), "peak_tflops": round(peak, 1),
            "frac_of_peak": round(tf / peak, 4),
            "peak_kind": ("FFMA: %d SMs x %d lanes x 2 x %.0f MHz" % (sms, FP32_LANES_PER_SM, sm_max))
            if w.dtype == "f32" else f"dense BF16/FP16 tensor, {peaks_src} burst",
        }
    share = {n: sum(per_ms[i]) for i, n in enumerate(per_kernel)}
    dominant = max(share, key=share.get)
    dk = per_kernel[dominant]
    traffic = load_traffic(dominant)
    roofline = {"bound": "alu" if dominant.startswith("f32") else "tensor",
                "achieved": dk["tflops"], "peak": dk["peak_tflops"], "unit": "TFLOP/s",
                "frac": dk["frac_of_peak"], "traffic": traffic,
                "kernel": dominant, "peak_source": "derived from unit counts and max SM clock "
                "(152 SMs x 128 FFMA lanes x 2 x sm_max_mhz); the FFMA probe's measured rate is "
                "in measured_peak" if dominant.startswith("f32")
                else f"{peaks_src} (MEASURED_PEAKS.json bf16_tflops)"}
    roofline_tensor = None
    tname = next((n for n in per_kernel if not n.startswith("f32")), None)
    if tname is not None:
        tk = per_kernel[tname]
        roofline_tensor = {"bound": "tensor", "achieved": tk["tflops"], "peak": tk["peak_tflops"],
                           "unit": "TFLOP/s", "frac": tk["frac_of_peak"],
                           "traffic": load_traffic(tname), "kernel": tname,
                           "peak_source": f"{peaks_src} bf16_tflops (FP16 dense rate equals BF16)"}

    # End to end through the C ABI with host buffers.
    e2e = None if args.no_e2e else run_e2e(dg, cases, dev, stream, args)

    # The measured FFMA peak, every configuration, and the sustained leg.
    ffma = None if args.no_extra else ffma_probe(dg, dev, stream, sms)
    if ffma is not None:
        roofline["measured_peak"] = {"ffma_tflops": ffma["tflops"], "sm_mhz": ffma["sm_mhz"],
                                     "frac": round(roofline["achieved"] / ffma["tflops"], 4)
                                     if dominant.startswith("f32") else None,
                                     "source": "gemm_probe_ffma (fma.rn.f32x2, registers only)"}
    configs = None if args.no_extra else run_configs(
        dg, dev, stream, sms, ffma_peak, ffma["tflops"] if ffma else None, tensor_peak, peaks_src,
        check=not args.no_cpu_baseline)
    sustained = None if args.no_extra else run_sustained(dg, cases, dev, stream)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32+f16", "data": "synthetic",
        "config": {"workload": "SGEMM FP32 4096^3 (uniform[-1,1], seed 2) + GEMM FP16 4096^3 "
                               "(normal/sqrt(K), seed 3), row-major, lda=K, ldb=ldc=N",
                   "l2": "flushed (512 MiB write) before each GEMM, outside the timed events",
                   "parallelism": f"replicas{ws}",
                   "epilogue": {"alpha": args.alpha, "beta": args.beta}},
        "per_kernel": per_kernel, "roofline": roofline, "roofline_tensor": roofline_tensor,
        "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks, "device": {"name": props.name, "sms": sms},
    }
    if not args.no_extra:
        out["peaks"] = {"ffma": ffma, "tensor_bf16_burst": tensor_peak,
                        "tensor_source": f"{peaks_src} (MEASURED_PEAKS.json bf16_tflops)"}
        out["configs"] = configs
        out["sustained"] = sustained
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        if args.beta != 0.0:
            # One call on the seeded old C, so the sample check sees a single update.
            for c in cases:
                c["C"].copy_(c["C_cpu"])
                launch(c)
            torch.cuda.synchronize(dev)
        out["cpu_baseline"] = cpu_baseline(cases, args.cpu_seconds, check=True,
                                           alpha=args.alpha, beta=args.beta)
    return out


def run_e2e(dg, cases, dev, stream, args):
    """Same step through the public C ABI's host-memory entry (gemm_host)
    with A, B and C in pinned host memory: the host->device copies of A and
    B (and of the old C when beta != 0), the kernels and the device->host
    copy of C are all inside the timed events; gemm_host overlaps them
    block by block, and the step's GEMMs run on separate streams."""
    host = []
    for c in cases:
        host.append({"A": c["A_cpu"].pin_memory(), "B": c["B_cpu"].pin_memory(),
                     "C_in": c["C_cpu"].pin_memory(),
                     "C": torch.empty(c["C"].shape, dtype=c["C"].dtype).pin_memory()})
    read_c = args.beta != 0.0
    if read_c:
        # Each step reads the C the one before wrote (C := alpha A.B + beta C
        # stays bounded for |beta| < 1); it starts from the seeded old C.
        for h in host:
            h["C"].copy_(h["C_in"])
    h2d = sum(h["A"].numel() * h["A"].element_size() + h["B"].numel() * h["B"].element_size()
              + (h["C_in"].numel() * h["C_in"].element_size() if read_c else 0) for h in host)
    d2h = sum(h["C"].numel() * h["C"].element_size() for h in host)

    # The GEMMs of a step are independent problems: each goes on its own
    # stream (forked from and joined back to the timed stream), so one's
    # copies can overlap another's kernels.
    streams = [stream] + [torch.cuda.Stream(dev) for _ in cases[1:]]

    def step():
        fork = torch.cuda.Event()
        fork.record(stream)
        for c, h, s in zip(cases, host, streams):
            w = c["w"]
            s.wait_event(fork)
            st = dg.gemm_host(w.dtype, "N", "N", w.M, w.N, w.K, args.alpha, h["A"].data_ptr(),
                              w.K, h["B"].data_ptr(), w.N, args.beta, h["C"].data_ptr(), w.N,
                              s.cuda_stream)
            if st != dg.GEMM_OK:
                raise RuntimeError(dg.status_string(st))
        for s in streams[1:]:
            join = torch.cuda.Event()
            join.record(s)
            stream.wait_event(join)

    steps = max(3, min(args.steps, 10))
    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    flops = sum(c["w"].flops for c in cases)
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


KERNEL_SOURCES = {"f32": ("sgemm_simt.cuh", "sgemm_simt.cu"),
                  "f16": ("gemm_tc.cu", "gemm_tc2.cu", "tcgen05.cuh"),
                  "bf16": ("gemm_tc.cu", "gemm_tc2.cu", "tcgen05.cuh")}


def kernel_source_hash(workload_name):
    """SHA-256 of the kernel source a workload runs (with the shared headers)."""
    import hashlib
    dt = workloads.WORKLOADS[workload_name].dtype
    csrc = os.path.join(ROOT, "dense_gemm_major_gb300", "csrc")
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[dt] + ("ptx.cuh", "launch.h", "api.cu"):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(workload_name):
    """DRAM bytes (read + write) per launch from the committed ncu summary,
    or None when there is none or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f).get(workload_name)
    except (OSError, ValueError):
        return None
    if not d or d.get("kernel_sha") != kernel_source_hash(workload_name):
        return None
    return d.get("dram_bytes")


# ------------------------------------------------------------ CPU oracle

def cpu_baseline(cases, seconds, check=False, alpha=1.0, beta=0.0):
    """Time the oracle, as it stands, on a bounded row sample of each
    workload (rows chosen so the whole leg takes about `seconds`).  With
    check=True the sampled GPU rows are also compared with the oracle's
    alpha * A.B + beta * C_in (the case's "C" must hold one such call's
    result on the old C "C_cpu")."""
    import oracle
    from oracle import normalized_error
    tol = {"f32": 1e-5, "f16": 2e-3, "bf16": 1e-2}
    cores = oracle.num_threads()
    # Rate probe: a few rows per workload.
    budget = seconds / len(cases)
    total_flops, total_s, sample_desc, checks = 0, 0.0, [], {}
    for c in cases:
        w = c["w"]
        a = workloads.to_numpy_bits(c["A_cpu"])
        b = workloads.to_numpy_bits(c["B_cpu"])
        probe = np.arange(min(8, w.M), dtype=np.int64)
        t0 = time.perf_counter()
        oracle.gemm(w.dtype, a, b, rows=probe, with_scale=False)
        per_row = (time.perf_counter() - t0) / len(probe)
        nrows = int(max(len(probe), min(w.M, budget / max(per_row, 1e-9))))
        rows = np.sort(np.random.default_rng(w.seed).choice(w.M, size=nrows, replace=False))
        t0 = time.perf_counter()
        ref, S = oracle.gemm(w.dtype, a, b, rows=rows, with_scale=check)
        dt = time.perf_counter() - t0
        if check and (alpha != 1.0 or beta != 0.0):
            # Scaled reference for the check (outside the timed sample).
            c_in = workloads.to_numpy_bits(c["C_cpu"]) if beta != 0.0 else None
            ref, S = oracle.gemm_scaled(w.dtype, alpha, a, b, beta, c_in, rows=rows)
        fl = 2 * nrows * w.N * w.K
        total_flops += fl
        total_s += dt
        sample_desc.append(f"{nrows} of {w.M} rows of {w.name} ({fl / 1e9:.1f} GFLOP, {dt:.1f} s)")
        if check and "C" in c:
            got = c["C"].float().cpu().numpy()[rows].astype(np.float64)
            err, idx, bad = normalized_error(got, ref, S)
            checks[w.name] = {"rows": nrows, "max_normalised_error": err, "tolerance": tol[w.dtype],
                              "pass": bool(err <= tol[w.dtype] and bad == 0)}
    out = {"value": round(total_flops / total_s / 1e12, 6), "unit": UNIT, "cores": cores,
           "kind": "oracle", "sample": "; ".join(sample_desc),
           "seconds": round(total_s, 2)}
    if check:
        out["parity_on_sample"] = checks
    return out


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    cases = []
    for name in args.workloads:
        w = workloads.WORKLOADS[name]
        A, B = workloads.make(w)
        cases.append({"w": w, "A_cpu": A, "B_cpu": B})
    per_step = max(2.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(min(args.warmup, 1)):
        cpu_baseline(cases, min(per_step, 2.0))
    vals, secs = [], []
    for _ in range(args.steps):
        r = cpu_baseline(cases, per_step)
        vals.append(r["value"])
        secs.append(r["seconds"])
    value = statistics.median(vals)
    cb = {"value": value, "unit": UNIT, "cores": r["cores"], "kind": "oracle", "sample": r["sample"]}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1000 * statistics.median(secs), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "SGEMM FP32 4096^3 (uniform[-1,1], seed 2) + GEMM FP16 4096^3 "
                                   "(normal/sqrt(K), seed 3), row-major; CPU oracle on a row sample",
                       "parallelism": "host cores"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="time budget of the CPU oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the FFMA probe, the per-configuration table and the sustained leg")
    ap.add_argument("--alpha", type=float, default=1.0, help="scale of A.B (default 1)")
    ap.add_argument("--beta", type=float, default=0.0, help="scale of the old C (default 0)")
    ap.add_argument("--workloads", default=",".join(STEP_WORKLOADS),
                    help="comma-separated workload names (default: the 4096^3 step)")
    args = ap.parse_args()
    args.workloads = [x for x in args.workloads.split(",") if x]
    for n in args.workloads:
        if n not in workloads.WORKLOADS:
            ap.error(f"unknown workload {n}; known: {', '.join(workloads.WORKLOADS)}")
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    ws, rank, local = dist_env()
    if ws > 1 and args.impl == "ours":
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.impl == "reference":
        out = run_reference(args, ws, rank)
    else:
        out = run_ours(args, ws, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if ws > 1 and args.impl == "ours":
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
