#!/usr/bin/env python3
"""Benchmark of the dense GEMM library on one or more GB300 GPUs.

One step is one pass of the whole hot path over one batch of synthetic
input: the FP32 SGEMM 4096^3 (CUDA cores) followed by the BF16 GEMM 4096^3
(tcgen05 tensor cores, fp32 accumulate, bf16 out).  `--workload` selects a
single workload instead (see gemm_inputs/workloads.py).

Timing: W untimed warm-up steps, then K timed steps.  Before every step the
129 MB L2 is flushed, outside the timed events: a 256 MiB buffer is written
(evicting every line), then a second 256 MiB buffer is read, so that the
dirty lines the write leaves are written back before the step instead of
during it (measured on GB300: left dirty, their write-back slows a
bandwidth-bound kernel by 5-7 us, a cost of the flush, not of the kernel;
the workloads timed after the step also report the write-only flush).
Each kernel is bracketed by CUDA events on the stream it is launched on.
`value` = work of all ranks / the slowest rank's summed step time.  Prints
one JSON line (rank 0).  For context, after the timed region each kernel
also runs back to back without the flush (`kernels.*.warm_l2`).

`--impl reference` times the CPU oracle instead (the reference arm: the
plain double-precision triple loop, on the host cores), on a bounded sample
of rows of the same workload.

Multi-GPU: the GEMM is run as independent replicas, one per rank (no data
exchange); ranks only meet for a barrier and a max-reduction of times.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (BF16 tcgen05, FP32 SIMT) at 4096^3 and % of chip peak"
# The step's products, in launch order.  The BF16 product runs first, right
# after the L2 flush like every other timed call: behind the SGEMM it reads
# its operands while L2 writes back the SGEMM's 64 MiB of dirty C lines
# (measured on GB300: 83.8 against 80.9 us; the SGEMM takes 2.127 ms either
# way).
STEP_WORKLOADS = ("bf16_4096", "sgemm_4096")
FLUSH_BYTES = 256 << 20
WARM_REPS = 20  # back-to-back calls per kernel in the warm-L2 context pass
# L2-flushed calls timed for each workload outside the headline step
EXTRA_REPS = {"sgemm_256": 200, "bf16_mlp_8192x14336x4096": 20, "bf16_decode_64x8192x8192": 100}
# Before each step the GPU idles this many cycles (~100 us) while the host
# enqueues the step, so the host's launch overhead never shows up inside a
# kernel's event window; the idle time is outside the timed events.
HOST_AHEAD_CYCLES = 200_000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
# Published number for the same workload on other hardware (context only):
# FP32 SGEMM 4096^3, final hand-written version on an RTX 3090.
PAGE_SGEMM_4096_TFLOPS = 10.23
FP32_LANES_PER_SM = 128  # FP32 FMA units per Blackwell SM (4 partitions x 32)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--variant", default="plain",
                    help="operand layouts and fused epilogue of the extended entry points, "
                         "comma-separated: a layout nn|tn|nt|tt (t: that operand stored "
                         "transposed), 'bias' (N fp32 values), an activation relu|gelu; "
                         "'plain' = the plain entry points")
    ap.add_argument("--batch", type=int, default=1,
                    help="run each workload as a strided batch of this many products "
                         "(gemm_batched, one launch)")
    ap.add_argument("--shape", default=None, metavar="MxNxK",
                    help="override the workload's M, N, K (same distributions)")
    ap.add_argument("--config", action="append", default=[], metavar="KEY=VALUE",
                    help="library tuning knob (gemm_set_config), may repeat")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads (256^3, MLP and decode shapes) that the "
                         "default step run also times and checks after its timed region")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the oracle comparison of the timed outputs")
    ap.add_argument("--no-integer-pass", action="store_true",
                    help="skip the bit-exact integer-operand pass of the parity check")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workloads_for(name):
    from gemm_inputs.workloads import WORKLOADS

    if name == "step":
        return [WORKLOADS[n] for n in STEP_WORKLOADS]
    if name not in WORKLOADS:
        raise SystemExit(f"unknown workload {name!r}; choose step or one of {list(WORKLOADS)}")
    return [WORKLOADS[name]]


# ---------------------------------------------------------------- distributed

class Dist:
    def __init__(self, gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            backend = "nccl" if _cuda_ok() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist
        self.gpus = gpus

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        dev = "cuda" if _cuda_ok() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        dev = "cuda" if _cuda_ok() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def _cuda_ok():
    import torch

    return torch.cuda.is_available()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"gemm_bench_clocks_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1])]
        smax = max((num(r[2]) for r in rows if num(r[2])), default=None)
        power = [num(r[3]) for r in rows if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if smax and s > 0.3 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": smax, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- oracle timing

def _sample_operands(w, rows, B_cache):
    if w.name not in B_cache:
        B_cache[w.name] = w.operands(rows=slice(0, 1))[1]
    A, _, C = w.operands(rows=slice(0, rows))
    return A, B_cache[w.name], C


def oracle_sample_time(workloads, seconds_target, operands=None, keep=False):
    """Times the CPU oracle (all host threads) on the leading rows of each
    workload, with the row count chosen from a one-row-per-thread
    calibration so the sample takes about seconds_target (at most all M
    rows).  `operands` maps a workload name to its full (A, B, C) host
    arrays (else they are drawn here).  Returns (flops, seconds, rows,
    threads, results); results maps each name to the oracle's double
    product of those rows when `keep` is set."""
    import oracle

    oracle.build()
    threads = oracle.default_threads()
    max_rows = min(w.M for w in workloads)
    B_cache = {}

    def ops_for(rows):
        out = []
        for w in workloads:
            if operands is not None and w.name in operands:
                A, B, C = operands[w.name]
                out.append((w, A[:rows], B, None if C is None else C[:rows]))
            else:
                out.append((w, *_sample_operands(w, rows, B_cache)))
        return out

    def timed(rows):
        ops = ops_for(rows)
        res = {}
        t0 = time.perf_counter()
        for w, A, B, C in ops:
            res[w.name] = oracle.gemm(A, B, C, alpha=w.alpha, beta=w.beta, threads=threads)
        return time.perf_counter() - t0, res

    cal_rows = min(threads, max_rows)
    t_cal, res = timed(cal_rows)
    rows = int(cal_rows * seconds_target / max(t_cal, 1e-6))
    rows = max(cal_rows, min(max_rows, (rows // cal_rows) * cal_rows))
    if rows != cal_rows:
        dt, res = timed(rows)
    else:
        dt = t_cal
    flops = sum(2 * rows * w.N * w.K for w in workloads)
    return flops, dt, rows, threads, (res if keep else None)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine() or "unknown"


def parity_random(w, got, ref):
    """Elementwise comparison of a GPU output (uint16 bf16 bits or float32)
    with the oracle's double result under the workload's tolerance: FP32
    |C - C_ref| <= 1e-5 K, BF16 |C - C_ref| <= 2^-7 |C_ref| + 1e-2."""
    import numpy as np

    import gemm_inputs as gi

    gv = (gi.bf16_bits_to_f32(got) if w.out == "bf16" else got).astype(np.float64)
    err = np.abs(gv - ref)
    if w.dtype == "f32":
        tol = np.full(1, 1e-5 * w.K)
        tol_s = f"max|C - C_ref| <= 1e-5*K = {1e-5 * w.K:g}"
    else:
        tol = (2.0 ** -7) * np.abs(ref) + 1e-2
        tol_s = "|C - C_ref| <= 2^-7 |C_ref| + 1e-2 elementwise"
    bad = (err > tol) | ~np.isfinite(gv)
    big = np.abs(ref) >= 1e-2  # relative error where the absolute floor does not dominate
    rel = err[big] / np.abs(ref[big])
    return {"compared": int(gv.size), "rows": int(gv.shape[0]),
            "max_abs_err": float(np.max(err)) if err.size else 0.0,
            "max_rel_err": float(np.max(rel)) if rel.size else 0.0,
            "violations": int(bad.sum()), "tolerance": tol_s}


def parity_integer(w, got, ref):
    """Bit-exact comparison of a GPU output on {-2..2} operands with the
    oracle's double result rounded once to the output type."""
    import oracle

    want = oracle.round_bf16(ref) if w.out == "bf16" else oracle.round_f32(ref)
    return {"compared": int(got.size), "mismatches": int((got != want).sum()),
            "rule": "bit-exact against the oracle rounded once to the output type"}


def run_reference(args, dist):
    workloads = workloads_for(args.workload)
    if dist.rank != 0:
        return 0
    import oracle

    oracle.build()
    threads = oracle.default_threads()
    # bounded sample: about five times --cpu-seconds of oracle work over all
    # steps (a minute by default), at least a few milliseconds per step
    per_step_target = max(0.005, min(60.0, 5.0 * args.cpu_seconds) /
                          max(1, args.steps + args.warmup))
    _flops, _dt, rows, _threads, _res = oracle_sample_time(workloads, per_step_target)
    B_cache = {}
    inputs = [(w, *_sample_operands(w, rows, B_cache)) for w in workloads]

    def step():
        for w, A, B, C in inputs:
            oracle.gemm(A, B, C, alpha=w.alpha, beta=w.beta, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    flops = args.steps * sum(2 * rows * w.N * w.K for w in workloads)
    value = flops / dt / 1e12
    sample = (f"leading {rows} rows of each of {', '.join(w.name for w in workloads)} "
              f"(full K and N), double-precision triple loop on {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(workloads, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

def config_block(workloads, args):
    name = "+".join(w.name for w in workloads)
    return {
        "workload": name,
        "shapes": {w.name: {"M": w.M, "N": w.N, "K": w.K, "in": w.dtype, "out": w.out,
                            "alpha": w.alpha, "beta": w.beta, "dist": w.description}
                   for w in workloads},
        "layout": "row-major A (MxK), B (KxN), C (MxN), contiguous",
        "l2": ("flushed before every step (outside the timed events): a 256 MiB buffer written, "
               "then a second 256 MiB buffer read, so no dirty line is left to write back"),
        "host_ahead": "the GPU idles ~100 us before each step (outside the timed events) so "
                      "kernel events exclude host launch overhead",
        "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU",
        "variant": getattr(args, "variant", "plain"),
        "batch": getattr(args, "batch", 1),
        "library_config": list(getattr(args, "config", [])),
    }


def kernel_source_hash(w):
    """Hash of the kernel's source code with comments and whitespace runs
    removed, so that a comment edit keeps the recorded traffic valid and
    any code edit invalidates it."""
    fname = "sgemm_tma.cu" if w.dtype == "f32" else "gemm_bf16_tc.cu"
    path = os.path.join(ROOT, "dense_gemm_02_gb300", "csrc", fname)
    with open(path, encoding="utf-8") as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256(" ".join(src.split()).encode()).hexdigest()[:16]


def kernel_name(w):
    """The kernel the library launches for this workload (as profiled)."""
    if w.dtype == "f32":
        return "sgemm_tma_kernel"
    return "bf16_tc2_kernel" if w.M > 128 and w.M * w.N >= 2 * 152 * 128 * 256 else "bf16_tc_kernel"


def recorded_traffic(w):
    """DRAM bytes per launch from a committed ncu capture of this exact
    kernel source, else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(w.name)
    if not rec or rec.get("source_sha256_16") != kernel_source_hash(w):
        return None
    return rec.get("dram_bytes_per_launch")


def parse_variant(spec):
    """(trans_a, trans_b, bias, act) of a --variant string."""
    ta = tb = False
    bias, act = False, "none"
    for tok in [t for t in spec.split(",") if t and t != "plain"]:
        if tok in ("nn", "tn", "nt", "tt"):
            ta, tb = tok[0] == "t", tok[1] == "t"
        elif tok == "bias":
            bias = True
        elif tok in ("relu", "gelu"):
            act = tok
        else:
            raise SystemExit(f"unknown --variant item {tok!r}")
    return ta, tb, bias, act


def run_ours(args, dist):
    import torch

    import dense_gemm_02_gb300 as g
    from dense_gemm_02_gb300 import _build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (use --impl reference for the CPU oracle)")
    torch.cuda.set_device(dist.local_rank)
    _build.build()
    g.binding.lib()
    for kv in args.config:
        key, val = kv.split("=", 1)
        g.set_config(key, int(val))
    import dataclasses

    import numpy as np

    import gemm_inputs as gi

    workloads = workloads_for(args.workload)
    if args.shape:
        M, N, K = (int(x) for x in args.shape.lower().split("x"))
        workloads = [dataclasses.replace(w, M=M, N=N, K=K, name=f"{w.name}@{M}x{N}x{K}")
                     for w in workloads]
    nb = max(1, args.batch)
    v_ta, v_tb, v_bias, v_act = parse_variant(args.variant)
    extended = args.variant != "plain" or nb > 1
    if extended:
        args.no_e2e = True  # the host-buffer API runs the plain entry points
    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(dist.local_rank)
    sms = props.multi_processor_count

    # ---- inputs resident in HBM
    dev_ops = []
    host_ops = []
    host_np = {}  # name -> (A, B, C) host arrays of a single product, for the parity check
    for w in workloads:
        A, B, C = w.operands()
        if nb == 1:
            host_np[w.name] = (A, B, C)
        if nb > 1:  # matrices 0..nb-1 of a strided batch, stacked
            ops = [w.batch_operands(i) for i in range(nb)]
            A = np.stack([o[0] for o in ops])
            B = np.stack([o[1] for o in ops])
            C = np.stack([o[2] for o in ops]) if ops[0][2] is not None else None
        if w.dtype == "f32":
            hA, hB = torch.from_numpy(A), torch.from_numpy(B)
        else:
            hA = torch.from_numpy(A.view("int16")).view(torch.bfloat16)
            hB = torch.from_numpy(B.view("int16")).view(torch.bfloat16)
        out_dt = torch.float32 if w.out == "f32" else torch.bfloat16
        if C is not None:
            hC = (torch.from_numpy(C) if w.out == "f32"
                  else torch.from_numpy(C.view("int16")).view(torch.bfloat16))
        else:
            hC = None
        dA, dB = hA.cuda(), hB.cuda()
        # Transposed storage: the same logical operand, held K x M (or N x
        # K) row-major; the library reads that layout in place.
        if v_ta:
            dA = dA.transpose(-1, -2).contiguous().transpose(-1, -2)
        if v_tb:
            dB = dB.transpose(-1, -2).contiguous().transpose(-1, -2)
        cshape = (nb, w.M, w.N) if nb > 1 else (w.M, w.N)
        dC = hC.cuda() if hC is not None else torch.empty(cshape, dtype=out_dt, device="cuda")
        bias = (torch.from_numpy(gi.draw("normal", 0xB1A5 + w.index, 3, (w.N,))).cuda()
                if v_bias else None)
        dev_ops.append((w, dA, dB, dC, bias))
        host_ops.append((w, hA.pin_memory(), hB.pin_memory(),
                         hC.pin_memory() if hC is not None else None, out_dt))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def flush_l2(write_only=False):
        flush.zero_()  # evicts every line of L2 (its own lines stay, dirty)
        if not write_only:
            flush_rd.sum()  # evicts those, writing them back; leaves clean lines

    def launch(w, dA, dB, dC, bias):
        if nb > 1:
            g.gemm_batched(dA, dB, dC, alpha=w.alpha, beta=w.beta, bias=bias, act=v_act)
        elif extended:
            g.gemm_ex(dA, dB, dC, alpha=w.alpha, beta=w.beta, bias=bias, act=v_act)
        elif w.dtype == "f32":
            g.sgemm(dA, dB, dC, alpha=w.alpha, beta=w.beta)
        else:
            g.gemm_bf16(dA, dB, dC, alpha=w.alpha, beta=w.beta)

    for _ in range(args.warmup):
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        flush_l2()
        for op in dev_ops:
            launch(*op)
    torch.cuda.synchronize()
    g.binding.check(g.binding.get_device_status(), "warm-up device status")

    nk = len(dev_ops)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
              for _ in range(args.steps)]
    clocks = ClockSampler(dist.local_rank)
    dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for s in range(args.steps):
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        flush_l2()
        ev = events[s]
        ev[0].record(stream)
        for i, op in enumerate(dev_ops):
            launch(*op)
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    wall = time.perf_counter() - t_wall0
    g.binding.check(g.binding.get_device_status(), "timed-region device status")

    # Context only, outside the timed region: each kernel again, back to back
    # without the flush, so operands that fit in L2 stay there between calls.
    warm_ms = []
    for op in dev_ops:
        wev = [torch.cuda.Event(enable_timing=True) for _ in range(WARM_REPS + 1)]
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        launch(*op)
        wev[0].record(stream)
        for r in range(WARM_REPS):
            launch(*op)
            wev[r + 1].record(stream)
        torch.cuda.synchronize()
        warm_ms.append([wev[r].elapsed_time(wev[r + 1]) for r in range(WARM_REPS)])
    g.binding.check(g.binding.get_device_status(), "warm-L2 pass device status")

    per_kernel_ms = [[ev[i].elapsed_time(ev[i + 1]) for ev in events] for i in range(nk)]
    step_ms = [sum(per_kernel_ms[i][s] for i in range(nk)) for s in range(args.steps)]
    total_s = dist.max(sum(step_ms) / 1e3)
    flops_step = sum(w.flops for w in workloads) * nb
    value = dist.sum(flops_step * args.steps) / total_s / 1e12
    gpu_launches = nk * args.steps

    sm_max = peaks.get("sm_max_mhz") or 2070.0
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12

    def roofline_of(w, ms, batch=1, traffic_ok=True):
        tflops = w.flops * batch / (ms / 1e3) / 1e12
        gbs = w.min_bytes() * batch / (ms / 1e3) / 1e9
        traffic = recorded_traffic(w) if traffic_ok else None
        if w.dtype == "f32":
            return {"bound": "alu", "achieved": tflops, "peak": fp32_peak, "unit": "TFLOP/s",
                    "frac": tflops / fp32_peak, "traffic": traffic,
                    "peak_source": f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 "
                                   f"x {sm_max:.0f} MHz (max SM clock)",
                    "kernel": kernel_name(w)}
        if w.M * w.N * w.K / (w.min_bytes() / 2) < 300:  # intensity below the ridge: HBM
            peak_bw = peaks["hbm_gbs"]
            return {"bound": "hbm", "achieved": gbs, "peak": peak_bw, "unit": "GB/s",
                    "frac": gbs / peak_bw, "traffic": traffic,
                    "peak_source": f"{peak_src} hbm_gbs (of measured copy bandwidth)"
                    if peak_src == "measured" else "fallback hbm_gbs",
                    "tensor_frac_of_bf16_peak": tflops / peaks["bf16_tflops"],
                    "kernel": kernel_name(w)}
        pk = peaks["bf16_tflops"]
        return {"bound": "tensor", "achieved": tflops, "peak": pk, "unit": "TFLOP/s",
                "frac": tflops / pk, "traffic": traffic,
                "peak_source": f"{peak_src} bf16_tflops (burst)",
                "frac_of_sustained": tflops / peaks.get("bf16_tflops_sustained", pk),
                "kernel": kernel_name(w)}

    kernels = {}
    rooflines = {}
    for i, w in enumerate(workloads):
        ms = statistics.mean(per_kernel_ms[i])
        warm = statistics.median(warm_ms[i])
        kernels[w.name] = {
            "ms_mean": ms, "ms_median": statistics.median(per_kernel_ms[i]),
            "ms_min": min(per_kernel_ms[i]), "tflops": w.flops * nb / (ms / 1e3) / 1e12,
            "min_bytes": w.min_bytes() * nb,
            "achieved_gbs_min_bytes": w.min_bytes() * nb / (ms / 1e3) / 1e9,
            "calls": args.steps, "timed": "inside the headline timed region",
            "warm_l2": {"ms_median": warm, "tflops": w.flops * nb / (warm / 1e3) / 1e12,
                        "calls": WARM_REPS}}
        rooflines[w.name] = roofline_of(w, ms, nb, traffic_ok=not extended)

    # ---- the other workloads (256^3, MLP and decode shapes): after the
    # headline's timed region, each timed alone over a fixed number of
    # L2-flushed calls, each with its own roofline; their outputs feed the
    # parity check below.  Not part of `value`.
    from gemm_inputs.workloads import WORKLOADS

    run_extra = (args.workload == "step" and not extended and not args.shape
                 and not args.no_extra and dist.rank == 0 and args.gpus == 1)
    extra_outputs = {}
    if run_extra:
        for w in WORKLOADS.values():
            if w.name in STEP_WORKLOADS:
                continue
            A, B, C = w.operands()
            host_np[w.name] = (A, B, C)
            dA, dB, dC, dC0 = _device_operands(torch, w, A, B, C)
            op = (w, dA, dB, dC, None)
            restore = (lambda dC=dC, dC0=dC0: dC.copy_(dC0)) if dC0 is not None else None
            reps = EXTRA_REPS.get(w.name, 20)
            for _ in range(3):
                launch(*op)
            torch.cuda.synchronize()
            def timed_calls(write_only):
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(reps)]
                for e0, e1 in evs:
                    if restore:
                        restore()
                    torch.cuda._sleep(HOST_AHEAD_CYCLES)
                    flush_l2(write_only)
                    e0.record(stream)
                    launch(*op)
                    e1.record(stream)
                torch.cuda.synchronize()
                g.binding.check(g.binding.get_device_status(), f"{w.name} device status")
                return [e0.elapsed_time(e1) for e0, e1 in evs]

            times_wo = timed_calls(True)
            times = timed_calls(False)  # last: its final call's output is checked below
            ms = statistics.mean(times)
            ms_wo = statistics.mean(times_wo)
            kernels[w.name] = {
                "ms_mean": ms, "ms_median": statistics.median(times), "ms_min": min(times),
                "tflops": w.flops / (ms / 1e3) / 1e12, "min_bytes": w.min_bytes(),
                "achieved_gbs_min_bytes": w.min_bytes() / (ms / 1e3) / 1e9, "calls": reps,
                "timed": "after the headline timed region, alone, L2 flushed before each call",
                "write_only_flush": {
                    "ms_mean": ms_wo, "ms_median": statistics.median(times_wo),
                    "tflops": w.flops / (ms_wo / 1e3) / 1e12,
                    "achieved_gbs_min_bytes": w.min_bytes() / (ms_wo / 1e3) / 1e9,
                    "note": "L2 flushed by the write alone, its dirty lines written back during "
                            "the call"}}
            rooflines[w.name] = roofline_of(w, ms)
            extra_outputs[w.name] = _host_output(torch, w, dC)  # C restored before the last call
            del dA, dB, dC, dC0
        torch.cuda.empty_cache()
    clock_info = clocks.stop()
    if clock_info is not None:
        clock_info["window"] = ("timed region, then the warm-L2 pass and the other workloads' "
                                "timed calls (GPU busy throughout)")

    dominant = max(range(nk), key=lambda i: statistics.mean(per_kernel_ms[i]))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(step_ms), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / PAGE_SGEMM_4096_TFLOPS
                        if [w.name for w in workloads] == ["sgemm_4096"] else None),
        "dtype": "+".join(sorted({w.dtype for w in workloads})),
        "data": "synthetic (seeded splitmix64 inputs; shapes and distributions of the workload)",
        "config": config_block(workloads, args),
        "roofline": rooflines[workloads[dominant].name],
        "rooflines": rooflines, "kernels": kernels,
        "gpu_launches": gpu_launches, "wall_s_timed_region": wall,
        "clocks": clock_info,
        "peaks": {"source": peak_src, "hbm_gbs": peaks["hbm_gbs"],
                  "bf16_tflops": peaks["bf16_tflops"], "fp32_tflops_derived": fp32_peak,
                  "sms": sms},
    }

    # ---- end to end through the public API with pinned host buffers
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 20))
        outs = [torch.empty((w.M, w.N), dtype=od, pin_memory=True)
                for (w, _a, _b, _c, od) in host_ops]

        # The host batch overlaps a product's copies with the compute of the
        # products before it, so the long FP32 product goes first.
        e2e_ops = sorted(zip(host_ops, outs), key=lambda t: t[0][0].dtype != "f32")

        def e2e_step():
            # One call for the step's products: the copies of each travel while
            # the one before it computes (gemm_host_batch).
            g.gemm_many([dict(A=hA, B=hB, C=hC, alpha=w.alpha, beta=w.beta, out_dtype=od,
                              out=out)
                         for (w, hA, hB, hC, od), out in e2e_ops])

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_s = dist.max(max(e0.elapsed_time(e1) / 1e3, time.perf_counter() - t0))
        h2d = sum((hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
                   + (hC.numel() * hC.element_size() if (hC is not None and w.beta != 0) else 0))
                  for (w, hA, hB, hC, od) in host_ops)
        d2h = sum(o.numel() * o.element_size() for o in outs)
        line["e2e"] = {"value": dist.sum(flops_step * e2e_steps) / e2e_s / 1e12,
                       "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                       "api": "dense_gemm_02_gb300.gemm_many(host pinned tensors) -> C ABI "
                              "gemm_host_batch (the step's products in one pipelined call)"}
    else:
        line["e2e"] = None

    # ---- outputs of the timed launches, for the parity check: with
    # beta == 0 every timed call wrote the same product; with beta != 0, C
    # is restored and the product computed once more, as timed.
    timed_outputs = {}
    if nb == 1 and not extended and not args.no_parity and dist.rank == 0:
        for (w, dA, dB, dC, bias), (_w, _hA, _hB, hC, _od) in zip(dev_ops, host_ops):
            if w.beta != 0:
                dC.copy_(hC.to(dC.device).view(dC.dtype))
                launch(w, dA, dB, dC, bias)
            timed_outputs[w.name] = _host_output(torch, w, dC)
        timed_outputs.update(extra_outputs)
        g.binding.check(g.binding.get_device_status(), "parity launch device status")

    # ---- integer-operand pass ({-2..2}): one launch per workload on the
    # same kernels, compared bit for bit below
    int_outputs, int_inputs = {}, {}
    if timed_outputs and not args.no_integer_pass:
        for name in timed_outputs:
            w = _workload_named(name, workloads)
            A, B, C = w.operands(integer=True)
            dA, dB, dC, _dC0 = _device_operands(torch, w, A, B, C)
            launch(w, dA, dB, dC, None)
            int_outputs[name] = _host_output(torch, w, dC)
            int_inputs[name] = (A, B, C)
            del dA, dB, dC, _dC0
        g.binding.check(g.binding.get_device_status(), "integer pass device status")
        torch.cuda.empty_cache()

    # ---- CPU oracle (rank 0, N = 1 only): the baseline is the oracle timed
    # on the headline workloads' own inputs (all host threads), and its
    # products are the reference of the parity check.
    if dist.rank == 0 and args.gpus == 1 and not args.no_cpu_baseline:
        import oracle

        ops = {n: host_np[n] for n in host_np if n in [w.name for w in workloads]}
        flops, dt, rows, threads, refs = oracle_sample_time(
            workloads, args.cpu_seconds, operands=ops if nb == 1 else None, keep=True)
        per = {}
        line["cpu_baseline"] = {
            "value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": (f"leading {rows} of {min(w.M for w in workloads)} rows of each of "
                       f"{', '.join(w.name for w in workloads)} (full K and N; the timed "
                       f"run's own inputs), {dt:.1f} s on {threads} threads"),
            "per_workload": per}
        parity = {}
        if timed_outputs:
            for w in workloads:
                if w.name in timed_outputs:
                    parity[w.name] = {"random": parity_random(
                        w, timed_outputs[w.name][:rows], refs[w.name])}
            for name in extra_outputs:
                w = WORKLOADS[name]
                A, B, C = host_np[name]
                t0 = time.perf_counter()
                ref = oracle.gemm(A, B, C, alpha=w.alpha, beta=w.beta, threads=threads)
                per[name] = {"all_cores_s": time.perf_counter() - t0, "threads": threads,
                             "tflops": w.flops / (time.perf_counter() - t0) / 1e12}
                parity[name] = {"random": parity_random(w, extra_outputs[name], ref)}
                del ref
            for name, got in int_outputs.items():
                w = _workload_named(name, workloads)
                A, B, C = int_inputs[name]
                ref = oracle.gemm(A, B, C, alpha=w.alpha, beta=w.beta, threads=threads)
                parity.setdefault(name, {})["integer"] = parity_integer(w, got, ref)
                del ref
            ok = all(v["random"]["violations"] == 0 and
                     v.get("integer", {"mismatches": 0})["mismatches"] == 0
                     for v in parity.values() if "random" in v)
            line["parity"] = {"ok": ok, "oracle": "double-precision triple loop (oracle/)",
                              "workloads": parity}
        # the 256^3 case on one core and on all cores
        w1 = WORKLOADS["sgemm_256"]
        A, B, C = host_np.get(w1.name) or w1.operands()
        for label, nt in (("one_core_s", 1), ("all_cores_s", threads)):
            reps, t0 = 0, time.perf_counter()
            while reps < 3 or time.perf_counter() - t0 < 0.5:
                oracle.gemm(A, B, C, alpha=w1.alpha, beta=w1.beta, threads=nt)
                reps += 1
            per.setdefault(w1.name, {})[label] = (time.perf_counter() - t0) / reps
        per[w1.name]["threads"] = threads
    if "parity" not in line:
        line["parity"] = None
    if dist.rank == 0:
        print(json.dumps(line))
    return 0


def _workload_named(name, workloads):
    from gemm_inputs.workloads import WORKLOADS

    for w in workloads:
        if w.name == name:
            return w
    return WORKLOADS[name]


def _device_operands(torch, w, A, B, C):
    """Device copies of one product's host operands (row-major, contiguous):
    (A, B, C, pristine C or None).  C is NaN-filled when beta == 0, so an
    output the kernel never writes cannot pass the parity check."""
    out_dt = torch.float32 if w.out == "f32" else torch.bfloat16

    def dev(x, kind):
        if kind == "f32":
            return torch.from_numpy(x).cuda()
        return torch.from_numpy(x.view("int16")).cuda().view(torch.bfloat16)

    dA, dB = dev(A, w.dtype), dev(B, w.dtype)
    if C is not None:
        dC0 = dev(C, w.out)
        dC = dC0.clone()
    else:
        dC0 = None
        dC = torch.full((w.M, w.N), float("nan"), dtype=out_dt, device="cuda")
    return dA, dB, dC, dC0


def _host_output(torch, w, dC):
    """A device C as a host array: float32, or the uint16 bits of bf16."""
    torch.cuda.synchronize()
    if w.out == "f32":
        return dC.cpu().numpy()
    return dC.contiguous().view(torch.int16).cpu().numpy().view("uint16")


def main():
    args = parse_args()
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, dist)
        return run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
