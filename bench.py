#!/usr/bin/env python3
"""Benchmark of the xSYMV hot path on GB300.

Workload: SSYMV, n = 32768, upper triangle stored, lda = n + 32, alpha = 1,
beta = 0 (the largest point of the single-precision size sweep n = 4096 ..
32768), synthetic U(-1, 1) data drawn on the device, NaN outside the stored
triangle.  One step = one call of the library's C ABI (main kernel + fixed-
order finaliser).  The stored triangle is 2.15 GB, far larger than the 129 MB
L2, so no flush is needed between steps.

Prints one JSON line: GFLOP/s (2 n^2 flops per call) over the timed steps,
the main kernel's achieved HBM bandwidth against the measured copy bandwidth
(roofline), the end-to-end rate through the host-buffer entry point with the
host<->device copies inside the timed region, SM clocks sampled during the
timed region (and, so that short runs get samples too, while the same steps
continue for at least a second after it), the number of kernels launched,
and the CPU oracle timed on a bounded sample of the same workload's data
(cpu_baseline).  Beside the headline: the size sweep (n = 4096 .. 32768),
small sizes (n = 512 .. 4096, the n = 1024 lower-triangle workload among
them), the other kinds, SYMV against GEMV, tickets against the workspace
reduction, and the block-column split run shard by shard on the one GPU.
``--impl reference`` times the CPU oracle alone on the same workload.

Multi-GPU (torchrun, one rank per GPU): the call is split by block columns
(each rank streams its panel of the stored triangle into a partial vector;
the partial vectors are all-gathered and added in rank order), a strong-
scaling workload: ``value`` is the one problem's flops per step over the
slowest rank's time.  ``--replicas`` runs one independent copy per rank
instead (weak scaling).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "xSYMV GFLOP/s & achieved HBM GB/s (% of GB300 peak) at n=8K–32K, 1 GPU"
UNIT = "GFLOP/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
L2_BYTES = 129e6
KERNEL = "symv_main"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--n", type=int, default=32768)
    ap.add_argument("--no-sweep", action="store_true", help="skip the n = 4096..32768 sweep")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kinds", action="store_true",
                    help="skip the one-shot measurements of DSYMV, CHEMV, ZHEMV, WSYMV")
    ap.add_argument("--no-gemv", action="store_true",
                    help="skip the SYMV-versus-GEMV comparison")
    ap.add_argument("--no-tickets", action="store_true",
                    help="skip the ordered-ticket versus workspace comparison")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--variant", default="",
                    help="time this compiled SSYMV variant (by name) instead of the tuned choice")
    ap.add_argument("--replicas", action="store_true",
                    help="with several ranks: independent replicas instead of the block-column split")
    ap.add_argument("--no-shards", action="store_true",
                    help="skip the block-column split run shard by shard on one GPU")
    ap.add_argument("--no-small", action="store_true", help="skip the small sizes n = 512 .. 4096")
    ap.add_argument("--gemv-n", type=int, default=0,
                    help="order of the SYMV-versus-GEMV comparison (default: 32768 for S, "
                         "24576 for D)")
    return ap.parse_args()


def flops(n: int) -> float:
    return 2.0 * n * n


def triangle_bytes(n: int, es: int = 4) -> float:
    return n * (n + 1) / 2.0 * es


def workload_config(n: int, world: int = 1, replicas: bool = False) -> dict:
    """The workload, the same in both arms (kernel variant and samples are
    reported beside it, not in it)."""
    cfg = {"workload": "ssymv n=%d uplo=U lda=n+32 alpha=1 beta=0 U(-1,1) seed=%d" % (n, n),
           "l2": "inputs larger than L2 (triangle %.2f GB vs 129 MB L2), "
           "no flush" % (triangle_bytes(n) / 1e9)}
    if world > 1:
        cfg["parallelism"] = ("replicas x%d" % world if replicas
                              else "block-column split x%d (rank-order reduction)" % world)
    return cfg


# ----------------------------------------------------------------- helpers --

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the files that define the main kernel's device code (the compiled variant
# is identified separately, by its name)
KERNEL_SOURCES = ("xsymv_kernels.cuh", "xsymv_plan.h", "xsymv_scalar.cuh")


def kernel_source_digest() -> str:
    """digest of the main kernel's code: its headers without // comments and
    blank lines, so that a comment edit does not void a traffic record"""
    csrc = os.path.join(ROOT, "symmetric_matrix_vector_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f)) as fh:
            code = [re.sub(r"//.*$", "", line).rstrip() for line in fh]
        h.update(f.encode())
        h.update("\n".join(line for line in code if line).encode())
    return h.hexdigest()[:16]


def recorded_traffic(n: int, variant: str):
    """DRAM bytes per launch of the main kernel from the committed ncu
    summary, scaled to n by stored elements; None when the kernel sources
    changed since the capture or no capture matches."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except Exception:
        return None
    # the partition's diagonal cost (_g<G>) does not change the compiled kernel
    same_kernel = re.sub(r"_g\d+", "", rec.get("variant", "")) == re.sub(r"_g\d+", "", variant)
    if rec.get("source_digest") != kernel_source_digest() or not same_kernel:
        return None
    n0 = rec["n"]
    per_elem = rec["dram_bytes_per_launch"] / (n0 * (n0 + 1) / 2.0)
    return per_elem * n * (n + 1) / 2.0


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line.strip()))

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_stop(self):
        self.t_stop = time.perf_counter()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        inside = [s for t, s in self.samples
                  if self.t_start is not None and self.t_start <= t <= (self.t_stop or t)]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons = [], None, set()
        for s in inside:
            parts = [p.strip() for p in s.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def host_link_gbs(torch, nbytes=1 << 30, reps=5):
    """Host-to-device bandwidth of this machine's CPU-GPU link: the best of a few
    copies of a pinned host buffer to the device (CUDA events)."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None or ms < best else best
    del h, d
    return nbytes / (best * 1e-3) / 1e9


def parse_cpulist(text: str):
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        else:
            cpus.add(int(part))
    return cpus


def gpu_host_placement(dev: int):
    """The GPU's PCI address, its NUMA node and the host CPUs local to it
    (from sysfs), and the CPUs this process may run on; None where unknown."""
    info = {"gpu_pci": None, "gpu_numa_node": None, "local_cpus": None,
            "process_cpus": len(os.sched_getaffinity(0))}
    try:
        bus = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                              "-i", str(dev)], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        dom, rest = bus.split(":", 1)
        path = "/sys/bus/pci/devices/%s:%s" % (dom[-4:].lower(), rest.lower())
        info["gpu_pci"] = bus
        with open(path + "/numa_node") as f:
            info["gpu_numa_node"] = int(f.read())
        with open(path + "/local_cpulist") as f:
            info["local_cpus"] = sorted(parse_cpulist(f.read()))
    except Exception:
        pass
    return info


def max_over_ranks(value: float, dist, device="cuda") -> float:
    """The largest value over all ranks (for times: the slowest rank)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist, device="cuda") -> float:
    """The sum of value over all ranks."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def replica_rate(world: int, flops_per_step: float, ms_per_step: float) -> float:
    """Whole-job GFLOP/s when each of `world` ranks runs its own replica and
    the slowest rank takes ms_per_step per step."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e9


# per kind: (workload name, flops per call / n^2, fp64 instructions per stored
# element: D 2 DFMA; Z 8 DFMA; W 2 double-double multiply-adds of 24 (a
# 4-operation exact product, the 20-operation accurate addition) + 3 to
# renormalise the element as it is read)
KIND_WORKLOADS = {
    "d": ("dsymv", 2, 2), "c": ("chemv", 8, 0), "z": ("zhemv", 8, 8), "w": ("wsymv", 2, 51),
}


# FP64 issue rate of GB300: the nominal 1.25 TFLOP/s over 152 SMs x 2 flops x
# 2.07 GHz is 1.99, i.e. 2 FP64 FMAs per clock per SM.  A loop of FMAs with
# register operands reaches it (the same-run probe); DADD, DMUL and FMAs with
# an immediate operand issue at about 1.68 per clock.
FP64_PER_CLK_PER_SM = 2
NOMINAL_SM_MHZ = 2070.0


def fp64_issue_peak(torch, sm_max_mhz=None):
    """FP64 instructions per second at the maximum SM clock"""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return FP64_PER_CLK_PER_SM * sms * (sm_max_mhz or NOMINAL_SM_MHZ) * 1e6


def measure_kinds(xs, inputs, torch, peaks, reps=10):
    """One timed measurement per other kind at its workload size (whole
    calls, CUDA events); HBM roofline for c, FP64 ALU roofline for d, z, w."""
    out = []
    for kind, (name, fl, f64) in KIND_WORKLOADS.items():
        spec = {"dsymv": ("L", 24576, dict(dist="normal", diag_shift=4.0), -0.75, 2.0, 7),
                "chemv": ("U", 16384, {}, complex(1, 0.5), complex(0.5, -0.25), 11),
                "zhemv": ("U", 16384, {}, complex(1, 0.5), complex(0.5, -0.25), 11),
                "wsymv": ("L", 8192, {}, (1.0, 0.0), (1.0, 0.0), 13)}[name]
        uplo, n, kw, al, be, seed = spec
        pr = inputs.device_problem(kind, uplo, n, lda=n, alpha=al, beta=be, seed=seed, **kw)
        A, x, y = pr["A"], pr["x"], pr["y"]
        for _ in range(3):
            xs.check(xs.symv(kind, uplo, n, al, A, n, x, 1, be, y, 1))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            xs.check(xs.symv(kind, uplo, n, al, A, n, x, 1, be, y, 1))
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        elems = n * (n + 1) / 2
        gbs = elems * inputs.ELEM_BYTES[kind] / (ms * 1e-3) / 1e9
        rec = {"kind": kind, "workload": "%s n=%d uplo=%s lda=n" % (name, n, uplo), "ms": ms,
               "gflops": fl * n * n / (ms * 1e-3) / 1e9, "gbs": gbs,
               "variant": xs.xsymv_variant_name(kind, xs.xsymv_selected_variant(kind, uplo, n))}
        if f64:
            issue = fp64_issue_peak(torch, peaks.get("sm_max_mhz"))
            probe = peaks["fp64_tflops"] * 1e12 / 2          # register-operand FMA loop, same run
            ach = elems * f64 / (ms * 1e-3)
            rec["roofline"] = {"bound": "alu", "unit": "FP64 inst/s", "achieved": ach,
                               "peak": issue, "frac": ach / issue, "per_element": f64,
                               "peak_source": "%d FP64 FMA/clock/SM x SMs x max SM clock"
                                              % FP64_PER_CLK_PER_SM,
                               "probe_fma": probe, "frac_of_probe": ach / probe}
        else:
            rec["roofline"] = {"bound": "hbm", "unit": "GB/s", "achieved": gbs,
                               "peak": peaks["hbm"], "frac": gbs / peaks["hbm"]}
        out.append(rec)
        del pr, A, x, y
        torch.cuda.empty_cache()
    return out


def _time_calls(torch, fn, reps):
    """average ms of `reps` back-to-back calls (inputs larger than L2)"""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def ticket_variants(xs, kind):
    return [i for i in range(xs.xsymv_variant_count(kind))
            if xs.xsymv_variant_name(kind, i).endswith("_tk")]


def time_variant(xs, torch, kind, variant, fn, reps):
    """average ms of one call with `variant` forced for `kind`"""
    assert xs.xsymv_set_variant(kind, variant) == 0
    try:
        return _time_calls(torch, fn, reps)
    finally:
        xs.xsymv_set_variant(kind, -1)


def measure_tickets(xs, inputs, torch, reps=10):
    """The report's ordered tickets (one launch; dynamic block IDs, per-chunk
    tickets passed in block order) against the workspace reduction (main
    kernel + fixed-order finaliser), both bit-identical run to run: whole
    calls at each kind's workload, the tuned workspace variant against the
    fastest ticket variant."""
    cases = [("s", "U", 32768, 32, 1.0, 0.0, {}), ("s", "U", 8192, 32, 1.0, 0.0, {}),
             ("d", "L", 24576, 0, -0.75, 2.0, dict(dist="normal", diag_shift=4.0)),
             ("c", "U", 16384, 0, complex(1, 0.5), complex(0.5, -0.25), {}),
             ("z", "U", 16384, 0, complex(1, 0.5), complex(0.5, -0.25), {}),
             ("w", "L", 8192, 0, (1.0, 0.0), (1.0, 0.0), {})]
    out = []
    for kind, uplo, n, pad, al, be, kw in cases:
        lda = n + pad
        pr = inputs.device_problem(kind, uplo, n, lda=lda, alpha=al, beta=be, seed=n, **kw)

        def call():
            xs.check(xs.symv(kind, uplo, n, al, pr["A"], lda, pr["x"], 1, be, pr["y"], 1))

        ws_v = xs.xsymv_selected_variant(kind, uplo, n)
        ws = time_variant(xs, torch, kind, ws_v, call, reps)
        tk = sorted((time_variant(xs, torch, kind, v, call, reps), v)
                    for v in ticket_variants(xs, kind))
        out.append({"kind": kind, "workload": "%s n=%d uplo=%s lda=%d" % (kind, n, uplo, lda),
                    "workspace_ms": ws, "workspace_variant": xs.xsymv_variant_name(kind, ws_v),
                    "tickets_ms": tk[0][0], "tickets_variant": xs.xsymv_variant_name(kind, tk[0][1]),
                    "tickets_over_workspace": tk[0][0] / ws,
                    "all_ticket_variants_ms": {xs.xsymv_variant_name(kind, v): t for t, v in tk}})
        del pr
        torch.cuda.empty_cache()
    return out


def measure_gemv(xs, inputs, torch, reps=20, n_over=0):
    """SYMV against the general product GEMV on the same loader (the
    report's §1 expects SYMV at about twice GEMV's speed when memory-bound),
    with cuBLAS's GEMV (torch.mv) beside it as an outside reference."""
    out = []
    for kind, n, uplo, lda_pad in (("s", 32768, "U", 32), ("d", 24576, "L", 0)):
        n = n_over or n
        lda = n + lda_pad
        es = 4 if kind == "s" else 8
        g = inputs.device_general(kind, n, lda=lda, alpha=1.0, beta=0.0, seed=n)
        A, x, y = g["A"], g["x"], g["y"]
        best = None
        for v in range(xs.xgemv_variant_count(kind)):
            xs.xgemv_set_variant(kind, v)
            ms = _time_calls(torch, lambda: xs.check(xs.gemv(kind, n, 1.0, A, lda, x, 1, 0.0, y, 1)),
                             reps)
            if best is None or ms < best[0]:
                best = (ms, xs.xgemv_variant_name(kind, v))
        xs.xgemv_set_variant(kind, -1)
        M = A[:, :n].t()                      # M[i, j] = A(i, j), strided view (no copy)
        cub = _time_calls(torch, lambda: torch.mv(M, x, out=y), reps)
        del g, A, x, y, M
        torch.cuda.empty_cache()
        s = inputs.device_problem(kind, uplo, n, lda=lda, alpha=1.0, beta=0.0, seed=n)
        sy = _time_calls(torch, lambda: xs.check(xs.symv(kind, uplo, n, 1.0, s["A"], lda, s["x"],
                                                         1, 0.0, s["y"], 1)), reps)
        svar = xs.xsymv_variant_name(kind, xs.xsymv_selected_variant(kind, uplo, n))
        del s
        torch.cuda.empty_cache()
        out.append({
            "kind": kind, "n": n, "lda": lda, "symv_uplo": uplo,
            "symv_ms": sy, "symv_variant": svar,
            "gemv_ms": best[0], "gemv_variant": best[1],
            "gemv_over_symv": best[0] / sy,
            "symv_gflops": 2.0 * n * n / (sy * 1e-3) / 1e9,
            "gemv_gflops": 2.0 * n * n / (best[0] * 1e-3) / 1e9,
            "symv_gbs": n * (n + 1) / 2 * es / (sy * 1e-3) / 1e9,
            "gemv_gbs": float(n) * n * es / (best[0] * 1e-3) / 1e9,
            "cublas_gemv_ms": cub, "cublas_gemv_over_symv": cub / sy,
            "note": "gemv_over_symv ~ 2 when both are memory-bound (half the bytes); ~ 1 when "
                    "both are FP64-bound (the same n*n multiply-adds)",
        })
    return out


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ CPU oracle ---

def oracle_block_call(o, A, lda, x, y, ns):
    """One oracle SSYMV (the report's three-part algorithm, binary64
    accumulator) on the leading ns-by-ns principal block of the workload's
    matrix: the same array, lda and vectors (a principal block of a
    symmetric matrix is itself the stored triangle of one)."""
    info, _, _, _ = o.symv("s", "U", ns, 1.0, A[:ns], lda, x, 1, 0.0, y, 1)
    assert info == 0


def oracle_block_size(o, A, lda, x, y, n, seconds_per_call):
    """the largest leading block (a multiple of 256, at most n) one oracle
    call finishes in about seconds_per_call, from a timed call on n=1024"""
    m = min(n, 1024)
    t0 = time.perf_counter()
    oracle_block_call(o, A, lda, x, y, m)
    rate = flops(m) / max(time.perf_counter() - t0, 1e-6)
    ns = int((seconds_per_call * rate / 2.0) ** 0.5)
    return n if ns >= n else max(256, ns // 256 * 256)


def cpu_oracle_rate(A, lda, x, y, n, seconds):
    """The CPU oracle on the workload's own data (host arrays), single-
    threaded, repeated until ``seconds`` have passed: each call on the whole
    matrix, or on its leading principal block if one call would take more
    than a third of the time.  Returns (GFLOP/s, calls, seconds, block)."""
    import oracle

    o = oracle.get()
    ns = oracle_block_size(o, A, lda, x, y, n, seconds / 3.0)
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle_block_call(o, A, lda, x, y, ns)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return flops(ns) * calls / el / 1e9, calls, el, ns


def run_reference(args):
    """The CPU oracle, timed step by step on the benchmark's workload: one
    step = one oracle call on the whole n=32768 matrix (host recipe of the
    same workload), or on its leading principal block when K + W whole calls
    would not end within about 90 s."""
    world, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from symmetric_matrix_vector_gb300 import inputs

    o = oracle.get()
    n = args.n
    t_gen = time.perf_counter()
    p = inputs.workload("ssymv_sweep", n=n)
    t_gen = time.perf_counter() - t_gen
    ns = oracle_block_size(o, p.A, p.lda, p.x, p.y, n, 90.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_block_call(o, p.A, p.lda, p.x, p.y, ns)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_block_call(o, p.A, p.lda, p.x, p.y, ns)
    el = time.perf_counter() - t0
    value = flops(ns) * args.steps / el / 1e9
    what = ("the workload's whole matrix" if ns == n else
            "the leading %d-by-%d principal block of the workload's matrix (a bounded sample)"
            % (ns, ns))
    sample = ("each step: the oracle's three-part SSYMV (binary64 accumulator), single-threaded, "
              "on %s (host recipe: numpy PCG64, seed n; generated in %.1f s before the timed "
              "steps)" % (what, t_gen))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "strong" if (world > 1 and not args.replicas) else "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(n, world, args.replicas),
        "sample_n": ns,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- our arm ----

def l2_flush_buffers(torch):
    """a 512 MB buffer to write and a 512 MB one to read: evicts the L2 and
    has the evicted dirty lines written back before the next timed call"""
    return (torch.empty(512 << 20, dtype=torch.uint8, device="cuda"),
            torch.zeros(64 << 20, dtype=torch.int64, device="cuda"))


def trimmed_mean(values, cut=0.1):
    """mean without the lowest and highest `cut` fraction: CUDA event times
    are quantised (on GB300 to about 2 us), and over many calls the quantum's
    phase varies, so a mean resolves what a median cannot"""
    v = sorted(values)
    k = int(len(v) * cut)
    v = v[k:len(v) - k] or v
    return sum(v) / len(v)


def time_flushed(torch, stream, fn, flush, reps=60):
    """ms of fn() with the L2 flushed before each call: the trimmed mean over
    `reps` calls (nothing synchronises inside the loop, so the events time the
    GPU work only)"""
    evs = []
    for _ in range(reps):
        flush[0].fill_(1)
        flush[1].sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return trimmed_mean([a.elapsed_time(b) for a, b in evs])


def host_us_per_call(torch, fn, calls=50):
    """the host's cost of issuing one call (Python binding, library, launch)"""
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(calls):
        fn()
    dt = (time.perf_counter() - t0) / calls
    torch.cuda.synchronize()
    return dt * 1e6


def time_back_to_back(torch, stream, fn, reps):
    """ms per call of `reps` calls enqueued back to back.  The GPU first
    spins for longer than the host needs to enqueue them all, so that the
    calls run back to back on the GPU and the events time the GPU's work,
    not the host's rate of issuing calls.  A few calls queued the same way
    beforehand leave the library in the state it keeps for back-to-back
    calls (it learns it from the calls it has run on the stream)."""
    per_call_s = host_us_per_call(torch, fn, 20) * 1e-6
    torch.cuda._sleep(int((1.5 * per_call_s * 10 + 2e-4) * NOMINAL_SM_MHZ * 1e6))
    for _ in range(10):
        fn()
    torch.cuda.synchronize()
    host_s = per_call_s * reps
    torch.cuda._sleep(int((1.5 * host_s + 2e-4) * NOMINAL_SM_MHZ * 1e6))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def measure_sweep(xs, inputs, torch, stream, peak, flush):
    """The workload's size sweep n = 4096 .. 32768 step 4096, each size
    timed with the L2 flushed and back to back."""
    sweep = []
    for m in range(4096, 32768 + 1, 4096):
        pm = inputs.device_problem("s", "U", m, lda=m + 32, alpha=1.0, beta=0.0, seed=m)

        def call():
            xs.check(xs.xsymv_s("U", m, 1.0, pm["A"], m + 32, pm["x"], 1, 0.0, pm["y"], 1))

        for _ in range(5):
            call()
        torch.cuda.synchronize()
        t_cold = time_flushed(torch, stream, call, flush)
        t_b2b = time_back_to_back(torch, stream, call, max(10, min(200, int(4e10 / triangle_bytes(m)))))
        # the headline figure of each size: flushed while the triangle
        # could partly stay in L2 (under 4x its 129 MB), else back to back
        cold = triangle_bytes(m) < 4 * L2_BYTES
        t = t_cold if cold else t_b2b
        sweep.append({"n": m, "gflops": flops(m) / (t * 1e-3) / 1e9,
                      "gbs": triangle_bytes(m) / (t * 1e-3) / 1e9,
                      "frac": triangle_bytes(m) / (t * 1e-3) / 1e9 / peak,
                      "l2": "flushed (write 512 MB, read 512 MB) before each call, trimmed mean "
                            "of 60"
                      if cold else "inputs larger than L2, back-to-back calls",
                      "gbs_l2_flushed": triangle_bytes(m) / (t_cold * 1e-3) / 1e9,
                      "gbs_back_to_back": triangle_bytes(m) / (t_b2b * 1e-3) / 1e9,
                      "variant": xs.xsymv_variant_name("s", xs.xsymv_selected_variant("s", "U", m))})
        del pm
    torch.cuda.empty_cache()
    return sweep


def measure_small(xs, inputs, torch, stream, peak, flush):
    """Small sizes, whose triangle fits the L2 (n <= 4096: at most 34 MB):
    the n = 1024 lower-triangle workload (lda = n, alpha = 1.25, beta = 0.5)
    and upper triangles n = 512 .. 4096 (lda = n + 32), each call's time
    with the L2 flushed before it (trimmed mean of 60) and back to back."""
    cases = [("ssymv n=1024 uplo=L lda=n alpha=1.25 beta=0.5 seed=0", "L", 1024, 1024, 1.25, 0.5, 0)]
    cases += [("ssymv n=%d uplo=U lda=n+32 alpha=1 beta=0 seed=%d" % (m, m), "U", m, m + 32, 1.0,
               0.0, m) for m in (512, 1024, 2048, 3072, 4096)]
    out = []
    for name, uplo, m, lda, al, be, seed in cases:
        pm = inputs.device_problem("s", uplo, m, lda=lda, alpha=al, beta=be, seed=seed)

        def call():
            xs.check(xs.xsymv_s(uplo, m, al, pm["A"], lda, pm["x"], 1, be, pm["y"], 1))

        for _ in range(5):
            call()
        torch.cuda.synchronize()
        t_cold = time_flushed(torch, stream, call, flush)
        t_b2b = time_back_to_back(torch, stream, call, 200)
        host = host_us_per_call(torch, call)
        out.append({"workload": name, "n": m, "uplo": uplo,
                    "us_l2_flushed": t_cold * 1e3, "us_back_to_back": t_b2b * 1e3,
                    "host_us_per_call": host,
                    "gflops_l2_flushed": flops(m) / (t_cold * 1e-3) / 1e9,
                    "gflops_back_to_back": flops(m) / (t_b2b * 1e-3) / 1e9,
                    "gbs_l2_flushed": triangle_bytes(m) / (t_cold * 1e-3) / 1e9,
                    "gbs_back_to_back": triangle_bytes(m) / (t_b2b * 1e-3) / 1e9,
                    "frac_l2_flushed": triangle_bytes(m) / (t_cold * 1e-3) / 1e9 / peak,
                    "variant": xs.xsymv_variant_name("s", xs.xsymv_selected_variant("s", uplo, m))})
        del pm
    torch.cuda.empty_cache()
    return out


def panel_elements(uplo, n, c0, c1):
    """stored elements of the columns c0 .. c1-1"""
    if uplo == "U":
        return (c1 * (c1 + 1) - c0 * (c0 + 1)) // 2
    return (c1 - c0) * n - (c1 * (c1 - 1) - c0 * (c0 - 1)) // 2


def measure_shards_one_gpu(xs, inputs, torch, stream, n, peak, flush):
    """The block-column split of the headline workload run on this one GPU,
    shard after shard (each panel in its own allocation, as on its own GPU):
    each shard call's time with the L2 flushed before it, and the rank-order
    reduction of the N partial vectors.  A rank's step would be its shard,
    an all-gather of N vectors of n elements, and the reduction; the slowest
    shard plus the reduction is that step without the all-gather."""
    from symmetric_matrix_vector_gb300 import sharded

    prob = inputs.device_problem("s", "U", n, lda=n + 32, alpha=1.0, beta=0.0, seed=n)
    A, x = prob["A"], prob["x"]
    y = torch.empty_like(prob["y"])
    out = []
    for N in (2, 4, 8):
        panels = sharded.split("U", n, N)
        parts = torch.empty((N, n), dtype=torch.float32, device="cuda")
        shards = []
        for r, (c0, c1) in enumerate(panels):
            panel, ldp = sharded.extract_panel(torch, A, "s", "U", n, n + 32, c0, c1)

            def call(panel=panel, ldp=ldp, c0=c0, c1=c1, r=r):
                xs.check(xs.xsymv_s_shard("U", n, c0, c1, panel, ldp, x, 1, parts[r]))

            for _ in range(3):
                call()
            ms = time_flushed(torch, stream, call, flush, reps=30)
            el = panel_elements("U", n, c0, c1)
            shards.append({"cols": [c0, c1], "ms": ms, "gbs": el * 4 / (ms * 1e-3) / 1e9,
                           "variant": xs.xsymv_variant_name(
                               "s", xs.xsymv_selected_variant("s", "U", int((2 * el) ** 0.5)))})
            del panel
        red = time_flushed(torch, stream,
                           lambda: xs.check(xs.xsymv_s_reduce(n, N, 1.0, parts, n, 0.0, y, 1)),
                           flush, reps=30)
        worst = max(sh["ms"] for sh in shards)
        out.append({"ranks": N, "shards": shards, "max_shard_ms": worst, "reduce_ms": red,
                    "step_ms_without_gather": worst + red,
                    "gflops_without_gather": flops(n) / ((worst + red) * 1e-3) / 1e9,
                    "slowest_shard_frac_of_hbm": max(sh["gbs"] for sh in shards if sh["ms"] == worst)
                    / peak})
        del parts
        torch.cuda.empty_cache()
    del prob, A, x, y
    torch.cuda.empty_cache()
    return out


def soak_for_clocks(torch, clocks, step, seconds=1.0):
    """keep running the same steps (untimed) until `seconds` have passed
    since the timed region began, so that the clock record has samples
    however short the timed region is"""
    while time.perf_counter() - clocks.t_start < seconds:
        for _ in range(20):
            step()
        torch.cuda.synchronize()
    clocks.mark_stop()


def clocks_summary(clocks, timed_s):
    c = clocks.summary()
    c["window"] = ("the timed region (%.4f s) and the same steps continued after it, %.2f s in "
                   "all" % (timed_s, (clocks.t_stop or 0) - (clocks.t_start or 0)))
    return c


def run_sharded(args, xs, inputs, torch, dist, world, rank, dev):
    """N ranks, one GPU each: the block-column split of the workload (strong
    scaling: the same one problem per step whatever N)."""
    from symmetric_matrix_vector_gb300 import sharded

    n = args.n
    lda = n + 32
    c0, c1 = sharded.split("U", n, world)[rank]
    prob = inputs.device_problem("s", "U", n, lda=lda, alpha=1.0, beta=0.0, seed=n)
    panel, ldp = sharded.extract_panel(torch, prob["A"], "s", "U", n, lda, c0, c1)
    x, y = prob["x"], prob["y"]
    del prob
    torch.cuda.empty_cache()
    job = sharded.ShardedSymv(torch, dist, "s", "U", n, c0, c1, panel, ldp, x, 1, world)
    stream = torch.cuda.current_stream()

    def step():
        job.step(1.0, 0.0, y, 1)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = xs.xsymv_launch_count()
    clocks.mark_start()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    timed_s = time.perf_counter() - clocks.t_start
    launches = xs.xsymv_launch_count() - l0
    soak_for_clocks(torch, clocks, step)
    dist.barrier()
    clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), dist)
    ms_per_step = ms / args.steps
    value = flops(n) / (ms_per_step * 1e-3) / 1e9
    launches_all = int(sum_over_ranks(float(launches), dist))

    # this rank's shard kernel (library events), the slowest rank's figure
    xs.xsymv_timing_enable(True)
    for _ in range(args.steps):
        xs.check(xs.xsymv_s_shard("U", n, c0, c1, panel, ldp, x, 1, job.partial))
    calls, main_ms, call_ms = xs.xsymv_timing_read()
    xs.xsymv_timing_enable(False)
    main_avg = main_ms / max(calls, 1)
    alg = panel_elements("U", n, c0, c1) * 4.0
    rate = alg / (main_avg * 1e-3) / 1e9
    slowest_main = max_over_ranks(main_avg, dist)
    peak, peak_src = measured_peak()
    rate_min = -max_over_ranks(-rate, dist)

    # end to end: this rank's panel and x from pinned host memory, y back
    hp = torch.empty(panel.shape, dtype=panel.dtype, pin_memory=True)
    hp.copy_(panel)
    hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    hx.copy_(x)
    hy = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)

    def estep():
        panel.copy_(hp, non_blocking=True)
        x.copy_(hx, non_blocking=True)
        step()
        hy.copy_(y, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        estep()
    esteps = max(3, min(args.steps, 50))
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(esteps):
        estep()
    e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    ems = max_over_ranks(e0.elapsed_time(e1) / esteps, dist)
    h2d = sum_over_ranks(float(hp.numel() * hp.element_size() + hx.numel() * 4), dist)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(n, world, False),
            "kernel_variant": xs.xsymv_variant_name(
                "s", xs.xsymv_selected_variant("s", "U", int((2 * alg / 4) ** 0.5))),
            "roofline": {"bound": "hbm", "achieved": rate_min, "peak": peak, "unit": "GB/s",
                         "frac": rate_min / peak, "traffic": None, "peak_source": peak_src,
                         "kernel": KERNEL, "main_kernel_ms_slowest_rank": slowest_main,
                         "note": "the slowest rank's shard kernel over its panel's stored bytes"},
            "e2e": {"value": flops(n) / (ems * 1e-3) / 1e9, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": n * 4 * world,
                    "ms_per_step": ems, "steps": esteps,
                    "api": "per rank: panel and x copied from pinned host memory, shard, "
                           "all-gather, reduce, y copied back"},
            "cpu_baseline": None, "clocks": clocks_summary(clocks, timed_s),
            "gpu_launches": launches_all,
        }
        print(json.dumps(line), flush=True)
    dist.destroy_process_group()


def run_ours(args):
    import torch

    import symmetric_matrix_vector_gb300 as xs
    from symmetric_matrix_vector_gb300 import _build, inputs

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    _build.build()
    xs.load()
    if world > 1 and not args.replicas:
        return run_sharded(args, xs, inputs, torch, dist, world, rank, dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    n = args.n
    if args.variant:
        names = [xs.xsymv_variant_name("s", i) for i in range(xs.xsymv_variant_count("s"))]
        if args.variant not in names:
            raise SystemExit("unknown SSYMV variant %r; compiled: %s" % (args.variant, names))
        xs.check(xs.xsymv_set_variant("s", names.index(args.variant)))
    prob = inputs.device_problem("s", "U", n, lda=n + 32, alpha=1.0, beta=0.0, seed=n)
    A, x, y = prob["A"], prob["x"], prob["y"]
    lda = prob["lda"]
    stream = torch.cuda.current_stream()
    variant = xs.xsymv_variant_name("s", xs.xsymv_selected_variant("s", "U", n))

    def step():
        xs.check(xs.xsymv_s("U", n, 1.0, A, lda, x, 1, 0.0, y, 1))

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # ---- timed region 1: the value (no hooks inside the library)
    clocks = ClockSampler(dev)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = xs.xsymv_launch_count()
    clocks.mark_start()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    timed_s = time.perf_counter() - clocks.t_start
    launches = xs.xsymv_launch_count() - l0
    soak_for_clocks(torch, clocks, step)
    barrier()
    clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), dist)
    ms_per_step = ms / args.steps
    value = replica_rate(world, flops(n), ms_per_step)

    # ---- timed region 2: per-kernel durations via the library's events
    xs.xsymv_timing_enable(True)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    calls, main_ms, call_ms = xs.xsymv_timing_read()
    xs.xsymv_timing_enable(False)
    main_avg = main_ms / max(calls, 1)
    peak, peak_src = measured_peak()
    alg = triangle_bytes(n)
    achieved = alg / (main_avg * 1e-3) / 1e9
    probes = xs.xsymv_probe_peaks() if rank == 0 else {}
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": recorded_traffic(n, variant),
                "peak_source": peak_src, "kernel": KERNEL, "main_kernel_ms": main_avg,
                "call_ms": call_ms / max(calls, 1), "algorithmic_bytes": alg,
                "nominal_gbs": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS}
    if probes:
        roofline["same_run"] = {k: round(v, 2) for k, v in probes.items()}
        roofline["frac_same_run_copy"] = achieved / probes["copy_gbs"]
        roofline["frac_same_run_read"] = achieved / probes["read_gbs"]

    # ---- beside the headline: sweep, small sizes, the split on one GPU
    sweep, small, shards = [], [], []
    if rank == 0 and not (args.no_sweep and args.no_small and (args.no_shards or world > 1)):
        del prob, A, x, y
        torch.cuda.empty_cache()
        flush = l2_flush_buffers(torch)
        if not args.no_sweep:
            sweep = measure_sweep(xs, inputs, torch, stream, peak, flush)
        if not args.no_small:
            small = measure_small(xs, inputs, torch, stream, peak, flush)
        if not args.no_shards and world == 1:
            shards = measure_shards_one_gpu(xs, inputs, torch, stream, n, peak, flush)
        del flush
        torch.cuda.empty_cache()
        prob = inputs.device_problem("s", "U", n, lda=n + 32, alpha=1.0, beta=0.0, seed=n)
        A, x, y = prob["A"], prob["x"], prob["y"]

    # ---- end to end through the host-buffer entry point
    e2e = None
    hA = hx = hy = None
    if not args.no_e2e:
        # the host link's rate as the process starts, then with the process
        # (and so its page-locked buffers, placed where they are first
        # touched) on the CPUs local to the GPU, when sysfs names a proper
        # subset of them
        placement = gpu_host_placement(dev)
        placement["link_gbs_default"] = host_link_gbs(torch)
        local = set(placement["local_cpus"] or [])
        allowed = os.sched_getaffinity(0)
        if local and (local & allowed) and (local & allowed) != allowed:
            os.sched_setaffinity(0, local & allowed)
            placement["bound_to_local_cpus"] = True
        else:
            placement["bound_to_local_cpus"] = False
        hA = torch.empty(A.shape, dtype=A.dtype, pin_memory=True)
        hA.copy_(A)
        hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        hx.copy_(x)
        hy = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        del prob, A, x, y
        torch.cuda.empty_cache()

        def hstep():
            xs.check(xs.xsymv_s_host("U", n, 1.0, hA, lda, hx, 1, 0.0, hy, 1))

        for _ in range(3):
            hstep()
        esteps = max(3, min(args.steps, 50))
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(esteps):
            hstep()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1) / esteps, dist)
        h2d, d2h = xs.xsymv_host_traffic()
        link = host_link_gbs(torch)
        moved = (h2d + d2h) / (ems * 1e-3) / 1e9
        e2e = {"value": replica_rate(world, flops(n), ems), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems,
               "steps": esteps,
               "api": "xsymv_s_host on pinned host buffers (read in place over the host link)",
               "host_placement": placement,
               "roofline": {"bound": "host link", "achieved": moved, "peak": link, "unit": "GB/s",
                            "frac": moved / link,
                            "peak_source": "pinned host -> device copy of 1 GiB, same run"}}

    kinds = []
    if rank == 0 and not args.no_kinds and probes:
        kinds = measure_kinds(xs, inputs, torch, {"hbm": peak, **probes,
                                                  "sm_max_mhz": clocks.summary().get("sm_max_mhz")})

    gemv_cmp = []
    if rank == 0 and not args.no_gemv:
        gemv_cmp = measure_gemv(xs, inputs, torch, n_over=args.gemv_n)

    tickets = []
    if rank == 0 and not args.no_tickets:
        tickets = measure_tickets(xs, inputs, torch)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if hA is None:           # the workload's data on the host
            hA, hx, hy = A.cpu(), x.cpu(), y.cpu()
        rate, calls_c, el, ns = cpu_oracle_rate(hA.numpy(), lda, hx.numpy(), hy.numpy(), n,
                                                args.cpu_seconds)
        what = ("the whole n=%d matrix" % n if ns == n else
                "the leading %d-by-%d principal block of the n=%d matrix" % (ns, ns, n))
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "the oracle's three-part SSYMV (binary64 accumulator), single-threaded, "
                         "on %s of this run's own data (copied from the GPU): %d calls in %.1f s"
                         % (what, calls_c, el)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(n, world, True),
            "kernel_variant": variant,
            "hbm_gbs": triangle_bytes(n) / (ms_per_step * 1e-3) / 1e9,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks_summary(clocks, timed_s), "gpu_launches": launches, "sweep": sweep,
            "small_n": small, "shards_one_gpu": shards,
            "kinds": kinds, "gemv_vs_symv": gemv_cmp, "tickets_vs_workspace": tickets,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
