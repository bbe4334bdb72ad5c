"""Benchmark: one batched owner-side Muon step per timed step, on synthetic
LLM-shaped matrix sets (default: the Llama-3.1-8B projection set, 224
matrices, bf16 weights and grads, fp32 momentum, ns_steps=5).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line. ``value`` is the algorithmic Newton-Schulz throughput
(TFLOP/s, symmetric products counted once) over the whole step time
(momentum pass + Newton-Schulz + update) for all ranks together; ``ms_per_step``
is the step time. With N > 1 (torchrun) each rank runs its own replica of the
matrix set (independent matrices, no collective on the data path): weak
scaling; the time is the max over ranks.

``--impl reference`` times the fp64 CPU oracle instead (on the host cores, a
bounded sample of the same workload per step).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon step ms & NS TFLOP/s (% of GB300 bf16 peak) per model matrix set, 1 GPU"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "gemm": ["tc_ns.cu", "tc_ns2.cu", "tc_epilogue.cuh", "ptx.cuh", "internal.h"],
    "gram": ["tc_ns.cu", "tc_ns2.cu", "tc_epilogue.cuh", "ptx.cuh", "internal.h"],
    "poly": ["tc_ns.cu", "tc_ns2.cu", "tc_epilogue.cuh", "ptx.cuh", "internal.h"],
    "momentum": ["momentum.cu", "stream_tile.cuh", "internal.h"],
    "norm": ["momentum.cu", "stream_tile.cuh", "internal.h"],
}


# --------------------------------------------------------------------------- helpers
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def replica_seed_offset(rank: int) -> int:
    """Each rank draws its own replica of the matrix set."""
    return 100_000 * rank


def aggregate(flops_per_step_per_rank: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s: all ranks' work divided by the slowest rank's time."""
    return flops_per_step_per_rank * steps * world / max_seconds / 1e12


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def _code_only(src: str) -> str:
    """Source text without comments and blank space, so that the fingerprint
    changes with the code and not with its comments."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_sha(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kind, []):
        with open(os.path.join(ROOT, "matrix_optimizer_update_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_for(kind: str, workload: str):
    """DRAM bytes per launch of ``kind`` from the committed ncu summary, or None
    when there is none for this workload or the kernel source changed since."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(workload, {}).get(kind)
    if not e or e.get("source_sha") != kernel_source_sha(kind):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"dmuon_bench_clocks_{os.getpid()}_{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        note = None
        if not rows:
            # a timed region shorter than the sampling period: one reading right after it
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=30)
                parts = [p.strip() for p in out.stdout.strip().splitlines()[0].split(",")]
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                note = "timed region shorter than the 200 ms sampling period: one reading taken right after it"
            except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
                return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 300.0] or rows
        clk = {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
               "reasons": reasons, "samples": 0 if note else len(rows), "samples_under_load": 0 if note else len(loaded),
               "power_w_max": max(r[2] for r in rows)}
        if note:
            clk["note"] = note
        return clk


# --------------------------------------------------------------------------- host buffers
class HostBuffer:
    """Page-locked host memory for the end-to-end copies: torch's pinned
    allocation, or anonymous memory advised to use transparent huge pages and
    registered with the CUDA driver (use_thp). Which is faster differs from one
    machine to another: measured host-device rates ranged from 28 to 211 GB/s for either
    kind, depending on the machine and on what ran on it before."""

    def __init__(self, like, use_thp: bool):
        import mmap

        import torch

        self.registered = False
        self.mm = None
        nbytes = like.numel() * like.element_size()
        if use_thp:
            align = 2 << 20
            self.mm = mmap.mmap(-1, nbytes + align, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            self.mm.madvise(mmap.MADV_HUGEPAGE)
            raw = torch.frombuffer(self.mm, dtype=torch.uint8)
            off = (-raw.data_ptr()) % align
            t = raw[off:off + nbytes].view(like.dtype)
            t.zero_()  # touch every page before registration
            rc = torch.cuda.cudart().cudaHostRegister(t.data_ptr(), nbytes, 0)
            if int(rc) != 0:
                raise OSError(f"cudaHostRegister failed ({rc})")
            self.registered = True
            self.tensor = t
            self.kind = "transparent huge pages + cudaHostRegister"
        else:
            self.tensor = torch.empty(like.shape, dtype=like.dtype, device="cpu", pin_memory=True)
            self.kind = "torch pin_memory"

    def release(self):
        import torch

        if self.registered:
            torch.cuda.cudart().cudaHostUnregister(self.tensor.data_ptr())
            self.registered = False
        self.tensor = None
        self.mm = None


def fastest_host_buffer(dev, to_device: bool):
    """The faster of the two kinds of host buffer for copies to (or from) the
    device tensor `dev`, timed on one full copy each (outside any timed region)."""
    import torch

    best, best_s = None, None
    for use_thp in (False, True):
        try:
            hb = HostBuffer(dev, use_thp)
        except (OSError, AttributeError, ValueError, RuntimeError):
            continue
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if to_device:
            dev.copy_(hb.tensor, non_blocking=True)
        else:
            hb.tensor.copy_(dev, non_blocking=True)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        if best is None or dt < best_s:
            if best is not None:
                best.release()
            best, best_s = hb, dt
        else:
            hb.release()
    best.rate_gbs = dev.numel() * dev.element_size() / best_s / 1e9
    return best


# --------------------------------------------------------------------------- CPU oracle timing
def oracle_sample(workload, budget_s: float, start_layer: int = 0, max_mats=None):
    """Time the fp64 oracle on whole matrices of the workload, in layer order,
    until ``budget_s`` is spent. Returns (seconds, algorithmic NS flops, names)."""
    import numpy as np

    from matrix_optimizer_update_gb300 import workloads as wl
    from oracle import muon_ref as ref

    rng = np.random.default_rng(12345)
    done_flops, names, spent = 0, [], 0.0
    for li, (layer, role, r, c, e) in enumerate(workload.matrices()):
        if layer < start_layer:
            continue
        G = rng.standard_normal((r, c)) * workload.grad_std
        W = rng.standard_normal((r, c)) * workload.weight_std
        M = np.zeros((r, c))
        t0 = time.perf_counter()
        ref.muon_step(W, G, M, lr=workload.lr, mu=workload.mu, nesterov=workload.nesterov,
                      ns_steps=workload.ns_steps, coeffs=workload.coeffs, eps=workload.eps)
        spent += time.perf_counter() - t0
        done_flops += wl.ns_flops(r, c, workload.ns_steps)
        names.append(f"L{layer}.{role}" + (f".e{e}" if e >= 0 else "") + f" {r}x{c}")
        if spent >= budget_s or (max_mats is not None and len(names) >= max_mats):
            break
    return spent, done_flops, names


def cpu_model() -> str:
    """The host CPU's model name (lscpu), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    return "unknown"


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from matrix_optimizer_update_gb300 import workloads as wl

    w = wl.get(args.workload)
    # per step: the first matrices of the set in layer order, bounded to ~4 s of CPU work
    per_step_budget = 4.0
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, max_mats=1)
    total_s, total_f, names = 0.0, 0, []
    for k in range(args.steps):
        s, f, nm = oracle_sample(w, per_step_budget)
        total_s += s
        total_f += f
        names = nm
    value = total_f / total_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "matrices": len(w.shapes), "sample_per_step": names},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"per step: {', '.join(names)} (fp64 numpy oracle, whole matrices)",
                         "cpu_model": cpu_model(),
                         "extrapolated_step_ms": wl.totals(w)["ns_flops"] / (value * 1e12) * 1e3},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm
NS_KINDS = ("gram", "poly", "gemm", "symm")


def alu_peak_tflops(peaks, local):
    """fp32 FFMA peak: SMs x 128 lanes x 2 flops x max SM clock."""
    import torch

    props = torch.cuda.get_device_properties(local)
    return props.multi_processor_count * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12


def timed_steps(plan, step, steps, stream, launches_per_step, local, world, barrier, sample_clocks=True):
    """Time ``steps`` calls of ``step`` with CUDA events on ``stream`` (after the caller's
    warm-up), recording an event pair around every launch. Returns the elapsed ms (max over
    ranks), the per-kind totals, the launches counted, the device status and the clocks."""
    import torch

    from matrix_optimizer_update_gb300 import dmuon as dm

    clocks = ClockSampler(local) if sample_clocks else None
    if clocks:
        clocks.start()
    plan.profile_begin(steps * launches_per_step)
    c0 = plan.launch_count()
    torch.cuda.synchronize()
    barrier()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = ev[0].elapsed_time(ev[-1])
    timed_steps.last_step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    launches = plan.launch_count() - c0
    prof = plan.profile_end(steps * launches_per_step)
    clk = clocks.stop() if clocks else None
    status = plan.read_device_status(stream.cuda_stream)
    # the first timed step, launch by launch: ms of each product per Newton-Schulz step
    by_step = {}
    for (kind, kms, _), L in zip(prof[:launches_per_step], plan.describe()["launches"]):
        if L["step"] >= 0:
            by_step.setdefault(dm.KIND_NAMES[kind], {}).setdefault(L["step"], 0.0)
            by_step[dm.KIND_NAMES[kind]][L["step"]] += kms
    timed_steps.last_by_step = {k: [round(v[t], 4) for t in sorted(v)] for k, v in by_step.items()}
    per_kind = {}
    for kind, kms, work in prof:
        d = per_kind.setdefault(dm.KIND_NAMES[kind], {"ms": 0.0, "work": 0.0, "launches": 0})
        d["ms"] += kms
        d["work"] += work
        d["launches"] += 1
    return max_over_ranks(elapsed_ms, world, f"cuda:{local}"), per_kind, launches, status, clk


def step_stats(ms_list):
    """Median, 90th percentile and range of per-step times (ms)."""
    xs = sorted(ms_list)
    if not xs:
        return None
    p90 = xs[min(len(xs) - 1, int(round(0.9 * (len(xs) - 1))))]
    return {"median": statistics.median(xs), "p90": p90, "min": xs[0], "max": xs[-1]}


def graph_replay(plan_step, stream, steps, warmup):
    """One step captured in a CUDA graph on ``stream`` and replayed: ``warmup`` untimed replays,
    then ``steps`` timed ones with an event between every two. Returns per-step ms. The caller
    has already run the step with the same pointers, so the capture records no host copies."""
    import torch

    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        plan_step()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(steps):
            g.replay()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    out = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    del g
    return out


def cta_tails(plan, step, stream):
    """One more step with per-CTA start/end records; per kind of tensor-core launch, the tail
    (last CTA's end minus the median CTA's end) as a fraction of the launch's span (first start to
    last end), worst and mean over the step's launches, and the fraction of CTA time left idle."""
    import statistics as st

    import torch

    from matrix_optimizer_update_gb300 import dmuon as dm

    plan.profile_cta_times(True)
    step()
    torch.cuda.synchronize()
    out = {}
    for li, L in enumerate(plan.describe()["launches"]):
        rec = plan.read_cta_times(li, stream.cuda_stream)
        if not rec:
            continue
        t0 = min(a for a, _ in rec)
        ends = sorted(b for _, b in rec)
        span = ends[-1] - t0
        if span <= 0:
            continue
        busy = sum(b - a for a, b in rec)
        d = out.setdefault(dm.KIND_NAMES[L["kind"]], {"tails": [], "idle": []})
        d["tails"].append((ends[-1] - st.median(ends)) / span)
        d["idle"].append(1.0 - busy / (len(rec) * span))
    plan.profile_cta_times(False)
    return {k: {"tail_frac_max": max(v["tails"]), "tail_frac_mean": st.fmean(v["tails"]),
                "idle_frac_mean": st.fmean(v["idle"]), "launches": len(v["tails"])} for k, v in out.items()}


def kernel_table(per_kind, steps, tensor_peak, hbm_peak, alu_peak, compute, workload_name):
    kernels = {}
    for k, v in per_kind.items():
        if k in NS_KINDS:
            a = v["work"] / (v["ms"] * 1e-3) / 1e12
            peak = alu_peak if compute == "f32" else tensor_peak
            kernels[k] = {"ms_per_step": v["ms"] / steps, "tflops": a,
                          ("frac_of_alu_peak" if compute == "f32" else "frac_of_tensor_peak"): a / peak}
        else:
            a = v["work"] / (v["ms"] * 1e-3) / 1e9
            kernels[k] = {"ms_per_step": v["ms"] / steps, "gbs": a, "frac_of_hbm_peak": a / hbm_peak,
                          "traffic": traffic_for(k, workload_name)}
    return kernels


def measure_workload(name, args, local, tensor_peak, hbm_peak, alu_peak):
    """Step time, Newton-Schulz throughput and per-kernel figures of one more matrix set (its own
    inputs, plan and workspace, freed afterwards): the per_workload block of the bench line."""
    import torch

    from matrix_optimizer_update_gb300 import dmuon as dm
    from matrix_optimizer_update_gb300 import workloads as wl
    from matrix_optimizer_update_gb300.inputs import make_matrix_set

    w = wl.get(name)
    tot = wl.totals(w)
    ms = make_matrix_set(w, f"cuda:{local}")
    stream = torch.cuda.Stream()
    muon = dm.Muon.create(w.shapes, ns_steps=w.ns_steps, coeffs=w.coeffs, eps=w.eps, param=w.param_dtype,
                          grad=w.grad_dtype, compute=w.compute, flags=plan_flags(args), device=f"cuda:{local}",
                          stream=stream)
    plan = muon.plan
    lps = len(plan.describe()["launches"])
    Wp, Gp, Mp = ms.ptrs(ms.W), ms.ptrs(ms.G), ms.ptrs(ms.M)

    def step():
        plan.step(Wp, Gp, Mp, w.lr, w.mu, w.nesterov, stream.cuda_stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    steps = args.per_workload_steps
    ms_tot, per_kind, launches, status, clk = timed_steps(plan, step, steps, stream, lps, local, 1, lambda: None)
    ns_ms = sum(per_kind.get(k, {}).get("ms", 0.0) for k in NS_KINDS) / steps
    ns_tflops = tot["ns_flops"] / (ns_ms * 1e-3) / 1e12 if ns_ms else None
    peak = alu_peak if w.compute == "f32" else tensor_peak
    out = {"matrices": tot["matrices"], "params": tot["params"], "ns_flops_per_step": tot["ns_flops"],
           "steps": steps, "warmup": args.warmup, "ms_per_step": ms_tot / steps,
           "value": aggregate(tot["ns_flops"], steps, 1, ms_tot * 1e-3),
           "matrices_per_s": tot["matrices"] * steps / (ms_tot * 1e-3),
           "ns_ms_per_step": ns_ms, "ns_tflops": ns_tflops,
           ("ns_frac_of_alu_peak" if w.compute == "f32" else "ns_frac_of_sustained_peak"):
               (ns_tflops / peak) if ns_tflops else None,
           "compute": w.compute, "kernels": kernel_table(per_kind, steps, tensor_peak, hbm_peak, alu_peak, w.compute,
                                                         w.name),
           "ms_by_ns_step": timed_steps.last_by_step, "step_ms": step_stats(timed_steps.last_step_ms),
           **({"tuned_buckets": tuned_buckets(plan)} if args.tune else {}),
           "gpu_launches": launches, "device_status": status, "clocks": clk,
           "cta_tails": cta_tails(plan, step, stream) if w.compute == "bf16" else None}
    del muon, plan, ms
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def tuned_buckets(plan):
    """A tuned plan's choice per bucket, with the measured cost (SM-ms per matrix) of each candidate:
    one-SM 128 wide, one-SM 256 wide, two-SM pairs (0 = not timed), and the gemm's part of it."""
    return [{k: b[k] for k in ("m", "n", "pair", "bn_sym", "bn_gemm", "tune_cost", "tune_cost_gemm")}
            for b in plan.describe()["buckets"]]


def tile_kinds(plan):
    """Matrices per tile kind of a plan: two-SM 256 x 256 pairs or one-SM 128-row tiles."""
    out = {}
    for b in plan.describe()["buckets"]:
        k = "two-SM 256x256" if b["pair"] else f"one-SM 128x{b['bn_sym']}/128x{b['bn_gemm']}"
        out[k] = out.get(k, 0) + b["count"]
    return out


def plan_flags(args):
    from matrix_optimizer_update_gb300 import dmuon as dm

    return ((dm.FLAG_ONE_SM_TILES if args.one_sm else 0) | (dm.FLAG_STATIC_TILES if args.static_tiles else 0)
            | (dm.FLAG_TUNE if args.tune else 0))


def run_ours(args):
    import torch

    from matrix_optimizer_update_gb300 import build as build_mod
    from matrix_optimizer_update_gb300 import dmuon as dm
    from matrix_optimizer_update_gb300 import workloads as wl
    from matrix_optimizer_update_gb300.inputs import make_matrix_set

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    build_mod.build()
    w = wl.get(args.workload)
    if args.layers or args.experts:
        import dataclasses

        if args.layers:
            w = dataclasses.replace(w, layers=args.layers, name=f"{w.name}[{args.layers} layers]")
        if args.experts and w.experts:
            w = dataclasses.replace(w, experts=args.experts, name=f"{w.name}[{args.experts} experts]")
    tot = wl.totals(w)
    ms = make_matrix_set(w, f"cuda:{local}", seed_offset=replica_seed_offset(rank))
    stream = torch.cuda.Stream()
    tile_flags = plan_flags(args)
    muon = dm.Muon.create(w.shapes, ns_steps=w.ns_steps, coeffs=w.coeffs, eps=w.eps, param=w.param_dtype,
                          grad=w.grad_dtype, compute=w.compute, flags=tile_flags, device=f"cuda:{local}",
                          stream=stream)
    plan = muon.plan
    desc = plan.describe()
    launches_per_step = len(desc["launches"])
    headline_buckets = tuned_buckets(plan) if args.tune else None
    tiles = tile_kinds(plan)
    Wp, Gp, Mp = ms.ptrs(ms.W), ms.ptrs(ms.G), ms.ptrs(ms.M)
    sh = stream.cuda_stream

    def step():
        plan.step(Wp, Gp, Mp, w.lr, w.mu, w.nesterov, sh)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    barrier()

    # ---- device-resident timed region
    max_ms, per_kind, launches, status, clk = timed_steps(plan, step, args.steps, stream, launches_per_step, local,
                                                          world, barrier)
    ms_by_ns_step = timed_steps.last_by_step

    # ---- per-kind accounting from the live events
    ns_ms = sum(per_kind.get(k, {}).get("ms", 0.0) for k in NS_KINDS) / args.steps
    peaks, peak_src = load_peaks()
    tensor_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    alu_peak = alu_peak_tflops(peaks, local)
    ns_kinds = {k: v for k, v in per_kind.items() if k in NS_KINDS}
    dom = max(ns_kinds, key=lambda k: ns_kinds[k]["ms"]) if ns_kinds else max(per_kind, key=lambda k: per_kind[k]["ms"])
    d = per_kind[dom]
    if dom in NS_KINDS and w.compute == "f32":
        achieved = d["work"] / (d["ms"] * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": achieved / alu_peak, "peak_source": "SMs x 128 FP32 lanes x 2 x max SM clock",
                "work_per_launch": d["work"] / d["launches"], "ms_per_launch": d["ms"] / d["launches"],
                "traffic": None}
    elif dom in NS_KINDS:
        achieved = d["work"] / (d["ms"] * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": achieved / tensor_peak, "peak_source": f"{peak_src} bf16_tflops_sustained",
                "work_per_launch": d["work"] / d["launches"], "ms_per_launch": d["ms"] / d["launches"],
                "traffic": traffic_for(dom, w.name)}
    else:
        achieved = d["work"] / (d["ms"] * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "peak_source": f"{peak_src} hbm_gbs",
                "work_per_launch": d["work"] / d["launches"], "ms_per_launch": d["ms"] / d["launches"],
                "traffic": traffic_for(dom, w.name)}
    kernels = kernel_table(per_kind, args.steps, tensor_peak, hbm_peak, alu_peak, w.compute, w.name)
    step_ms = step_stats(timed_steps.last_step_ms)
    tails = cta_tails(plan, step, stream) if w.compute == "bf16" else None

    # ---- the same step captured once in a CUDA graph and replayed (no host work per step)
    graph = None
    if not args.no_graph:
        try:
            g_ms = graph_replay(step, stream, args.steps, args.warmup)
            graph = {"ms_per_step": sum(g_ms) / len(g_ms), **step_stats(g_ms), "steps": len(g_ms),
                     "device_status": plan.read_device_status(sh)}
        except RuntimeError as e:  # the line keeps its other figures if capture is refused
            torch.cuda.synchronize()
            graph = {"error": str(e).splitlines()[0][:200]}

    # ---- the Gram-space form of the iteration on the same matrix set (reported beside the headline):
    # its speed-up over the standard form, and the throughput of the flops it actually executes
    gram = None
    if not args.no_gram and w.compute == "bf16":
        gm = dm.Muon.create(w.shapes, ns_steps=w.ns_steps, coeffs=w.coeffs, eps=w.eps, param=w.param_dtype,
                            grad=w.grad_dtype, compute=w.compute, flags=dm.FLAG_GRAM_NS | tile_flags,
                            device=f"cuda:{local}", stream=stream)
        gplan = gm.plan
        glps = len(gplan.describe()["launches"])

        def gstep():
            gplan.step(Wp, Gp, Mp, w.lr, w.mu, w.nesterov, sh)

        for _ in range(args.warmup):
            gstep()
        torch.cuda.synchronize()
        barrier()
        gms, gkind, _, gstatus, _ = timed_steps(gplan, gstep, args.steps, stream, glps, local, world, barrier,
                                                sample_clocks=False)
        g_ns_ms = sum(gkind.get(k, {}).get("ms", 0.0) for k in NS_KINDS) / args.steps
        g_ns_work = sum(gkind.get(k, {}).get("work", 0.0) for k in NS_KINDS) / args.steps
        executed = g_ns_work / (g_ns_ms * 1e-3) / 1e12
        gram = {"ms_per_step": gms / args.steps, "ns_ms_per_step": g_ns_ms,
                "speedup_vs_standard": (max_ms / args.steps) / (gms / args.steps),
                "ns_flops_executed_per_step": g_ns_work,
                "executed_tflops": executed, "executed_frac_of_sustained_peak": executed / tensor_peak,
                "launches_per_step": glps, "device_status": gstatus}
        del gm, gplan

    # ---- end to end through the public API. Every step copies that step's gradients in from
    # host memory, runs dmuon_step, and returns the step's results to the host: every updated
    # weight, and the device status word (which also synchronises the host). The upload of step
    # k+1's gradients (into a second device buffer, on a copy stream) overlaps step k; the copy of
    # step k's weights (on a third stream) overlaps step k+1's momentum pass and its Newton-Schulz
    # steps before the last: the library orders only its W-writing launches after that copy
    # (dmuon_set_weight_events).
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(2, args.steps)  # as many steps as the device-timed region
        g_copy = ms.G.clone()  # the timing copy overwrites ms.G
        hbG = fastest_host_buffer(ms.G, to_device=True)
        hG = hbG.tensor
        hG.copy_(g_copy)
        ms.G.copy_(g_copy)
        del g_copy
        hbW = fastest_host_buffer(ms.W, to_device=False)  # reads W, leaves it as it is
        hW = hbW.tensor
        gbuf = [ms.G, torch.empty_like(ms.G)]
        gptrs = [Gp, ms.ptrs(gbuf[1])]
        copy_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        used = [torch.cuda.Event(), torch.cuda.Event()]
        w_ready, w_copied = torch.cuda.Event(), torch.cuda.Event()
        w_ready.record(stream)  # creates both events (no work behind them yet)
        w_copied.record(d2h_stream)
        plan.set_weight_events(w_copied.cuda_event, w_ready.cuda_event)
        torch.cuda.synchronize()
        barrier()
        def ev_pairs():
            return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(e2e_steps)]

        step_ev, h2d_ev, d2h_ev = ev_pairs(), ev_pairs(), ev_pairs()
        t0 = time.perf_counter()
        bits = 0
        with torch.cuda.stream(copy_stream):
            h2d_ev[0][0].record(copy_stream)
            gbuf[0].copy_(hG, non_blocking=True)
            h2d_ev[0][1].record(copy_stream)
            copied[0].record(copy_stream)
        for k in range(e2e_steps):
            b = k & 1
            if k + 1 < e2e_steps:  # upload the next step's gradients while this step runs
                nb = (k + 1) & 1
                with torch.cuda.stream(copy_stream):
                    if k >= 1:
                        copy_stream.wait_event(used[nb])
                    h2d_ev[k + 1][0].record(copy_stream)
                    gbuf[nb].copy_(hG, non_blocking=True)
                    h2d_ev[k + 1][1].record(copy_stream)
                    copied[nb].record(copy_stream)
            stream.wait_event(copied[b])
            step_ev[k][0].record(stream)
            plan.step(Wp, gptrs[b], Mp, w.lr, w.mu, w.nesterov, sh)  # W writes wait for w_copied
            step_ev[k][1].record(stream)
            used[b].record(stream)
            with torch.cuda.stream(d2h_stream):  # this step's weights back to the host
                d2h_stream.wait_event(w_ready)
                d2h_ev[k][0].record(d2h_stream)
                hW.copy_(ms.W, non_blocking=True)
                d2h_ev[k][1].record(d2h_stream)
                w_copied.record(d2h_stream)
            bits |= plan.read_device_status(sh)
        torch.cuda.synchronize()
        wall_ms = (time.perf_counter() - t0) * 1e3
        plan.set_weight_events(0, 0)
        dev_ms = sum(a.elapsed_time(b) for a, b in step_ev) / e2e_steps
        h2d_gbs = hG.numel() * hG.element_size() * e2e_steps / (sum(a.elapsed_time(b) for a, b in h2d_ev) * 1e-3) / 1e9
        d2h_gbs = hW.numel() * hW.element_size() * e2e_steps / (sum(a.elapsed_time(b) for a, b in d2h_ev) * 1e-3) / 1e9
        returned_ok = bool(torch.equal(hW.to(ms.W.device), ms.W))
        barrier()
        e2e_ms = max_over_ranks(wall_ms, world, f"cuda:{local}")
        e2e = {"value": aggregate(tot["ns_flops"], e2e_steps, world, e2e_ms * 1e-3), "unit": UNIT,
               "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
               "device_ms_per_step": dev_ms,
               "copy_gbs_in_loop": {"h2d": h2d_gbs, "d2h": d2h_gbs},
               "h2d_bytes_per_step": hG.numel() * hG.element_size(),
               "d2h_bytes_per_step": hW.numel() * hW.element_size() + 4,
               "result_read": "every updated weight (to host memory) and the device status word, every step",
               "returned_weights_match_device": returned_ok,
               "timing": "host wall clock from the first upload to the end of the last weight copy",
               "overlap": "next step's gradient upload overlaps the current step (two device buffers); each step's "
                          "weight copy overlaps the next step up to its last Newton-Schulz product",
               "host_memory": f"grads: {hbG.kind} ({hbG.rate_gbs:.0f} GB/s to the device); weights: {hbW.kind} "
                              f"({hbW.rate_gbs:.0f} GB/s from the device); the faster of two kinds each",
               "device_status": bits}
        del gbuf[1]
        del hG, hW
        torch.cuda.synchronize()
        hbG.release()
        hbW.release()

    # ---- optional: the AdamW kernel over the parameters Muon does not own (embedding, LM head and
    # norms of Llama-3.1-8B: 2 x 128256 x 4096 + 65 x 4096 elements), bf16 params and grads, fp32 moments
    adamw = None
    if args.adamw:
        n_aw = 2 * 128256 * 4096 + 65 * 4096
        ap = torch.randn(n_aw, dtype=torch.bfloat16, device=f"cuda:{local}") * 0.02
        ag = torch.randn(n_aw, dtype=torch.bfloat16, device=f"cuda:{local}") * 1e-3
        am = torch.zeros(n_aw, dtype=torch.float32, device=f"cuda:{local}")
        av = torch.zeros(n_aw, dtype=torch.float32, device=f"cuda:{local}")
        torch.cuda.synchronize()

        def aw_step(t):
            dm.dmuon_adamw_flat(ap.data_ptr(), ag.data_ptr(), am.data_ptr(), av.data_ptr(), n_aw, "bf16", "bf16",
                                lr=1e-3, step=t, stream=sh)

        for t in range(1, args.warmup + 1):
            aw_step(t)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for t in range(args.steps):
            aw_step(args.warmup + 1 + t)
        a1.record(stream)
        torch.cuda.synchronize()
        aw_ms = a0.elapsed_time(a1) / args.steps
        aw_bytes = n_aw * (2 + 2 + 2 + 8 + 8)  # p read + write, g read, m and v read + write
        adamw = {"elements": n_aw, "ms_per_step": aw_ms, "gbs": aw_bytes / (aw_ms * 1e-3) / 1e9,
                 "frac_of_hbm_peak": aw_bytes / (aw_ms * 1e-3) / 1e9 / hbm_peak,
                 "bytes_per_element": 22, "launches_per_step": 1}
        del ap, ag, am, av

    # ---- the other matrix sets, one at a time (one GPU only; each with its own inputs and plan)
    del muon, plan, ms
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    per_workload = None
    if world == 1 and not args.no_per_workload and not (args.layers or args.experts):
        per_workload = {}
        for name in wl.WORKLOADS:
            if name != w.name:
                per_workload[name] = measure_workload(name, args, local, tensor_peak, hbm_peak, alu_peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s, f, names = oracle_sample(w, args.cpu_budget)
        cpu = {"value": f / s / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{len(names)} whole matrices of layer 0 in order ({'; '.join(names)}), fp64 numpy, "
                         f"{s:.1f} s",
               "cpu_model": cpu_model(),
               "extrapolated_step_ms": tot["ns_flops"] / (f / s) * 1e3}

    value = aggregate(tot["ns_flops"], args.steps, world, max_ms * 1e-3)
    ns_tflops = tot["ns_flops"] / (ns_ms * 1e-3) / 1e12 if ns_ms else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": max_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.compute == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "matrices": tot["matrices"], "params": tot["params"],
                   "ns_steps": w.ns_steps, "ns_flops_per_step": tot["ns_flops"],
                   "storage": {"param": w.param_dtype, "grad": w.grad_dtype, "momentum": "f32"},
                   "parallelism": f"replicas{world}", "tiles": tiles,
                   "tile_schedule": "dealt round-robin" if args.static_tiles else "claimed from a counter",
                   "tuned": bool(args.tune),
                   **({"tuned_buckets": headline_buckets} if args.tune else {}),
                   "l2": "inputs larger than L2 (whole matrix set resident in HBM, no flush needed)"},
        "matrices_per_s": tot["matrices"] * world * args.steps / (max_ms * 1e-3),
        "ns_ms_per_step": ns_ms, "ns_tflops": ns_tflops,
        "ns_frac_of_sustained_peak": ns_tflops / tensor_peak if ns_tflops else None,
        "step_ms": step_ms, "graph_replay": graph,
        "kernels": kernels, "ms_by_ns_step": ms_by_ns_step, "cta_tails": tails, "roofline": roof, "gram_form": gram, "cpu_baseline": cpu, "e2e": e2e,
        "per_workload": per_workload,
        **({"adamw_other_params": adamw} if adamw is not None else {}),
        "gpu_launches": launches,
        "clocks": clk, "device_status": status,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama-3.1-8b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=0, help="truncate the workload to its first N layers (profiling)")
    ap.add_argument("--experts", type=int, default=0, help="truncate an MoE workload to N experts per layer (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gram", action="store_true", help="skip the Gram-space form measurement")
    ap.add_argument("--no-per-workload", action="store_true", help="skip the other matrix sets")
    ap.add_argument("--per-workload-steps", type=int, default=10, help="timed steps per other matrix set")
    ap.add_argument("--one-sm", action="store_true",
                    help="one-SM tiles everywhere instead of 256 x 256 tiles on CTA pairs where they fit")
    ap.add_argument("--static-tiles", action="store_true", help="deal tiles round-robin instead of claiming them")
    ap.add_argument("--no-graph", action="store_true", help="leave out the CUDA-graph replay timing")
    ap.add_argument("--tune", action="store_true", help="choose tile configurations by timing them at bind")
    ap.add_argument("--adamw", action="store_true",
                    help="also time the AdamW kernel over Llama-3.1-8B's non-matrix parameters")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps, always
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
