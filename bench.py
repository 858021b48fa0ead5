#!/usr/bin/env python
"""Throughput of the Muon step over stacked parameter banks on GB300.

One step ("bank-step") = one muon_multi_step over every bank of the
GPT-2-small Muon parameter set: the attention bank (40, 768, 768), the MLP
bank (24, 3072, 768) with its dead slot, smear_gate (1, 12, 768) and
attn_gate (10, 6, 12): momentum, Frobenius normalisation, five quintic
Newton-Schulz iterations and the bf16 + mantissa update, all in this
repository's CUDA kernels.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--workload 4|5|6]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
of the workload (the step has no cross-GPU exchange on one node's banks);
the value is all ranks' steps divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Muon bank-steps/sec & NS TFLOP/s vs bf16 peak; update GB/s vs HBM peak"
UNIT = "bank-steps/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NS_GEMM_SOURCES = ["newton_schulz_stacked_gb300/csrc/mb_ns_kernel.cuh", "newton_schulz_stacked_gb300/csrc/mb_ns_gemm.cu",
                   "newton_schulz_stacked_gb300/csrc/mb_device.cuh",
                   "newton_schulz_stacked_gb300/csrc/mb_internal.h"]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", type=int, default=4, choices=[4, 5, 6])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true", help="skip the GPT-2-medium line added to workload 4's")
    p.add_argument("--step-flags", type=int, default=0,
                   help="MB_STEP_* options of the step (1: update in the last Newton-Schulz epilogue, "
                        "2: NorMuon row sums there); 0, the library's default path, is what is reported")
    return p.parse_args()


# ---------------------------------------------------------------- work counts

def shapes_of(wl):
    return [(b.batch, b.rows, b.cols) for b in wl.banks]


def ns_flops(shapes, ns_steps):
    """Algorithmic Newton-Schulz flops per step (3 m^2 n + m^3 per matrix and iteration: A and A^2
    counted once, symmetric) split by phase, and the dense-equivalent total (4 m^2 n + 2 m^3)."""
    gram = poly = apply_ = small = dense = 0.0
    for (B, R, C) in shapes:
        m, n = min(R, C), max(R, C)
        if m <= 64:
            small += B * ns_steps * (3.0 * m * m * n + m ** 3)
            continue
        gram += B * ns_steps * m * m * n
        poly += B * ns_steps * float(m) ** 3
        apply_ += B * ns_steps * 2.0 * m * m * n
        dense += B * ns_steps * (4.0 * m * m * n + 2.0 * m ** 3)
    return dict(gram=gram, poly=poly, apply=apply_, small=small, gemm=gram + poly + apply_, dense_gemm=dense)


def elems(shapes):
    return sum(B * R * C for (B, R, C) in shapes)


STEP_FUSE_UPDATE, STEP_FUSE_ROWSTATS = 1, 2     # the library's MB_STEP_* options


def last_epilogue_share(wl, flags):
    """Elements whose last Newton-Schulz epilogue also finishes the step, as the MB_STEP_* flags
    ask: without NorMuon it applies the update (tensor-core banks whose columns are a multiple of
    8, at least 3 steps); with NorMuon it sums v^2 per row, so the row statistics make no pass
    over v."""
    n = 0
    for b in wl.banks:
        if min(b.rows, b.cols) <= 64 or wl.ns_steps < 3:
            continue
        if (wl.normuon and flags & STEP_FUSE_ROWSTATS) or (
                not wl.normuon and flags & STEP_FUSE_UPDATE and b.cols % 8 == 0):
            n += b.batch * b.rows * b.cols
    return n


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_text(src: str) -> str:
    """C++ source without its comments and with runs of whitespace collapsed: what the compiler
    sees (these sources hold no comment markers inside string literals)."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_hash():
    """Hash of the NS kernel's code (comments and layout excluded), to match profiled counters."""
    h = hashlib.sha256()
    for rel in NS_GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per NS GEMM launch from the committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ns_gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_sha") != kernel_hash():
        return None
    return d.get("workloads", {}).get(str(workload), {}).get("bytes_per_launch")


# ---------------------------------------------------------------- ranks

def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (x itself outside torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = device if device is not None and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, steps: int, slowest_ms: float) -> float:
    """Whole-job rate: every rank runs `steps` steps; the job lasts as long as its slowest rank."""
    return world * steps / (slowest_ms / 1e3)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [ln.strip().split(", ") for ln in f if ln.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle baseline

def one_matrix_states(wl, seed):
    """One matrix's seeded state and gradient per bank (the oracle's cost depends on the shape only)."""
    import numpy as np
    import synth
    out = []
    for bi, spec in enumerate(wl.banks):
        rng = np.random.default_rng(seed * 100 + bi)
        one = synth.BankSpec(spec.name, 1, spec.rows, spec.cols, spec.grad_kind, spec.grad_std)
        w, mant, mom, row = synth.draw_state(rng, one)
        out.append((w, mant, mom, row, synth.draw_grad(rng, one)))
    return out


def oracle_matrix_step(wl, state):
    """The fp64 oracle's whole step (momentum, Newton-Schulz, NorMuon if on, update) on one matrix."""
    import oracle as O
    w, mant, mom, row, g = state
    O.bank_step(w, mant, mom, g, wl.lr, wl.wd, wl.mu, wl.ns_steps,
                normuon_beta2=wl.beta2 if wl.normuon else None, row_state=row)


def cpu_oracle_sample(wl, per_bank, seed_step=1):
    """Time the fp64 oracle on a bounded sample of the workload; extrapolate to one full step."""
    total_est, sampled, desc = 0.0, 0, []
    states = one_matrix_states(wl, seed_step)
    for bi, spec in enumerate(wl.banks):
        n = min(per_bank.get(spec.name, 1), spec.batch)
        t0 = time.perf_counter()
        for _ in range(n):
            oracle_matrix_step(wl, states[bi])
        dt = time.perf_counter() - t0
        total_est += dt / n * spec.batch
        sampled += n
        desc.append(f"{n}/{spec.batch} of {spec.name}")
    return total_est, sampled, ", ".join(desc)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cores():
    """The host threads the fp64 oracle can use: the affinity set, capped by a BLAS thread limit."""
    n = host_cores()
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            n = min(n, int(v))
    return n


# ---------------------------------------------------------------- reference arm

# Fraction of a bank-step that one reference step processes: the same share of every bank, so
# that the work done is that fraction of the whole step whatever each bank costs.
REF_FRACTION = {4: 1 / 8, 5: 1 / 48, 6: 1 / 8}


def ref_window(batch, f, k):
    """Slots of a bank that reference step k processes: a window of f * batch slots that moves on
    by that much every step (cumulative floors), so consecutive steps cover the bank in turn and
    any K steps process floor-differences summing to K * f * batch within one slot."""
    lo, hi = math.floor(k * batch * f), math.floor((k + 1) * batch * f)
    return [i % batch for i in range(lo, hi)]


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and os.environ.get("OMP_NUM_THREADS") == "1":
        # torchrun gives every rank one BLAS thread by default; rank 0 alone runs this arm, so it
        # takes the host's cores as a single-process run would (set before NumPy loads its BLAS)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = str(host_cores())
    import synth
    wl = synth.WORKLOADS[args.workload]
    f = REF_FRACTION[args.workload]
    states = one_matrix_states(wl, 1)

    def ref_step(k):
        done = {}
        for bi, spec in enumerate(wl.banks):
            slots = ref_window(spec.batch, f, k)
            for _ in slots:
                oracle_matrix_step(wl, states[bi])
            done[spec.name] = done.get(spec.name, 0) + len(slots)
        return done

    for k in range(args.warmup):
        ref_step(k)
    processed = {}
    t0 = time.perf_counter()
    for k in range(args.warmup, args.warmup + args.steps):
        for name, n in ref_step(k).items():
            processed[name] = processed.get(name, 0) + n
    wall = time.perf_counter() - t0
    # the banks of the window's width f * batch (an integer for the large banks) make exactly
    # steps * f bank-steps; the small gate banks rotate one matrix at a time within that share
    work = args.steps * f
    value = work / wall
    desc = ", ".join(f"{processed.get(b.name, 0)} of {b.name} (batch {b.batch})" for b in wl.banks)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded PCG64 banks)",
        "config": config_of(wl, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores(), "kind": "oracle",
                         "sample": f"each timed step runs the fp64 oracle's whole step on 1/{round(1 / f)} of "
                                   f"every bank (a window moving through the slots); {args.steps} steps "
                                   f"processed {desc} = {work:.3f} bank-steps in {wall:.2f} s"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl, args):
    return {
        "workload": f"{wl.name}: " + " + ".join(f"{b.name} {b.batch}x{b.rows}x{b.cols}" for b in wl.banks),
        "banks": [{"name": b.name, "shape": [b.batch, b.rows, b.cols], "grad": b.grad_kind,
                   "dead_slots": list(b.dead_slots)} for b in wl.banks],
        "ns_steps": wl.ns_steps, "lr": wl.lr, "wd": wl.wd, "mu": wl.mu, "normuon": wl.normuon,
        "l2": "no flush: inputs larger than L2 (%.2f GB of step state read and written per step)" % (
            elems(shapes_of(wl)) * (2 + 2 + 4 + 2) / 1e9),
        "parallelism": f"replicas x{args.gpus}",
        **({"step_flags": args.step_flags} if getattr(args, "step_flags", 0) else {}),
    }


# ---------------------------------------------------------------- native arm

class DeviceWorkload:
    """A workload's banks resident on one GPU (two alternating gradient draws), stepped through
    muon_multi_step, and the device-timed measurement of K steps."""

    def __init__(self, nss, wl, dev, flags=0):
        import numpy as np
        import torch
        import synth
        self.nss, self.wl, self.dev, self.flags = nss, wl, dev, flags
        self.shapes = shapes_of(wl)
        t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
        self.banks, self.grads, self.grads_host = [], [], []
        for bi, spec in enumerate(wl.banks):
            w, mant, mom, row = synth.init_state(wl.wid, bi)
            g_steps = [synth.grad(wl.wid, s, bi) for s in (1, 2)]
            self.grads.append([t16(g) for g in g_steps])
            self.grads_host.append([torch.from_numpy(g.view(np.int16)).pin_memory() for g in g_steps])
            self.banks.append(nss.BankState(t16(w), self.grads[-1][0], torch.from_numpy(mom).to(dev), t16(mant),
                                            torch.from_numpy(row).to(dev) if wl.normuon else None))
        self.ws = torch.empty(nss.mb_multi_workspace_bytes(self.banks, wl.normuon), dtype=torch.uint8, device=dev)

    def step(self, k):
        for b, g in zip(self.banks, self.grads):
            b.grad = g[k & 1]
        self.run_step()

    def run_step(self):
        wl = self.wl
        self.nss.muon_multi_step(self.banks, wl.lr, wl.wd, wl.mu, normuon=wl.normuon, beta2=wl.beta2,
                                 ns_steps=wl.ns_steps, workspace=self.ws, flags=self.flags)

    def timed(self, steps, warmup, world, gpu_index):
        """W warm-up steps, then K steps timed with CUDA events on the launching stream (barrier and
        synchronise on both sides, max over ranks), the library's stage events and launch counter over
        the same steps, and the SM clocks sampled meanwhile."""
        import torch
        import torch.distributed as dist
        nss = self.nss
        for k in range(max(warmup, 3)):
            self.step(k)
        torch.cuda.synchronize()
        if nss.mb_sync_status() != 0:
            raise RuntimeError("device-side status set during warm-up")
        stream = torch.cuda.current_stream()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = nss.mb_launch_count()
        with ClockSampler(gpu_index) as clocks:
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            with nss.StageTimer(max_marks=64 * steps + 64) as timer:
                ev0.record(stream)
                for k in range(steps):
                    self.step(k)
                ev1.record(stream)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
        launches = nss.mb_launch_count() - n0
        elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), self.dev)
        if nss.mb_sync_status() != 0:
            raise RuntimeError("device-side status set during the timed steps")
        return dict(elapsed_ms=elapsed_ms, stages=timer.totals(), launches=launches, clocks=clocks.summary(),
                    steps=steps)

    def rates(self, t):
        """Per-stage throughput from one timed() result: NS TFLOP/s (algorithmic flops of the fused
        launch over its stage time) and the element-wise stages' GB/s over their algorithmic bytes."""
        steps = t["steps"]
        per = {k: v[0] / steps for k, v in t["stages"].items()}
        gemm_ms = per.get("ns_gemm", 0.0)
        gemm_launches = t["stages"].get("ns_gemm", (0, 0))[1]
        fl = ns_flops(self.shapes, self.wl.ns_steps)
        E = elems(self.shapes)
        # elements the update kernel and the row-statistics pass still handle (the rest are done
        # in the last Newton-Schulz epilogue; their bytes are then part of the fused launch's time)
        fused = last_epilogue_share(self.wl, self.flags)
        E_upd = E - fused if not self.wl.normuon else E
        E_row = E - fused if self.wl.normuon else 0
        r = dict(per=per, flops=fl, gemm_ms=gemm_ms, gemm_launches=gemm_launches)
        r["ns_tflops"] = fl["gemm"] / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else None
        r["ns_tflops_dense_equiv"] = fl["dense_gemm"] / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else None
        r["momentum_gbs"] = 12.0 * E / (per["momentum"] * 1e-3) / 1e9 if per.get("momentum") else None
        # a GB/s figure only for a pass over most of the elements (not for a few gate matrices)
        r["update_gbs"] = (10.0 * E_upd / (per["update"] * 1e-3) / 1e9
                           if per.get("update") and E_upd >= 0.5 * E else None)
        # NorMuon row statistics: each element of v read once (2 B); the per-row state is negligible
        r["normuon_rowstats_gbs"] = (2.0 * E_row / (per["rowstats"] * 1e-3) / 1e9
                                     if per.get("rowstats") and E_row >= 0.5 * E else None)
        r["last_epilogue"] = (None if not fused else
                              ("row sums of v^2 for %d of %d elements" if self.wl.normuon else
                               "the update for %d of %d elements") % (fused, E))
        r["flops_per_launch"] = fl["gemm"] * steps / max(gemm_launches, 1)
        r["ms_per_launch"] = gemm_ms * steps / max(gemm_launches, 1)
        return r


def run_native(args):
    import torch
    import torch.distributed as dist

    import newton_schulz_stacked_gb300 as nss
    import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    nss.load_library()
    gpu_index = torch.cuda.current_device() if world == 1 else local

    wl = synth.WORKLOADS[args.workload]
    run = DeviceWorkload(nss, wl, dev, args.step_flags)
    banks, grads_host, ws = run.banks, run.grads_host, run.ws
    t = run.timed(args.steps, args.warmup, world, gpu_index)
    elapsed_ms, launches = t["elapsed_ms"], t["launches"]
    ms_per_step = elapsed_ms / args.steps
    value = job_rate(world, args.steps, elapsed_ms)
    r = run.rates(t)
    per, ns_tflops = r["per"], r["ns_tflops"]
    mom_gbs, upd_gbs, row_gbs = r["momentum_gbs"], r["update_gbs"], r["normuon_rowstats_gbs"]

    pk, pk_kind = peaks()
    # the timed region is tens to hundreds of milliseconds of steps: the burst peak applies; the
    # fraction of the sustained (power-capped, seconds-long) peak is reported beside it
    burst_peak = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained_peak = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    hbm_peak = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    roofline = {
        "bound": "tensor",
        "kernel": "ns_fused_kernel: all Newton-Schulz steps (A=XX^T, B'=aI+bA+cAA, X=B'X), %d launch(es) per step" % (
            r["gemm_launches"] // args.steps),
        "achieved": ns_tflops, "peak": burst_peak, "unit": "TFLOP/s",
        "frac": (ns_tflops / burst_peak) if ns_tflops else None,
        "peak_kind": f"{pk_kind} bf16 burst (the timed region lasts {elapsed_ms:.0f} ms)",
        "frac_of_sustained": (ns_tflops / sustained_peak) if ns_tflops else None,
        "flops_per_launch": r["flops_per_launch"], "ms_per_launch": r["ms_per_launch"],
        "traffic": profiled_traffic(args.workload),
    }

    extra = None
    if world == 1 and args.workload == 4 and not args.no_extra:
        # the largest configuration (GPT-2-medium banks with NorMuon), device-timed after the
        # headline; reported beside it, not in place of it
        wl5 = synth.WORKLOADS[5]
        run5 = DeviceWorkload(nss, wl5, dev, args.step_flags)
        k5 = max(3, min(args.steps, 20))
        t5 = run5.timed(k5, 3, world, gpu_index)
        r5 = run5.rates(t5)
        extra = {
            "workload": config_of(wl5, args)["workload"], "steps": k5, "warmup": 3,
            "value": job_rate(world, k5, t5["elapsed_ms"]), "unit": UNIT,
            "ms_per_step": t5["elapsed_ms"] / k5,
            "ns_tflops": r5["ns_tflops"],
            "ns_frac_of_burst": (r5["ns_tflops"] / burst_peak) if r5["ns_tflops"] else None,
            "ns_frac_of_sustained": (r5["ns_tflops"] / sustained_peak) if r5["ns_tflops"] else None,
            "momentum_gbs": r5["momentum_gbs"], "update_gbs": r5["update_gbs"],
            "normuon_rowstats_gbs": r5["normuon_rowstats_gbs"],
            "normuon_rowstats_of_hbm": (r5["normuon_rowstats_gbs"] / hbm_peak) if r5["normuon_rowstats_gbs"] else None,
            "last_newton_schulz_epilogue_also_does": r5["last_epilogue"],
            "stages_ms_per_step": r5["per"], "gpu_launches": t5["launches"], "clocks": t5["clocks"],
        }
        del run5
        torch.cuda.empty_cache()

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # two full steps of every bank (workload 4: ~11 s on 16 cores), or a slice of the larger ones
        sample = ({spec.name: spec.batch for spec in wl.banks} if args.workload == 4
                  else {"attn": 8, "mlp": 4, "qk": 16, "vo": 8})
        t0 = time.perf_counter()
        ests = [cpu_oracle_sample(wl, sample, seed_step=k + 1) for k in range(2)]
        est = statistics.mean(e[0] for e in ests)
        cpu_base = {"value": 1.0 / est, "unit": UNIT, "cores": cores(), "kind": "oracle",
                    "sample": f"fp64 oracle, 2 x ({ests[0][2]}) ({time.perf_counter() - t0:.1f} s), "
                              f"scaled to one full step"}

    e2e = None
    if not args.no_e2e:
        # End to end through the public call: every step uploads its gradients from pinned host
        # memory and brings the updated bf16 weights back to pinned host memory.  The copies run
        # on two copy streams beside the compute: step k+1's gradients upload while step k runs
        # (double-buffered device gradients), and step k's update also writes the new weights into
        # a second device buffer (the banks' bank_copy, double-buffered), downloaded while step
        # k+1 runs.
        main_s = torch.cuda.current_stream()
        h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        gdev = [[torch.empty_like(b.bank) for b in banks] for _ in range(2)]
        snap = [[torch.empty_like(b.bank) for b in banks] for _ in range(2)]
        host_out = [[torch.empty(b.bank.shape, dtype=torch.int16).pin_memory() for b in banks] for _ in range(2)]
        ev = lambda: torch.cuda.Event()
        ev_h2d, ev_gfree, ev_snap, ev_d2h = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]
        h2d = sum(g[0].numel() * 2 for g in grads_host)
        d2h = sum(b.numel() * 2 for b in host_out[0])

        def upload(k):
            b_ = k & 1
            with torch.cuda.stream(h2d_s):
                if k >= 2:
                    h2d_s.wait_event(ev_gfree[b_])
                for g, gh in zip(gdev[b_], grads_host):
                    g.copy_(gh[k & 1], non_blocking=True)
                ev_h2d[b_].record(h2d_s)

        def e2e_run(n):
            upload(0)
            for k in range(n):
                b_ = k & 1
                if k + 1 < n:
                    upload(k + 1)
                main_s.wait_event(ev_h2d[b_])
                if k >= 2:
                    main_s.wait_event(ev_d2h[b_])   # step k-2's weights have left snap[b_]
                for bank, g, sn in zip(banks, gdev[b_], snap[b_]):
                    bank.grad = g
                    bank.bank_copy = sn
                nss.muon_multi_step(banks, wl.lr, wl.wd, wl.mu, normuon=wl.normuon, beta2=wl.beta2,
                                    ns_steps=wl.ns_steps, workspace=ws, flags=args.step_flags)
                ev_gfree[b_].record(main_s)
                ev_snap[b_].record(main_s)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(ev_snap[b_])
                    for ho, sn in zip(host_out[b_], snap[b_]):
                        ho.copy_(sn, non_blocking=True)
                    ev_d2h[b_].record(d2h_s)
            main_s.wait_event(ev_d2h[(n - 1) & 1])

        k_e2e = max(1, min(args.steps, 50))
        e2e_run(3)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(main_s)
        e2e_run(k_e2e)
        e1.record(main_s)
        torch.cuda.synchronize()
        for bank in banks:
            bank.bank_copy = None
        e2e_ms = max_over_ranks(max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3), dev)
        e2e = {"value": job_rate(world, k_e2e, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": k_e2e,
               "what": "pinned host gradients -> device, muon_multi_step (its update also writes the new bf16 "
                       "weights to a second device buffer), that buffer -> pinned host; copies on two copy "
                       "streams overlap the neighbouring steps' compute"}

    if rank == 0:
        line = {
            "impl": "native", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded PCG64 banks; low-rank-plus-noise gradients, two alternating steps)",
            "config": config_of(wl, args),
            "roofline": roofline,
            "ns_tflops": ns_tflops,
            "ns_tflops_dense_equiv": r["ns_tflops_dense_equiv"],
            "momentum_gbs": mom_gbs, "update_gbs": upd_gbs,
            **({"normuon_rowstats_gbs": row_gbs} if row_gbs else {}),
            "last_newton_schulz_epilogue_also_does": r["last_epilogue"],
            "fractions": {"ns_of_bf16_burst": (ns_tflops / burst_peak) if ns_tflops else None,
                          "ns_of_bf16_sustained": (ns_tflops / sustained_peak) if ns_tflops else None,
                          "momentum_of_hbm": (mom_gbs / hbm_peak) if mom_gbs else None,
                          "update_of_hbm": (upd_gbs / hbm_peak) if upd_gbs else None,
                          **({"normuon_rowstats_of_hbm": row_gbs / hbm_peak} if row_gbs else {}),
                          "peaks": pk_kind},
            "stages_ms_per_step": per,
            "cpu_baseline": cpu_base,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": t["clocks"],
            **({"gpt2_medium_normuon": extra} if extra else {}),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
