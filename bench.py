"""Benchmark of the Muon optimizer step (libmuon on one GB300 per rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-cublas-side]

A step is one full Muon step (momentum, normalisation, five Newton-Schulz
iterations, weight update) over every matrix of the workload, with a fresh
synthetic gradient written before each step (outside the timed events).
The headline workload is the 4096 x 4096 bf16 matrix; the Qwen3-30B-A3B
block (388 matrices) is timed in the same run and reported under
"workloads" (--extra-workloads).
The metric is Muon-step TFLOP/s in useful FLOPs (symmetric products counted
on their upper triangle); GEMM-equivalent TFLOP/s, % of the measured dense
bf16 peak, ms/step and matrices/s are reported beside it.  L2 is flushed
before every timed step (a 512 MiB write, then a 512 MiB read that carries
the write's dirty lines out before the step begins).  Prints one JSON line on rank 0.
"cublas_side" times the same step written with torch operations (cuBLAS
batched matmuls) on the same workload, as a side comparison.

With N > 1 (torchrun) every rank runs the whole workload on its own GPU as an
independent replica (weak scaling); value = all ranks' FLOPs / the slowest
rank's time.  --impl reference times the float64 CPU oracle instead, on a
bounded sample of the same workload, with the same metric.
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

METRIC = ("Muon-step TFLOP/s (useful & GEMM-equiv) and % bf16 peak; "
          "ms/step per layer set")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,"
         "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        mx = max(r[1] for r in rows)
        loaded = [r for r in rows if r[0] > 0.5 * mx] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[2])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


def source_sha(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel and on this workload; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    ent = json.load(open(p)).get(f"{kernel}@{workload}")
    if not ent:
        return None
    if ent.get("source_sha") != source_sha(ent.get("source_files", [])):
        return None
    return ent.get("bytes_per_launch_full_workload")


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(wl, max_flops=2.2e12):
    """A bounded sample of the workload for the CPU oracle: its matrices in
    order until about `max_flops` GEMM-equivalent FLOPs (at least one)."""
    from newton_schulz_06_gb300 import flops
    picked, tot = [], 0
    for i, s in enumerate(wl.shapes):
        f = flops.gemm_equiv_flops([s], mode=wl.mode, nb=wl.nb)
        if picked and tot + f > max_flops:
            continue
        picked.append(i)
        tot += f
        if tot >= max_flops:
            break
    return picked


def time_oracle(wl, idx_list, host_inputs, reps=1):
    """Seconds per oracle step over the sampled matrices, useful FLOPs."""
    import numpy as np
    import oracle
    from newton_schulz_06_gb300 import flops
    a, b, c = (float(np.float32(x)) for x in (3.4445, -4.7750, 2.0315))
    useful = flops.useful_flops([wl.shapes[i] for i in idx_list],
                                mode=wl.mode, nb=wl.nb)
    t0 = time.perf_counter()
    for _ in range(reps):
        for W, G, M in host_inputs:
            oracle.muon_step(W, G, M, lr=0.02, beta=float(np.float32(0.95)),
                             nesterov=True, ns_steps=5, a=a, b=b, c=c,
                             mode=wl.mode, nb=wl.nb)
    return (time.perf_counter() - t0) / reps, useful


def host_sample(wl, idx_list):
    """Float64 host copies of the sampled matrices' first-step inputs,
    generated on the CPU from the same seeded recipe."""
    import torch
    from newton_schulz_06_gb300 import inputs as I
    out = []
    for i in idx_list:
        r, c = wl.shapes[i]
        W = I.make_weight((r, c), wl.w_dtype, "cpu", wl.name, i)
        M = I.make_momentum((r, c), wl.init_momentum, "cpu", wl.name, i)
        G = torch.empty((r, c), dtype=wl.g_dtype)
        I.fill_grad(G, wl, i, 0)
        out.append(tuple(t.to(torch.float64).numpy() for t in (W, G, M)))
    return out


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, wl, world, rank):
    if rank != 0:
        return None
    from newton_schulz_06_gb300 import flops
    idx = oracle_sample(wl)
    host = host_sample(wl, idx)
    full_useful = flops.useful_flops(wl.shapes, mode=wl.mode, nb=wl.nb)
    times = []
    for k in range(args.warmup + args.steps):
        dt, useful = time_oracle(wl, idx, host)
        if k >= args.warmup:
            times.append(dt)
    sec = statistics.mean(times)
    tflops = useful / sec / 1e12
    sample = (f"{len(idx)} of {wl.n_matrices} matrices "
              f"({useful / full_useful:.3%} of the step's useful FLOPs), "
              f"one float64 oracle step each per timed step")
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec * 1e3 * full_useful / useful,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "matrices": wl.n_matrices,
                   "mode": wl.mode, "nb": wl.nb, "ns_steps": 5},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s",
                         "cores": cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


# pinned host memory the end-to-end leg may take (G and W of its matrices)
E2E_MAX_HOST_BYTES = 8 << 30


class L2Flush:
    """Empties L2 of the workload's data between timed steps: writes a
    buffer four times the 129 MB L2, then reads a second one of the same
    size, so that the write's own dirty lines are written back here, not by
    the step that follows (which would otherwise pay for up to 129 MB of
    write-back it did not cause)."""
    BYTES = 512 * 1024 * 1024

    def __init__(self, dev):
        import torch
        self.w = torch.empty(self.BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(self.BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def device_timing(wl, args, dev, pg, steps):
    """Builds the workload's state on `dev` and times `steps` Muon steps
    (after the warm-up), each between CUDA events on the launch stream with
    L2 flushed before it; then `steps` more with libmuon's per-launch events
    for the stage split.  Returns the handle, its tensors and the timings."""
    import torch
    from newton_schulz_06_gb300 import Muon, mode_code
    from newton_schulz_06_gb300 import inputs as I
    Ws, Gs, Ms = I.make_state(wl, dev)
    trips = list(zip(Ws, Gs, Ms))
    opt = Muon(trips)
    mode = mode_code(wl.mode)
    opt.ensure_workspace(mode, wl.nb, args.max_workspace)
    info = opt.plan_info(mode, wl.nb)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def fresh_grads(step):
        for i, G in enumerate(Gs):
            if wl.grad == "log_scale_step" or step == 0:
                I.fill_grad(G, wl, i, step)

    kw = dict(lr=0.02, beta=0.95, nesterov=True, ns_steps=5, mode=mode,
              nb=wl.nb)
    for k in range(args.warmup):
        fresh_grads(k + 1)
        opt.step(**kw)
    opt.sync()
    torch.cuda.synchronize()

    # timed region: K steps, each between CUDA events on the launch stream;
    # no per-launch events here (they would serialise the kernels'
    # programmatic launch overlap)
    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(pg)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    launches = 0
    for k in range(steps):
        fresh_grads(args.warmup + k + 1)
        flush()
        ev[k][0].record(stream)
        opt.step(**kw)
        ev[k][1].record(stream)
        launches += opt.last_launch_count()
    torch.cuda.synchronize()
    barrier(pg)
    wall = time.perf_counter() - wall0
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    # per-kernel durations: K more steps right after, with CUDA events
    # around every launch (libmuon's stage timing, on the same stream)
    opt.set_profiling(True)
    stage_tot = {}
    prof_ms = []
    for k in range(steps):
        fresh_grads(args.warmup + steps + k + 1)
        flush()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        opt.step(**kw)
        a1.record(stream)
        opt.sync()
        prof_ms.append(a0.elapsed_time(a1))
        for name, (tms, n) in opt.stage_times().items():
            t, c = stage_tot.get(name, (0.0, 0))
            stage_tot[name] = (t + tms, c + n)
    opt.set_profiling(False)
    del flush
    return dict(opt=opt, trips=trips, kw=kw, info=info, ms=ms, wall=wall,
                launches=launches, stage_tot=stage_tot, prof_ms=prof_ms,
                fresh_grads=fresh_grads)


def roofline_of(wl, t, peak, peak_kind):
    """The dominant tensor-core kernel of a timed workload: per-launch
    algorithmic FLOPs / its mean event-timed launch duration."""
    from newton_schulz_06_gb300 import flops
    stage_tot, info = t["stage_tot"], t["info"]
    units = []
    for r, c in wl.shapes:
        units += flops.unit_shapes(r, c, wl.mode, wl.nb)
    per_launch = {
        "gemm": sum(2 * m * m * n for m, n in units),
        "syrk1": sum(m * (m + 1) * n for m, n in units),
        "syrk2": sum(m * (m + 1) * m for m, n in units),
    }
    # a chained launch runs every product of the step, the last X update too
    # unless that one ran as its own launch
    ns = t["kw"].get("ns_steps", 5)
    gemm_alone = stage_tot.get("gemm", (0, 0))[1] > 0
    per_launch["chain"] = (ns * (per_launch["syrk1"] + per_launch["syrk2"])
                           + (ns - 1 if gemm_alone else ns) * per_launch["gemm"])
    dom = max((k for k in per_launch if stage_tot.get(k, (0, 0))[1]),
              key=lambda k: stage_tot[k][0])
    t_dom, n_dom = stage_tot[dom]
    avg_launch_s = t_dom / n_dom / 1e3
    # per_launch counts every unit; with the workspace split into groups each
    # unit is in one group's launch, so the mean launch holds 1/groups of it
    # (all groups chained alike, as they are for these workloads)
    achieved = per_launch[dom] / max(1, info["groups"]) / avg_launch_s / 1e12
    op = {"gemm": 2, "syrk1": 0, "syrk2": 1, "chain": 3}[dom]
    pair = os.environ.get("MUON_CTA_GROUP", "2") != "1"
    kname = f"ns2_kernel<{op}>" if pair else f"ns_kernel<{op}>"
    return {"bound": "tensor", "kernel": kname, "stage": dom,
            "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak,
            "peak_kind": f"{peak_kind} dense bf16 (burst)",
            "traffic": traffic_for(kname, wl.name),
            "avg_launch_ms": t_dom / n_dom,
            "timing": "CUDA events around each launch of the kernel, on its stream, "
                      "over K steps run right after the timed region"}


def e2e_leg(wl, args, t, dev, pg, useful):
    """End to end through the C ABI with host buffers (muon_step_host): the
    step's gradients in from pinned memory, the step, the weights back out,
    timed on the host.  Pinned host memory is bounded: a workload whose G and
    W exceed E2E_MAX_HOST_BYTES runs this leg on its leading matrices, on a
    handle of their own."""
    import torch
    from newton_schulz_06_gb300 import Muon, flops
    opt, trips, kw = t["opt"], t["trips"], t["kw"]
    Ws = [x[0] for x in trips]
    Gs = [x[1] for x in trips]
    flush = L2Flush(dev)
    e2e_n = len(Gs)
    host = 0
    for i in range(len(Gs)):
        host += Gs[i].numel() * Gs[i].element_size() + Ws[i].numel() * Ws[i].element_size()
        if host > E2E_MAX_HOST_BYTES:
            e2e_n = max(1, i)
            break
    e2e_opt = opt
    e2e_useful = useful
    if e2e_n < len(Gs):
        e2e_opt = Muon(trips[:e2e_n])
        e2e_opt.ensure_workspace(kw["mode"], wl.nb, args.max_workspace)
        e2e_useful = flops.useful_flops(wl.shapes[:e2e_n], mode=wl.mode, nb=wl.nb)
    pinned_g = [torch.empty(G.shape, dtype=G.dtype, pin_memory=True)
                for G in Gs[:e2e_n]]
    for i, G in enumerate(Gs[:e2e_n]):
        pinned_g[i].copy_(G)
    pinned_w = [torch.empty(W.shape, dtype=W.dtype, pin_memory=True)
                for W in Ws[:e2e_n]]
    h2d = sum(x.numel() * x.element_size() for x in pinned_g)
    d2h = sum(x.numel() * x.element_size() for x in pinned_w)
    # two untimed calls first: the first copy into freshly pinned pages is
    # several times slower than later ones, and the first call builds the
    # pipelined plan (groups cut so that copies overlap compute)
    for k in range(2):
        e2e_opt.step_host(pinned_g, pinned_w, **kw)
        e2e_opt.sync()
    e2e_ms = []
    for k in range(max(3, min(args.steps, 10))):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_opt.step_host(pinned_g, pinned_w, **kw)
        e2e_opt.sync()
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e = max_over_ranks(pg, statistics.mean(e2e_ms))
    if e2e_opt is not opt:
        e2e_opt.close()
    del pinned_g, pinned_w, flush
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": world * e2e_useful / (e2e / 1e3) / 1e12,
            "unit": "TFLOP/s", "ms_per_step": e2e,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": ("muon_step_host: G from pinned host memory, the step, W back; "
                     "groups of about 1/16 of the set, copies on two streams overlapping "
                     "other groups' compute"),
            "matrices": e2e_n if e2e_n < len(Gs) else "all"}


# the side comparison stacks each shape's W, G and M (about 30 B per element
# with its temporaries): up to the Kimi-K2 layer, not the 48-layer set
CUBLAS_SIDE_MAX_ELEMENTS = 4 << 30


def cublas_side(wl, args, dev, useful, ours_ms):
    """The same Muon step written with torch operations, timed like the
    libmuon step (L2 flushed before each step, CUDA events on the stream): a
    side comparison of what the fused kernels replace, not a path of the
    library (none of its kernels run here).  Matrices of one shape are
    stacked; every product is a cuBLAS bf16 batched matmul with fp32
    accumulation, the symmetric ones computed in full, b*A + c*A*A and
    a*X + B*X folded into the matmuls (baddbmm); momentum, norm and update
    are separate element-wise kernels.  Full mode only, and only for
    workloads whose stacked state fits beside the bench's own."""
    import torch
    from newton_schulz_06_gb300 import inputs as I
    from newton_schulz_06_gb300.muon import DEFAULT_COEFFS
    if args.no_cublas_side or wl.mode != "full" or wl.n_elements > CUBLAS_SIDE_MAX_ELEMENTS:
        return None
    Ws, Gs, Ms = I.make_state(wl, dev)
    by_shape = {}
    for i, shape in enumerate(wl.shapes):
        by_shape.setdefault(tuple(shape), []).append(i)
    sets = []
    for (r, c), idx in by_shape.items():
        sets.append((r, c, torch.stack([Ws[i] for i in idx]), torch.stack([Gs[i] for i in idx]),
                     torch.stack([Ms[i] for i in idx])))
    del Ws, Gs, Ms
    a, b, c3 = DEFAULT_COEFFS
    beta, lr, eps = 0.95, 0.02, 1e-7

    def step():
        for r, c, W, G, M in sets:
            M.mul_(beta).add_(G)
            U = torch.add(G, M, alpha=beta)                  # Nesterov
            X = U.transpose(1, 2) if r > c else U
            inv = 1.0 / (torch.linalg.vector_norm(X, dim=(1, 2), keepdim=True) + eps)
            X = (X * inv).to(torch.bfloat16)
            for _ in range(5):
                A = torch.bmm(X, X.transpose(1, 2))
                B = torch.baddbmm(A, A, A, beta=b, alpha=c3)
                X = torch.baddbmm(X, B, X, beta=a, alpha=1.0)
            O = X.transpose(1, 2) if r > c else X
            W.add_(O, alpha=-lr * max(1.0, r / c) ** 0.5)

    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(min(args.steps, 10))]
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    del sets, flush
    torch.cuda.empty_cache()
    return {"ms_per_step": ms, "useful_tflops": useful / (ms / 1e3) / 1e12,
            "libmuon_speedup": ms / ours_ms, "steps": len(ev),
            "what": ("the same step in torch ops: cuBLAS bf16 batched matmuls (fp32 "
                     "accumulation), symmetric products in full, matrices of one shape "
                     "stacked; a side comparison, not a path of the library")}


def run_ours(args, wl, world, rank, local, pg):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from newton_schulz_06_gb300 import flops
    from newton_schulz_06_gb300 import inputs as I

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    peaks, peak_kind = load_peaks()
    peak = peaks["bf16_tflops"]
    # the power-capped figure, for context beside the burst one: long,
    # grouped steps run under the power limit
    peak_sus = peaks.get("bf16_tflops_sustained", peak)
    useful = flops.useful_flops(wl.shapes, mode=wl.mode, nb=wl.nb)
    gemm_eq = flops.gemm_equiv_flops(wl.shapes, mode=wl.mode, nb=wl.nb)
    # clocks are sampled from the first warm-up step to the end of the
    # last measurement, a window that contains the timed regions
    sampler = ClockSampler(local)
    sampler.start()
    t = device_timing(wl, args, dev, pg, args.steps)
    opt, trips, kw, info = t["opt"], t["trips"], t["kw"], t["info"]
    ms = max_over_ranks(pg, t["ms"])
    stage_tot = t["stage_tot"]
    e2e = e2e_leg(wl, args, t, dev, pg, useful)
    roofline = roofline_of(wl, t, peak, peak_kind)
    prof_ms, wall, launches = t["prof_ms"], t["wall"], t["launches"]
    opt.close()
    del opt, trips, t
    torch.cuda.empty_cache()
    side = cublas_side(wl, args, dev, useful, ms) if world == 1 else None

    # further workloads timed in the same run (the target configs besides
    # the headline one), each with its own state, freed before the next
    extra = {}
    for name in [x for x in args.extra_workloads.split(",") if x and x != "none"]:
        xw = I.workload(name)
        torch.cuda.empty_cache()
        xt = device_timing(xw, args, dev, pg, min(args.steps, 10))
        xu = flops.useful_flops(xw.shapes, mode=xw.mode, nb=xw.nb)
        xg = flops.gemm_equiv_flops(xw.shapes, mode=xw.mode, nb=xw.nb)
        xms = max_over_ranks(pg, xt["ms"])
        extra[name] = {
            "matrices": xw.n_matrices, "mode": xw.mode, "nb": xw.nb,
            "steps": min(args.steps, 10), "warmup": args.warmup,
            "ms_per_step": xms,
            "useful_tflops": world * xu / (xms / 1e3) / 1e12,
            "gemm_equiv_tflops": world * xg / (xms / 1e3) / 1e12,
            "pct_bf16_peak_useful": 100.0 * xu / (xms / 1e3) / 1e12 / peak,
            "pct_bf16_peak_gemm_equiv": 100.0 * xg / (xms / 1e3) / 1e12 / peak,
            "pct_bf16_sustained_peak_useful": 100.0 * xu / (xms / 1e3) / 1e12 / peak_sus,
            "stage_ms_per_step": {k: v[0] / len(xt["prof_ms"])
                                  for k, v in xt["stage_tot"].items()},
            "ms_per_step_with_stage_events": statistics.mean(xt["prof_ms"]),
            "gpu_launches": xt["launches"],
            "roofline": roofline_of(xw, xt, peak, peak_kind),
            "e2e": e2e_leg(xw, args, xt, dev, pg, xu),
        }
        xt["opt"].close()
        del xt
        torch.cuda.empty_cache()
        xs = cublas_side(xw, args, dev, xu, xms) if world == 1 else None
        if xs:
            extra[name]["cublas_side"] = xs
    clocks = sampler.stop()

    value = world * useful / (ms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "matrices": wl.n_matrices,
                   "elements": wl.n_elements, "mode": wl.mode, "nb": wl.nb,
                   "ns_steps": 5, "groups": info["groups"],
                   "l2": ("flushed before every timed step: 512 MiB written, then 512 MiB "
                          "read so that the write's dirty lines leave L2 before the step"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "gemm_equiv_tflops": world * gemm_eq / (ms / 1e3) / 1e12,
        "pct_bf16_peak_useful": 100.0 * useful / (ms / 1e3) / 1e12 / peak,
        "pct_bf16_peak_gemm_equiv": 100.0 * gemm_eq / (ms / 1e3) / 1e12 / peak,
        "pct_bf16_sustained_peak_useful": 100.0 * useful / (ms / 1e3) / 1e12 / peak_sus,
        "matrices_per_s": world * wl.n_matrices / (ms / 1e3),
        "useful_tflop_per_step": useful / 1e12,
        "gemm_equiv_tflop_per_step": gemm_eq / 1e12,
        # the plan's tiles per iteration (256 x 256 tiles on CTA pairs) and
        # the FLOPs the tensor cores execute (diagonal tiles whole, edge
        # tiles padded) over the useful ones
        "plan": {"units": info["units"], "groups": info["groups"],
                 "symmetric_product_tiles": info["syrk_tiles"],
                 "x_update_tiles": info["gemm_tiles"],
                 "elementwise_tiles": info["ew_tiles"],
                 "chained_groups": info["chained_groups"],
                 "executed_over_useful_flops": info["executed_flops"] / max(1, info["useful_flops"])},
        "stage_ms_per_step": {k: v[0] / args.steps for k, v in stage_tot.items()},
        "ms_per_step_with_stage_events": statistics.mean(prof_ms),
        "wall_s_timed_region": wall,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches,
        "roofline": roofline,
    }
    if side:
        line["cublas_side"] = side
    if extra:
        line["workloads"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        idx = oracle_sample(wl)
        host = host_sample(wl, idx)
        dt, u = time_oracle(wl, idx, host)
        full_useful = flops.useful_flops(wl.shapes, mode=wl.mode, nb=wl.nb)
        line["cpu_baseline"] = {
            "value": u / dt / 1e12, "unit": "TFLOP/s", "cores": cores(),
            "kind": "oracle",
            "sample": (f"{len(idx)} of {wl.n_matrices} matrices "
                       f"({u / full_useful:.3%} of the step's useful FLOPs), "
                       f"one float64 oracle step, {dt:.1f} s")}
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="square_4096_bf16")
    ap.add_argument("--max-workspace", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cublas-side", action="store_true",
                    help="skip the side comparison with the step in torch/cuBLAS ops")
    ap.add_argument("--extra-workloads", default="qwen3_30b_a3b_block",
                    help="comma-separated workloads also timed in the same run "
                         "and reported under 'workloads' ('none': skip)")
    ap.add_argument("--max-matrices", type=int, default=None,
                    help="profiling aid: keep only the first N matrices")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from newton_schulz_06_gb300 import inputs as I
    wl = I.workload(args.workload)
    if args.max_matrices:
        wl.shapes = wl.shapes[:args.max_matrices]
        wl.name = f"{wl.name}[:{args.max_matrices}]"
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, wl, world, rank)
    else:
        line = run_ours(args, wl, world, rank, local, pg)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
