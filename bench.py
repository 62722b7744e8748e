"""Benchmark of the fused registration objective (MI + LNCC, forward + backward).

One step = one ffdp_objective call on the 512^3 fp32 phantom pair (MI with 64
bins + LNCC with a 5^3 window, gradients to u, A and t): every row of the hot
path -- implicit sampler, histogram sweep, MI table, LNCC window sums, MI and
LNCC gradients, sampler backward, affine reductions.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 4|5] [--impl reference]
    python bench.py --path mse|compose|adam (the MSE objective / warp composition / the
                                            regularised Adam step of u on the 512^3
                                            pair; one JSON line each, same keys)

Under torch.distributed.run each rank evaluates its own independent pair
(weak scaling, no collective on the data path); the step time is the maximum
over ranks.  Rank 0 prints one JSON line.  --impl reference times the CPU
oracle (double precision, all host cores) on a bounded z-slab of the same
workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Gvoxels/s fused warp+MI/LNCC fwd+bwd on 1 GB300; % of HBM roofline"
UNIT = "Gvoxels/s"
# Algorithmic bytes per voxel (inputs read once per sweep, du written once):
# MI needs two sweeps because the histogram is a global dependency.
ALGO_BYTES = {4: 2 * (4 + 12 + 4) + 12, 5: 2 * (2 + 12 + 2) + 12}
# Single-pass lower bound: F, M and u read once, du written once.
SINGLE_PASS_BYTES = {4: 4 + 4 + 12 + 12, 5: 2 + 2 + 12 + 12}
# Algorithmic bytes per voxel of each kernel of the objective:
#   k_sweep1  F + u + M read (+ J and dJ/dq written when LNCC is on)
#   k_lncc_fw J + F read, the three g-terms written (forward window sums, cc)
#   k_lncc_bw g-terms + J + F + dJ/dq read, du written (backward window sums,
#             dL/dJ with the MI term, the sampler backward)
#   k_lncc    (the fused kernel of the FFDP_LNCC_FUSED build) F + J + dJ/dq
#             read, du written
#   k_sweep2  MI: F + u + M read, du written
#   (MI-only with stored J and slope: k_sweep1 also writes J + dJ/dq; k_sweep2
#   reads F + J + dJ/dq and writes du)
KERNEL_BYTES = {4: {"k_sweep1": 4 + 12 + 4 + 4 + 12, "k_lncc_fw": 4 + 4 + 12, "k_lncc_bw": 12 + 4 + 4 + 12 + 12,
                    "k_lncc": 4 + 4 + 12 + 12},
                5: {"k_sweep1": 2 + 12 + 2, "k_sweep2": 2 + 12 + 2 + 12}}
KERNEL_BYTES_STORED = {5: {"k_sweep1": 2 + 12 + 2 + 4 + 12, "k_sweep2": 2 + 4 + 12 + 12}}
# LNCC windows above 7 (--window): separable passes through two [5][N]
# buffers instead of k_lncc -- x sums of the products (J, F read, 5 sums
# written), y sums (5 + 5), z sums with cc and the g-terms (5 + 3), x and y
# sums of the g-terms (3 + 3 each), z sums with dL/dJ and the sampler backward
# (3 sums, F, J, dJ/dq read, du written)
KERNEL_BYTES_WIDE = {"k_sweep1": 4 + 12 + 4 + 4 + 12, "k_wide_prod_x": 4 + 4 + 20, "k_wide_y": 20 + 20,
                     "k_wide_cc": 20 + 12, "k_wide_gx": 12 + 12, "k_wide_gy": 12 + 12,
                     "k_wide_fin": 12 + 4 + 4 + 12 + 12}


def _kernel_bytes(args, wl):
    if wl.w_lncc != 0.0 and _window(args, wl) > 7:
        return KERNEL_BYTES_WIDE
    if wl.w_lncc == 0.0 and args.store_slope and args.workload in KERNEL_BYTES_STORED:
        return KERNEL_BYTES_STORED[args.workload]
    return KERNEL_BYTES[args.workload]
HBM_NOMINAL_GBS = 8000.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def _max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _aggregate_gvox(N, ws, ms):
    """Whole-job throughput: every rank evaluates its own N-voxel pair (weak
    scaling), timed by the slowest rank."""
    return N * ws / (ms * 1e-3) / 1e9


def _crop_transform(pair, ds):
    """x_bounds of the first ds planes of the fixed grid (same sample points)."""
    D = pair.F.shape[0]
    xmax = pair.xmax.copy()
    xmax[2] = pair.xmin[2] + (pair.xmax[2] - pair.xmin[2]) * (ds - 1) / (D - 1)
    return xmax


def _window(args, wl):
    """LNCC window of the run: the workload's, or --window."""
    return args.window if getattr(args, "window", 0) else wl.window


def oracle_sample(pair, ds, threads=None, window=None):
    """Time the CPU oracle on the first ds planes of the workload (one fwd+bwd)."""
    import oracle
    wl = pair.workload
    if threads:
        oracle.set_threads(threads)
    F = pair.F[:ds].float().cpu().numpy()
    M = pair.M.float().cpu().numpy()
    u = pair.u[:ds].cpu().numpy()
    xmax = _crop_transform(pair, ds)
    T = oracle.Transform(pair.A.astype(np.float64), pair.t.astype(np.float64), pair.S.astype(np.float64),
                         pair.xmin.astype(np.float64), xmax.astype(np.float32).astype(np.float64))
    P = oracle.ObjectiveParams(wl.w_mi, wl.w_lncc, wl.bins, pair.f_range, pair.m_range, window or wl.window,
                               wl.eps)
    t0 = time.perf_counter()
    if wl.w_lncc != 0.0:
        oracle.objective(F, M, u, T, P)
    else:
        oracle.objective_mi_slabs(F, M, u, T, P, slab=8)
    dt = time.perf_counter() - t0
    return F.size, dt, oracle.max_threads()


def _cpu_small(dev):
    """The oracle on the two small workloads in full (64^3 MI 32 + LNCC 5; 160x192x224
    MI 32), on one thread and on every host thread: context for the CPU baseline."""
    import oracle
    from voxel_grid_sampler_gb300 import synth
    cores = len(os.sched_getaffinity(0))
    res = {}
    try:
        for k in (1, 2):
            pair = synth.make_pair(k, device=dev)
            name = pair.workload.name
            r = {}
            for th in (1, cores):
                n, t, used = oracle_sample(pair, pair.F.shape[0], threads=th)
                r["threads_%d" % used] = {"value": n / t / 1e9, "unit": UNIT, "s": t}
            res[name] = r
            del pair
    finally:
        oracle.set_threads(cores)
    return res


def _sample_planes(pair, budget_s=12.0, window=None):
    """Planes of the bounded CPU sample: ~budget_s seconds of oracle work."""
    import oracle
    n1, t1, _ = oracle_sample(pair, 2, window=window)
    per_plane = t1 / 2.0
    ds = int(max(2, min(pair.F.shape[0], budget_s / max(per_plane, 1e-3))))
    return ds


def run_reference(args, ws, rank, local):
    from voxel_grid_sampler_gb300 import synth
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    pair = synth.make_pair(args.workload, device=dev)
    pair.F, pair.M, pair.u = pair.F.cpu(), pair.M.cpu(), pair.u.cpu()
    # each step a bounded sample so that warm-up + timed steps end within ~3 minutes
    budget = min(args.ref_step_s, 150.0 / max(1, args.steps + args.warmup))
    win = _window(args, pair.workload)
    ds = _sample_planes(pair, budget_s=budget, window=win)
    for _ in range(args.warmup):
        oracle_sample(pair, ds, window=win)
    times = []
    cores = 1
    for _ in range(args.steps):
        n, t, cores = oracle_sample(pair, ds, window=win)
        times.append(t)
    t = sum(times) / len(times)
    value = n / t / 1e9
    wl = pair.workload
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "shape": list(pair.F.shape), "lncc_window": win, "sample_planes": ds},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "oracle objective on fixed planes z<%d of the %s pair (%d voxels)"
                                   % (ds, "x".join(map(str, pair.F.shape)), n)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def _traffic_per_launch(kernel, workload, N):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    record (bytes per voxel x N), or None when the kernel's sources changed
    since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        import hashlib
        with open(p) as f:
            d = json.load(f)
        for rec in d.get("records", []):
            if rec.get("kernel") != kernel or rec.get("workload") != workload:
                continue
            src = "".join(open(os.path.join(ROOT, "voxel_grid_sampler_gb300", "csrc", s)).read()
                          for s in sorted(rec["sources"]))
            if hashlib.sha256(src.encode()).hexdigest()[:16] != rec["source_sha"]:
                return None
            return rec["bytes_per_voxel"] * N
    except Exception:
        return None
    return None


def _time_steps(step, n, stream, dev, ws, clocks=None):
    """Device time of n back-to-back steps (CUDA events on the launching stream,
    synchronised and barriered on both sides), max over ranks.  Returns the ms
    per step and the library launches inside the timed region."""
    from voxel_grid_sampler_gb300 import ffdp
    n0 = ffdp.launch_count()
    _barrier(ws)
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.start()
        time.sleep(0.15)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    _barrier(ws)
    clk = clocks.stop() if clocks is not None else None
    launches = ffdp.launch_count() - n0
    ms = _max_over_ranks(e0.elapsed_time(e1) / n, ws, dev)
    return ms, launches, clk


def _kernel_times(step, n, dev):
    """Per-kernel device times from a separate, instrumented pass of n steps
    (CUDA events around every launch); the headline loop runs without them."""
    from voxel_grid_sampler_gb300 import ffdp
    ffdp.timing_enable(n * 8)
    for _ in range(n):
        step()
    torch.cuda.synchronize(dev)
    kern = ffdp.timing_read()
    ffdp.timing_enable(0)
    return kern


def _roofline(kern, kb, N, peak, peak_kind, traffic_of):
    """Roofline of the dominant kernel: its algorithmic bytes per launch over
    its average launch time, against the copy-bandwidth peak."""
    dom_name, (dom_n, dom_ms) = max(kern.items(), key=lambda kv: kv[1][1])
    dom_avg = dom_ms / max(dom_n, 1)
    bpv = kb.get(dom_name, 0)
    achieved = bpv * N / (dom_avg * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": traffic_of(dom_name), "kernel": dom_name,
            "algorithmic_bytes_per_voxel": bpv, "peak_source": peak_kind,
            "kernels": {k: {"ms": v[1] / max(v[0], 1), "bytes_per_voxel": kb.get(k, 0),
                            "frac": kb.get(k, 0) * N / (v[1] / max(v[0], 1) * 1e-3) / 1e9 / peak}
                        for k, v in kern.items() if k in kb}}


def run_gpu(args, ws, rank, local):
    from voxel_grid_sampler_gb300 import build, ffdp, synth
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    shape = None if not args.shape else (args.shape,) * 3
    pair = synth.make_pair(args.workload, device=dev, shape=shape, seed=1000 + args.workload + 100 * rank)
    wl = pair.workload
    F, M, u = pair.F, pair.M, pair.u
    N = F.numel()
    T = ffdp.transform(pair.A, pair.t, pair.S, pair.xmin, pair.xmax)
    P = ffdp.objective_params(wl.w_mi, wl.w_lncc, wl.bins, pair.f_range, pair.m_range, _window(args, wl), wl.eps)
    stored = bool(args.store_slope)  # ffdp_objective_stored (MI only: J and slope kept) or ffdp_objective
    wsbuf = ffdp.workspace(_ws_op(stored), F.shape, P, dev)
    loss = torch.empty(3, device=dev)
    du = torch.empty(tuple(F.shape) + (3,), device=dev)
    dA = torch.empty(9, device=dev)
    dt = torch.empty(3, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ffdp.ffdp_objective(F, M, u, T, P, loss, du, dA, dt, wsbuf, stream, store_slope=stored)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)

    # ---- device-resident timed region: plain calls, no per-launch events
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    ms, launches, clk = _time_steps(step, args.steps, stream, dev, ws, clocks)
    value = _aggregate_gvox(N, ws, ms)
    # per-kernel times from a separate instrumented pass
    kern = _kernel_times(step, max(3, min(args.steps, 10)), dev)

    # the other MI mode of an MI-only objective, timed the same way for reference
    alt = None
    if wl.w_lncc == 0.0:
        ws2 = ffdp.workspace(_ws_op(not stored), F.shape, P, dev)

        def step2():
            ffdp.ffdp_objective(F, M, u, T, P, loss, du, dA, dt, ws2, stream, store_slope=not stored)
        for _ in range(3):
            step2()
        torch.cuda.synchronize(dev)
        ms2, _, _ = _time_steps(step2, max(3, min(args.steps, 10)), stream, dev, ws)
        alt = {"mi_mode": _mi_mode(not args.store_slope), "ms_per_step": ms2}
        del ws2
        torch.cuda.empty_cache()
        step()  # leave the outputs of the timed mode in place
        torch.cuda.synchronize(dev)

    # ---- end to end through the public API with host buffers
    if args.no_e2e:
        ms_e2e, h2d, d2h = float("nan"), 0, 0
    else:
        ms_e2e, h2d, d2h = _e2e(args, F, M, u, T, P, loss, du, dA, dt, wsbuf, stream, dev, ws, stored)
    out = _rest(args, ws, rank, pair, wl, F, N, ms, kern, launches, clk, loss, ms_e2e, h2d, d2h, alt)
    # ---- the gigavoxel workload, timed the same way, on the same line
    if (out is not None and args.workload == 4 and not args.shape and not args.window and not args.no_workload5
            and ws == 1):
        del pair, F, M, u, wsbuf, du, step
        torch.cuda.empty_cache()
        out["workload5"] = _workload5(args, dev, stream)
    if out is not None:
        print(json.dumps(out), flush=True)


def _workload5(args, dev, stream):
    """The 1024^3 fp16 MI-32 objective (stored J and slope, the default mode),
    timed like the headline: plain calls between CUDA events, per-kernel times
    from a separate instrumented pass."""
    from voxel_grid_sampler_gb300 import ffdp, synth
    free, _ = torch.cuda.mem_get_info(dev)
    if free < 64 * 2 ** 30:
        return {"skipped": "needs 64 GiB of free device memory, %.1f GiB free" % (free / 2 ** 30)}
    t0 = time.perf_counter()
    pair = synth.make_pair(5, device=dev)
    gen_s = time.perf_counter() - t0
    wl = pair.workload
    F, M, u = pair.F, pair.M, pair.u
    N = F.numel()
    T = ffdp.transform(pair.A, pair.t, pair.S, pair.xmin, pair.xmax)
    P = ffdp.objective_params(wl.w_mi, wl.w_lncc, wl.bins, pair.f_range, pair.m_range, wl.window, wl.eps)
    wsbuf = ffdp.workspace(ffdp.FFDP_OP_OBJECTIVE_STORED, F.shape, P, dev)
    loss = torch.empty(3, device=dev)
    du = torch.empty(tuple(F.shape) + (3,), device=dev)
    dA = torch.empty(9, device=dev)
    dt = torch.empty(3, device=dev)

    def step():
        ffdp.ffdp_objective(F, M, u, T, P, loss, du, dA, dt, wsbuf, stream, store_slope=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(torch.cuda.current_device())
    n = max(3, min(args.steps, 10))
    ms, launches, clk = _time_steps(step, n, stream, dev, 1, clocks)
    kern = _kernel_times(step, 3, dev)
    peak, peak_kind = _peaks()
    kb = KERNEL_BYTES_STORED[5]
    step_gbs = ALGO_BYTES[5] * N / (ms * 1e-3) / 1e9
    res = {"workload": wl.name, "shape": list(F.shape), "voxels": N, "steps": n, "warmup": 3,
           "ms_per_step": ms, "value": N / (ms * 1e-3) / 1e9, "unit": UNIT, "gpu_launches": int(launches),
           "mi_mode": _mi_mode(True), "dtype": "f32 (f16 storage)", "generate_s": gen_s,
           "pct_hbm_roofline": {"step_algorithmic_gbs": step_gbs, "of_8tbs": step_gbs / HBM_NOMINAL_GBS,
                                "of_measured": step_gbs / peak, "bytes_per_voxel": ALGO_BYTES[5]},
           "roofline": _roofline(kern, kb, N, peak, peak_kind, lambda k: _traffic_per_launch(k, wl.name, N)),
           "kernels_ms_per_launch": {k: v[1] / max(v[0], 1) for k, v in kern.items()},
           "clocks": clk, "loss": [float(x) for x in loss.tolist()]}
    del pair, F, M, u, wsbuf, du
    torch.cuda.empty_cache()
    return res


def _ws_op(stored):
    from voxel_grid_sampler_gb300 import ffdp
    return ffdp.FFDP_OP_OBJECTIVE_STORED if stored else ffdp.FFDP_OP_OBJECTIVE


def _e2e(args, F, M, u, T, P, loss, du, dA, dt, wsbuf, stream, dev, ws, stored):
    """End to end through ffdp_objective with host buffers: every step copies F,
    M and u in from pinned host memory and du, the losses, dA and dt out.
    Double-buffered on three streams (copy in / compute / copy out, ordered
    by events), so step k+1's inputs and step k-1's results move while step k
    computes; each step's copies are complete inside the timed region."""
    from voxel_grid_sampler_gb300 import ffdp
    Fh = F.cpu().pin_memory()
    Mh = M.cpu().pin_memory()
    uh = u.cpu().pin_memory()
    duh = torch.empty(du.shape, dtype=du.dtype).pin_memory()
    outh = torch.empty(15, dtype=torch.float32).pin_memory()
    sets = []
    for _ in range(2):
        sets.append(dict(F=torch.empty_like(F), M=torch.empty_like(M), u=torch.empty_like(u),
                         du=torch.empty_like(du), small=torch.empty(15, device=dev),
                         loss=torch.empty(3, device=dev), dA=torch.empty(9, device=dev), dt=torch.empty(3, device=dev),
                         ev_in=torch.cuda.Event(), ev_comp=torch.cuda.Event(), ev_out=torch.cuda.Event(),
                         used=False))
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    comp = stream

    def e2e_step(i):
        b = sets[i % 2]
        if b["used"]:
            s_in.wait_event(b["ev_comp"])  # this set's previous inputs are consumed
        with torch.cuda.stream(s_in):
            b["F"].copy_(Fh, non_blocking=True)
            b["M"].copy_(Mh, non_blocking=True)
            b["u"].copy_(uh, non_blocking=True)
            b["ev_in"].record(s_in)
        comp.wait_event(b["ev_in"])
        if b["used"]:
            comp.wait_event(b["ev_out"])  # this set's previous results are copied out
        ffdp.ffdp_objective(b["F"], b["M"], b["u"], T, P, b["loss"], b["du"], b["dA"], b["dt"], wsbuf, comp,
                            store_slope=stored)
        with torch.cuda.stream(comp):
            b["small"][0:3].copy_(b["loss"])
            b["small"][3:12].copy_(b["dA"])
            b["small"][12:15].copy_(b["dt"])
        b["ev_comp"].record(comp)
        s_out.wait_event(b["ev_comp"])
        with torch.cuda.stream(s_out):
            duh.copy_(b["du"], non_blocking=True)
            outh.copy_(b["small"], non_blocking=True)
            b["ev_out"].record(s_out)
        b["used"] = True

    e2e_steps = max(4, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    _barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    s_out.wait_event(sets[(e2e_steps - 1) % 2]["ev_out"])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    _barrier(ws)
    ms_e2e = _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, ws, dev)
    h2d = F.numel() * F.element_size() + M.numel() * M.element_size() + u.numel() * u.element_size()
    d2h = du.numel() * du.element_size() + 15 * 4
    del Fh, Mh, uh, duh, sets
    torch.cuda.empty_cache()
    return ms_e2e, h2d, d2h


def _mi_mode(store):
    return ("stored J and dJ/dp (16 B/voxel workspace), streaming gradient pass" if store
            else "implicit (no per-voxel workspace), gradient pass gathers M again")


def _rest(args, ws, rank, pair, wl, F, N, ms, kern, launches, clk, loss, ms_e2e, h2d, d2h, alt=None):
    value = _aggregate_gvox(N, ws, ms)
    # ---- roofline of the dominant kernel (algorithmic bytes / its own time)
    peak, peak_kind = _peaks()
    roofline = _roofline(kern, _kernel_bytes(args, wl), N, peak, peak_kind,
                         lambda k: _traffic_per_launch(k, wl.name, N))
    step_gbs = ALGO_BYTES[args.workload] * N / (ms * 1e-3) / 1e9
    if rank != 0:
        return None
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if wl.dtype == "f32" else "f32 (f16 storage)",
        "data": "synthetic",
        "config": {"workload": wl.name, "shape": list(F.shape), "voxels": N, "lncc_window": _window(args, wl),
                   "l2": "inputs larger than L2 (%.2f GB algorithmic bytes per step)"
                         % (ALGO_BYTES[args.workload] * N / 1e9),
                   "parallelism": "independent pair per rank" if ws > 1 else "single GPU",
                   "mi_mode": (_mi_mode(bool(args.store_slope)) if wl.w_lncc == 0.0
                               else "LNCC on: J and dJ/dp stored (16 B/voxel workspace)")},
        "other_mode": alt,
        "pct_hbm_roofline": {"step_algorithmic_gbs": step_gbs,
                             "of_8tbs": step_gbs / HBM_NOMINAL_GBS,
                             "of_measured": step_gbs / peak,
                             "bytes_per_voxel": ALGO_BYTES[args.workload],
                             "single_pass_bytes_per_voxel": SINGLE_PASS_BYTES[args.workload],
                             "single_pass_of_8tbs": SINGLE_PASS_BYTES[args.workload] * N / (ms * 1e-3) / 1e9
                                                    / HBM_NOMINAL_GBS},
        "roofline": roofline,
        "kernels_ms_per_launch": {k: v[1] / max(v[0], 1) for k, v in kern.items()},
        "gpu_launches": int(launches),
        "clocks": clk,
        "e2e": None if args.no_e2e else {
            "value": N * ws / (ms_e2e * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e},
        "loss": [float(x) for x in loss.tolist()],
    }
    if ws == 1 and not args.no_cpu_baseline:
        ds = _sample_planes(pair, budget_s=args.cpu_budget_s, window=_window(args, wl))
        n, t, cores = oracle_sample(pair, ds, window=_window(args, wl))
        out["cpu_baseline"] = {"value": n / t / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": "oracle objective on fixed planes z<%d of the %s pair "
                                         "(%d voxels, %.1f s)" % (ds, "x".join(map(str, F.shape)), n, t)}
        if not args.shape and not args.window:
            out["cpu_small"] = _cpu_small(F.device)
    return out


# ---------------------------------------------------------------- other paths
# The fused MSE objective (one pass: F + u + M read, du written) and warp
# composition (forward: u + V read, out written; backward: u + gout + V read,
# du and dV written) on the 512^3 workload-4 pair; V is a second smooth
# displacement field (the pair's own field mirrored in z), gout a seeded
# normal field.
PATH_METRIC = {"mse": "Gvoxels/s fused warp+MSE fwd+bwd on 1 GB300; % of HBM roofline",
               "adam": "Gvoxels/s Sobolev-regularised Adam step of u on 1 GB300; % of HBM roofline",
               "compose": "Gvoxels/s warp composition fwd+bwd (du, dA, dt, dV) on 1 GB300; % of HBM roofline"}
PATH_KERNEL_BYTES = {"mse": {"k_sweep2": 4 + 12 + 4 + 12},
                     "adam": {"k_reg_adam": 12 * 7},
                     "compose": {"k_chan_fwd": 12 + 12 + 12, "k_chan_bwd": 12 + 12 + 12 + 12 + 12,
                                 "k_zero_f32": 12}}
PATH_ALGO_BYTES = {"mse": 32, "compose": 36 + 60, "adam": 84}


def _path_setup(args, pair, dev):
    from voxel_grid_sampler_gb300 import ffdp
    F, M, u = pair.F, pair.M, pair.u
    T = ffdp.transform(pair.A, pair.t, pair.S, pair.xmin, pair.xmax)
    shape = tuple(F.shape)
    if args.path == "mse":
        o = dict(loss=torch.empty(2, device=dev), du=torch.empty(shape + (3,), device=dev),
                 dA=torch.empty(9, device=dev), dt=torch.empty(3, device=dev),
                 ws=ffdp.workspace(ffdp.FFDP_OP_OBJECTIVE_MSE, shape, None, dev))

        def call(F_, M_, u_, o_, stream):
            ffdp.ffdp_objective_mse(F_, M_, u_, T, 1.0, o_["loss"], o_["du"], o_["dA"], o_["dt"], o_["ws"], stream)
        ins = dict(F=F, M=M, u=u)
        outs = ("loss", "du", "dA", "dt")
    elif args.path == "adam":
        # u, the objective gradient g (a seeded field of du's scale) and the moments in;
        # u_out, the moments and R(u) out (u is not advanced between steps)
        g = torch.Generator(device=dev).manual_seed(2025)
        gr = torch.randn(shape + (3,), device=dev, generator=g) * 1e-6
        o = dict(u_out=torch.empty_like(u), loss=torch.empty(1, device=dev),
                 ws=ffdp.workspace(ffdp.FFDP_OP_SOBOLEV, shape, None, dev))
        P = ffdp.sobolev_adam_params(0.1, 1e-3, 0.9, 0.999, 1e-8, 1)

        def call(u_, g_, m1_, m2_, o_, stream):
            ffdp.ffdp_sobolev_adam_step(u_, g_, m1_, m2_, P, o_["u_out"], o_["loss"], o_["ws"], stream)
        ins = dict(u=u, g=gr, m1=torch.zeros_like(u), m2=torch.zeros_like(u))
        outs = ("u_out", "loss")
    else:
        g = torch.Generator(device=dev).manual_seed(2024)
        gout = torch.randn(shape + (3,), device=dev, generator=g)
        o = dict(out=torch.empty(shape + (3,), device=dev), du=torch.empty(shape + (3,), device=dev),
                 dA=torch.empty(9, device=dev), dt=torch.empty(3, device=dev), dV=torch.empty_like(u),
                 ws=ffdp.workspace(ffdp.FFDP_OP_SAMPLE_CHANNELS_BWD, shape, None, dev))

        def call(V_, g_, u_, o_, stream):
            ffdp.ffdp_sample_channels_fwd(V_, shape, u_, T, True, o_["out"], stream)
            ffdp.ffdp_sample_channels_bwd(V_, u_, T, g_, True, o_["du"], o_["dA"], o_["dt"], o_["dV"], o_["ws"],
                                          stream)
        ins = dict(V=u.flip(0).contiguous(), g=gout, u=u)
        outs = ("out", "du", "dA", "dt", "dV")
    return call, ins, o, outs


def _path_oracle_sample(args, pair, ds):
    """The oracle on the first ds fixed planes of the path (one fwd+bwd)."""
    import oracle
    F = pair.F[:ds].float().cpu().numpy()
    u = pair.u[:ds].cpu().numpy()
    xmax = _crop_transform(pair, ds)
    T = oracle.Transform(pair.A.astype(np.float64), pair.t.astype(np.float64), pair.S.astype(np.float64),
                         pair.xmin.astype(np.float64), xmax.astype(np.float32).astype(np.float64))
    t0 = time.perf_counter()
    if args.path == "mse":
        oracle.objective_mse(F, pair.M.float().cpu().numpy(), u, T, 1.0)
    elif args.path == "adam":
        g = np.random.default_rng(0).normal(size=u.shape) * 1e-6
        oracle.sobolev_adam_step(u, g, np.zeros(u.shape), np.zeros(u.shape), 0.1, 1e-3, 0.9, 0.999, 1e-8, 1)
    else:
        V = np.ascontiguousarray(pair.u.cpu().numpy()[::-1])
        g = np.random.default_rng(0).normal(size=u.shape)
        oracle.sample_channels(V, F.shape, u, T, True)
        oracle.sample_channels_bwd(V, F.shape, u, T, g, True)
    return F.size, time.perf_counter() - t0, oracle.max_threads()


def run_gpu_path(args, ws, rank, local):
    from voxel_grid_sampler_gb300 import build, ffdp, synth
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    shape = None if not args.shape else (args.shape,) * 3
    pair = synth.make_pair(4, device=dev, shape=shape, seed=1004 + 100 * rank)
    N = pair.F.numel()
    call, ins, o, outs = _path_setup(args, pair, dev)
    stream = torch.cuda.current_stream(dev)
    args_in = [ins[k] for k in ins]

    def step():
        call(*args_in, o, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    ms, launches, clk = _time_steps(step, args.steps, stream, dev, ws, clocks)
    kern = _kernel_times(step, max(3, min(args.steps, 10)), dev)
    value = _aggregate_gvox(N, ws, ms)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    # end to end: pinned host inputs copied in and every output copied out, each step
    e2e = None
    if not args.no_e2e:
        hin = [ins[k].cpu().pin_memory() for k in ins]
        din = [torch.empty_like(ins[k]) for k in ins]
        hout = [torch.empty(o[k].shape, dtype=o[k].dtype).pin_memory() for k in outs]
        n_e2e = max(4, min(args.steps, 10))

        def e2e_step():
            for d, h in zip(din, hin):
                d.copy_(h, non_blocking=True)
            call(*din, o, stream)
            for h, k in zip(hout, outs):
                h.copy_(o[k], non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        _barrier(ws)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms_e2e = _max_over_ranks(e0.elapsed_time(e1) / n_e2e, ws, dev)
        e2e = {"value": N * ws / (ms_e2e * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int(sum(h.numel() * h.element_size() for h in hin)),
               "d2h_bytes_per_step": int(sum(h.numel() * h.element_size() for h in hout))}
        del hin, din, hout
    if rank != 0:
        return
    peak, peak_kind = _peaks()
    kb = PATH_KERNEL_BYTES[args.path]
    step_gbs = PATH_ALGO_BYTES[args.path] * N / (ms * 1e-3) / 1e9
    roof = _roofline(kern, kb, N, peak, peak_kind, lambda k: _traffic_per_launch(k, "%s 512^3" % args.path, N))
    roof["kernels"] = {k: {"ms": v[1] / max(v[0], 1), "bytes_per_voxel": kb.get(k, 0),
                           "frac": kb.get(k, 0) * N / (v[1] / max(v[0], 1) * 1e-3) / 1e9 / peak}
                       for k, v in kern.items()}
    out = {
        "metric": PATH_METRIC[args.path], "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "%s on the %s pair" % (args.path, pair.workload.name), "shape": list(pair.F.shape),
                   "voxels": N, "l2": "inputs larger than L2 (%.2f GB algorithmic bytes per step)"
                                     % (PATH_ALGO_BYTES[args.path] * N / 1e9),
                   "parallelism": "independent pair per rank" if ws > 1 else "single GPU"},
        "pct_hbm_roofline": {"step_algorithmic_gbs": step_gbs, "of_8tbs": step_gbs / HBM_NOMINAL_GBS,
                             "of_measured": step_gbs / peak, "bytes_per_voxel": PATH_ALGO_BYTES[args.path]},
        "roofline": roof,
        "kernels_ms_per_launch": {k: v[1] / max(v[0], 1) for k, v in kern.items()},
        "gpu_launches": int(launches), "clocks": clk, "e2e": e2e,
    }
    if ws == 1 and not args.no_cpu_baseline:
        n1, t1, _ = _path_oracle_sample(args, pair, 2)
        ds = int(max(2, min(pair.F.shape[0], args.cpu_budget_s / max(t1 / 2.0, 1e-3))))
        n, t, cores = _path_oracle_sample(args, pair, ds)
        out["cpu_baseline"] = {"value": n / t / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": "oracle %s on fixed planes z<%d of the %s pair (%d voxels, %.1f s)"
                                         % ({"mse": "MSE objective fwd+bwd", "compose": "composition fwd+bwd",
                                             "adam": "regularised Adam step"}[args.path], ds,
                                            "x".join(map(str, pair.F.shape)), n, t)}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=4, choices=[4, 5])
    ap.add_argument("--impl", default="ffdp", choices=["ffdp", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=6.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-workload5", action="store_true",
                    help="skip the 1024^3 leg that the default workload-4 line carries")
    ap.add_argument("--shape", type=int, default=0, help="cube edge overriding the workload size (profiling)")
    ap.add_argument("--window", type=int, default=0,
                    help="LNCC window overriding the workload's (odd >= 3; above 7 the separable passes run)")
    ap.add_argument("--store-slope", type=int, default=1, choices=[0, 1],
                    help="MI-only objectives: store J and dJ/dp (1) or stay implicit (0)")
    ap.add_argument("--path", default="objective", choices=["objective", "mse", "compose", "adam"],
                    help="objective (default, --workload 4|5), or the MSE objective / warp composition "
                         "on the 512^3 pair")
    args = ap.parse_args()
    ws, rank, local = _dist()
    if ws > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank, local)
        elif args.path != "objective":
            run_gpu_path(args, ws, rank, local)
        else:
            run_gpu(args, ws, rank, local)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
