"""Benchmark of the canvas attention block on GB300.

One bench step = one canvas of the 48-step denoising loop (T=512 canvas rows, ctx=8192 cached
rows, nh=8, nkv=4, hd=256): the cache is prepared once, then 48 forwards run, each on a fresh
canvas Q/K/V (seed 3 + step) resident in HBM.  The metric is useful attention TFLOP/s
(4 * T * nh * (ctx + T) * hd per forward).

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle instead, on a bounded
sample of the same workload.  With torchrun (N > 1) each rank runs an independent replica on its
own GPU (the block has no cross-GPU exchange); value = work of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "canvas-attention TFLOP/s and us/denoise-step, % of TF32 tensor peak"
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25      # nominal dense tf32 / bf16 ratio of the part
# Workloads timed beside the bench workload, one forward each (a batch of canvases: all of them).
SIDE_WORKLOADS = ["tiny", "gqa_hd256_ctx1k", "gqa_hd128_ctx4k", "mha_canvas4k_x4"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attn_tc_kernel_denoise48_ctx8k.md")


def attn_traffic():
    """DRAM bytes per launch of the tensor-core attention kernel on the bench workload, from the
    ncu capture summarised in the profile summary's `traffic_per_launch_bytes:` line, or None
    when the kernel's sources have changed since that capture (its `kernel_source:` id)."""
    import re
    from gqa_canvas_attention_gb300.build import attn_kernel_source_id
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    text = open(PROFILE_SUMMARY).read()
    m = re.search(r"traffic_per_launch_bytes:\s*([0-9.eE+]+)\s+kernel_source:\s*(sha1:[0-9a-f]+)",
                  text)
    if not m or m.group(2) != attn_kernel_source_id():
        return None
    return float(m.group(1))


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="denoise48_ctx8k")
    ap.add_argument("--path", default="tc", choices=["tc", "fp32"])
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=80)
    ap.add_argument("--hidden", type=int, default=0,
                    help="run each forward from a residual stream of this width through the "
                         "projection step (input norm + q/k/v projections) instead of from q/k/v")
    ap.add_argument("--layer", action="store_true",
                    help="with --hidden: the whole attention branch of a layer (projections, "
                         "block, o_proj, post-attention norm, residual add) on the residual stream")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the 48 forwards one by one instead of replaying a CUDA graph")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--no-side", action="store_true",
                    help="skip the per-forward timings of the other workloads")
    ap.add_argument("--side-reps", type=int, default=20)
    ap.add_argument("--cpu-side-budget-s", type=float, default=3.0)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


_ORACLE_INPUTS = {}


def _oracle_inputs(w, unit):
    """Seeded inputs of one forward (denoising step, or canvas of a batch) of workload w as numpy
    arrays, with the cache it attends to (generated once per process)."""
    from gqa_canvas_attention_gb300.workloads import shared_cache, workload_inputs
    key = (w.name, unit)
    if key not in _ORACLE_INPUTS:
        d = workload_inputs(w, canvas=unit) if w.canvases > 1 else workload_inputs(w, step=unit)
        d = {k: (None if v is None else v.numpy()) for k, v in d.items()}
        if w.ctx > 0 and w.canvases == 1:
            if (w.name, "cache") not in _ORACLE_INPUTS:
                kc, vc = shared_cache(w)
                _ORACLE_INPUTS[(w.name, "cache")] = (kc.numpy(), vc.numpy())
            d["k_cache"], d["v_cache"] = _ORACLE_INPUTS[(w.name, "cache")]
        _ORACLE_INPUTS[key] = d
    return _ORACLE_INPUTS[key]


def oracle_rows(w, unit, rows):
    """The oracle's output rows [r0, r1) of one forward of w (fp64 [r1 - r0, nh*hd])."""
    import oracle
    from gqa_canvas_attention_gb300.workloads import EPS
    d = _oracle_inputs(w, unit)
    out = oracle.forward(d["q"], d["k_canvas"], d["v_canvas"], d["k_cache"], d["v_cache"], w.nh,
                         w.nkv, w.hd, d["q_norm_w"], d["k_norm_w"], eps=EPS, theta=w.theta,
                         pos0=w.pos0, rows=rows)
    return out[rows[0]:rows[1]]


def oracle_sample(w, budget_s: float, threads: int = 0):
    """Time the fp64 oracle on whole forwards' canvas rows, forward after forward, until about
    budget_s of CPU work (on `threads` OpenMP threads, 0 = all host cores).

    Returns (useful flops computed, seconds, threads used, description)."""
    import oracle
    from gqa_canvas_attention_gb300.workloads import EPS

    prev = oracle.set_threads(0)
    used = oracle.set_threads(threads) if threads else prev
    try:
        d = _oracle_inputs(w, 0)
        per_row = 4 * w.nh * w.S * w.hd
        cal = min(16, w.T)
        t0 = time.perf_counter()
        oracle.forward(d["q"], d["k_canvas"], d["v_canvas"], d["k_cache"], d["v_cache"], w.nh,
                       w.nkv, w.hd, d["q_norm_w"], d["k_norm_w"], eps=EPS, theta=w.theta,
                       pos0=w.pos0, rows=(0, cal))
        t_row = (time.perf_counter() - t0) / cal
        rows_total = max(1, int(budget_s / max(t_row, 1e-9)))
        flops, secs, unit, done = 0, 0.0, 0, 0
        while done < rows_total and unit < w.forwards():
            d = _oracle_inputs(w, unit)
            r = min(w.T, rows_total - done)
            t0 = time.perf_counter()
            oracle.forward(d["q"], d["k_canvas"], d["v_canvas"], d["k_cache"], d["v_cache"], w.nh,
                           w.nkv, w.hd, d["q_norm_w"], d["k_norm_w"], eps=EPS, theta=w.theta,
                           pos0=w.pos0, rows=(0, r))
            secs += time.perf_counter() - t0
            flops += per_row * r
            done += r
            unit += 1
    finally:
        oracle.set_threads(prev)
    what = "canvas" if w.canvases > 1 else "denoising step"
    desc = (f"{done} canvas rows x {w.nh} heads over {unit} {what}(s) of {w.name} "
            f"(ctx={w.ctx}, T={w.T}, hd={w.hd}), fp64, OpenMP over (row, head) on {used} "
            f"thread(s)")
    return flops, secs, used, desc


CHECK_TOL = {"tc": (5e-3, 5e-4), "fp32": (1e-5, 1e-6)}


def workload_config(w):
    """The `config` object of a line: the workload and its sizes (the same in both arms)."""
    return {"workload": w.name, "T": w.T, "ctx": w.ctx, "nh": w.nh, "nkv": w.nkv, "hd": w.hd,
            "denoise_steps": w.steps, "canvases": w.canvases,
            "l2": "inputs larger than L2 between reuses (a fresh canvas per forward, the cache "
                  "reused by a canvas's forwards)" if w.forwards() > 1 else
                  "L2 flushed (a 256 MiB write) before every timed forward"}


def check_rows(w, unit, got, path):
    """Compare 64 rows (four runs of 16 across the canvas) of one forward's output -- a CPU
    tensor [T, nh*hd] -- with the oracle's; raise if the parity tolerance is exceeded."""
    import numpy as np
    T = w.T
    starts = sorted({0, T // 3, (2 * T) // 3, max(0, T - 16)})
    spans = [(a, min(T, a + 16)) for a in starts]
    errs = []
    for a, b in spans:
        ref = oracle_rows(w, unit, (a, b))
        errs.append(np.abs(got[a:b].double().numpy() - ref).ravel())
    e = np.concatenate(errs)
    tmax, tmean = CHECK_TOL[path]
    res = {"forward": unit, "rows": [list(x) for x in spans], "max_err": float(np.max(e)),
           "mean_err": float(np.mean(e)), "tol_max": tmax, "tol_mean": tmean}
    if not (np.isfinite(e).all() and res["max_err"] <= tmax and res["mean_err"] <= tmean):
        raise RuntimeError(f"output check against the oracle failed: {res}")
    return res


def side_workloads(B, dev, args, peak, peaks):
    """One forward of each other workload, with its own cache passed in (converted by the call),
    L2 flushed before every timed forward: the median time of `side_reps` forwards, the attention
    kernel's own time (events around its launches, a second pass), sampled rows checked with the
    oracle, and the oracle's own rate (one core for single-forward workloads, all cores for a
    batch of canvases)."""
    import statistics
    import torch
    from gqa_canvas_attention_gb300.workloads import EPS, WORKLOADS, workload_inputs
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)      # 256 MiB > L2
    res = {}
    for name in SIDE_WORKLOADS:
        w = WORKLOADS[name]
        plan = B.Plan(w.nh, w.nkv, w.hd, w.ctx, w.T, EPS, w.theta)
        if w.pos0 is not None:
            plan.set(B.DG_OPT_POS0, w.pos0)
        plan.set(B.DG_OPT_PATH, B.DG_PATH_TC if args.path == "tc" else B.DG_PATH_FP32)
        ins = []
        for c in range(w.canvases):
            d = workload_inputs(w, canvas=c) if w.canvases > 1 else workload_inputs(w)
            ins.append({k: (v.to(dev) if v is not None else None) for k, v in d.items()})
        out = torch.empty((w.T, w.nh * w.hd), dtype=torch.float32, device=dev)

        def fwd():
            for d in ins:
                plan.forward(d["q"], d["k_canvas"], d["v_canvas"], d["k_cache"], d["v_cache"],
                             d["q_norm_w"], d["k_norm_w"], None, out)

        for _ in range(3):
            fwd()
        torch.cuda.synchronize()
        if plan.sync_status() != B.DG_OK:
            raise RuntimeError(f"{name}: device status after warm-up")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(args.side_reps):
            flush.zero_()
            e0.record()
            fwd()
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        fwd_us = statistics.median(times) * 1e3 / w.canvases
        plan.set(B.DG_OPT_PROFILE, 1)
        for _ in range(args.side_reps):
            flush.zero_()
            fwd()
        torch.cuda.synchronize()
        st = {k: B.dg_attn_profile_read(plan.handle, v) for k, v in
              (("attention", B.DG_STAGE_ATTENTION), ("norm_rope", B.DG_STAGE_NORM_ROPE),
               ("combine", B.DG_STAGE_COMBINE), ("cache", B.DG_STAGE_CACHE))}
        plan.set(B.DG_OPT_PROFILE, 0)
        if plan.sync_status() != B.DG_OK:
            raise RuntimeError(f"{name}: device status after the timed forwards")
        chk = check_rows(w, w.canvases - 1 if w.canvases > 1 else 0, out.cpu(), args.path)
        plan.close()
        flops = w.flops_per_forward()
        kern_us = st["attention"][0] / max(1, st["attention"][1]) * 1e3
        r = {"us_per_forward": fwd_us, "tflops": flops / (fwd_us * 1e-6) / 1e12,
             "attention_kernel_us": kern_us,
             "attention_kernel_tflops": flops / (kern_us * 1e-6) / 1e12,
             "frac": flops / (kern_us * 1e-6) / 1e12 / peak,
             "stage_us_per_forward": {k: v[0] * 1e3 / max(1, args.side_reps * w.canvases)
                                      for k, v in st.items()},
             "check": chk, "useful_flop_per_forward": flops}
        if not args.no_cpu_baseline:
            f, sec, thr, desc = oracle_sample(w, args.cpu_side_budget_s,
                                              threads=0 if w.canvases > 1 else 1)
            r["oracle"] = {"tflops": f / sec / 1e12, "cores": thr, "sample": desc}
        res[name] = r
    return res


def run_reference(args, w):
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.barrier()
            return
    per_step_budget = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, per_step_budget / 4)
    flops, secs = 0, 0.0
    desc = ""
    threads = 1
    for _ in range(args.steps):
        f, s, threads, desc = oracle_sample(w, per_step_budget)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc + " per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def main():
    args = parse()
    from gqa_canvas_attention_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    from gqa_canvas_attention_gb300 import binding as B
    from gqa_canvas_attention_gb300 import replicas
    from gqa_canvas_attention_gb300.workloads import EPS, shared_cache, workload_inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    # ---------------------------------------------------------------- inputs (resident)
    n_fwd = w.forwards()
    kc, vc = (None, None)
    if w.ctx > 0:
        kc, vc = shared_cache(w)
        kc, vc = kc.to(dev), vc.to(dev)
    canv = []
    for i in range(n_fwd):
        d = workload_inputs(w, step=i) if w.canvases == 1 else workload_inputs(w, canvas=i)
        canv.append({k: d[k].to(dev) if d[k] is not None else None
                     for k in ("q", "k_canvas", "v_canvas", "q_norm_w", "k_norm_w")})
    out = torch.empty((w.T, w.nh * w.hd), dtype=torch.float32, device=dev)

    plan = B.Plan(w.nh, w.nkv, w.hd, w.ctx, w.T, EPS, w.theta)
    if w.pos0 is not None:
        plan.set(B.DG_OPT_POS0, w.pos0)
    plan.set(B.DG_OPT_PATH, B.DG_PATH_TC if args.path == "tc" else B.DG_PATH_FP32)
    # the canvases are resident (or copied in ahead, ordered by events, in the end-to-end run)
    plan.set(B.DG_OPT_INPUTS_RESIDENT, 1)
    if args.splits:
        plan.set(B.DG_OPT_SPLITS, args.splits)
    splits = plan.get(B.DG_INFO_SPLITS_USED)

    hid = None
    if args.hidden:
        # residual-stream inputs [T, H] per forward and one set of projection weights
        # (1/sqrt(H)-scaled normals, so the projections are O(1) like the q/k/v draws)
        H = args.hidden
        g = torch.Generator().manual_seed(1000 + w.seed)
        r = lambda *sh: torch.randn(*sh, generator=g, dtype=torch.float32)
        ln = (1.0 + 0.1 * r(H)).to(dev)
        wq, wk, wv = (r(w.nh * w.hd, H) / H ** 0.5).to(dev), (r(w.nkv * w.hd, H) / H ** 0.5).to(dev), \
            (r(w.nkv * w.hd, H) / H ** 0.5).to(dev)
        plan.proj_prepare(H, ln, wq, wk, wv)
        hid = [r(w.T, H).to(dev) for _ in canv]
        del wq, wk, wv
        if args.layer:
            K = w.nh * w.hd
            plan.oproj_prepare(H, (r(H, K) / K ** 0.5).to(dev), (1.0 + 0.1 * r(H)).to(dev))

    def one_step():
        """One canvas: cache conversion once, then every denoising step's forward."""
        if w.ctx > 0:
            plan.cache_prepare(kc, vc)
        for i, c in enumerate(canv):
            if hid is not None and args.layer:
                plan.forward_layer(hid[i], None, None, c["q_norm_w"], c["k_norm_w"], None)
            elif hid is not None:
                plan.forward_hidden(hid[i], None, None, c["q_norm_w"], c["k_norm_w"], None, out)
            else:
                plan.forward(c["q"], c["k_canvas"], c["v_canvas"], None, None, c["q_norm_w"],
                             c["k_norm_w"], None, out)

    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize()
    if plan.sync_status() != B.DG_OK:
        raise RuntimeError("device wait timed out during warm-up")

    # The library's calls only enqueue work (no allocation, no host synchronisation), so the
    # whole canvas -- cache conversion and 48 forwards -- is captured once into a CUDA graph and
    # replayed; the kernels are the same.
    def make_runner():
        if args.no_graph:
            return one_step, None
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_step()
        for _ in range(max(3, args.warmup)):
            graph.replay()
        torch.cuda.synchronize()
        if plan.sync_status() != B.DG_OK:
            raise RuntimeError("device wait timed out during graph warm-up")
        return graph.replay, graph

    run_step, graph = make_runner()

    # ---------------------------------------------------------------- timed region
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            run_step()
        ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = ev0.elapsed_time(ev1)
    if plan.sync_status() != B.DG_OK:
        raise RuntimeError("device wait timed out in the timed region")
    # the last forward of the last replay left its output in `out`: compare sampled rows of it
    # with the oracle (outside the timed region); a mismatch fails the run
    checked = {"timed": None, "e2e": None}
    if not args.hidden and rank == 0:
        checked["timed"] = check_rows(w, n_fwd - 1, out.cpu(), args.path)

    # ---------------------------------------------------------------- per-kernel times
    # Each kernel of a forward may start while the one before it finishes (programmatic
    # dependent launch); an event recorded between two launches breaks that overlap.  So the
    # per-launch times come from a second pass over the same canvas with events around every
    # launch (DG_OPT_PROFILE), right after the timed region, and not from the timed region itself.
    del graph
    plan.set(B.DG_OPT_PROFILE, 1)
    run_step, graph = make_runner()
    # (switching profiling on empties the event record; a captured graph re-records the same
    # events on every replay, so the read below holds the last replay's launches)
    prof_steps = max(1, min(args.steps, 5))
    for _ in range(prof_steps):
        run_step()
    torch.cuda.synchronize()
    attn_ms, attn_n = B.dg_attn_profile_read(plan.handle, B.DG_STAGE_ATTENTION)
    norm_ms, norm_n = B.dg_attn_profile_read(plan.handle, B.DG_STAGE_NORM_ROPE)
    comb_ms, comb_n = B.dg_attn_profile_read(plan.handle, B.DG_STAGE_COMBINE)
    cache_ms, cache_n = B.dg_attn_profile_read(plan.handle, B.DG_STAGE_CACHE)
    proj_ms, proj_n = B.dg_attn_profile_read(plan.handle, B.DG_STAGE_PROJECTION)
    oproj_ms, oproj_n = B.dg_attn_profile_read(plan.handle, B.DG_STAGE_OPROJ)
    plan.set(B.DG_OPT_PROFILE, 0)
    del graph
    rec_steps = max(1, attn_n // n_fwd)      # steps whose launches the record holds
    flops_fwd = w.flops_per_forward()
    flops_step = flops_fwd * n_fwd
    ms, total_flops = replicas.aggregate(ms, flops_step * args.steps, dev if world > 1 else None)
    value = replicas.throughput(ms, total_flops) / 1e12
    ms_per_step = ms / args.steps

    # ---------------------------------------------------------------- roofline of the kernels
    peaks, src = measured_peaks()
    tc = args.path == "tc"
    # The tensor-core kernel runs kind::f16 MMAs (bf16 products for Q.K^T, fp16 for P.V): its
    # peak is the measured bf16 burst rate (the kernel is timed launch by launch).  It executes
    # two MMA units per useful one (three bf16 products for Q.K^T, one for P.V, against one each).
    # The exact path runs fp32 FMAs on the CUDA cores: 152 SMs x 128 lanes x 2 FLOP x the clock.
    if tc:
        attn_peak, attn_bound, exec_per_useful = peaks["bf16_tflops"], "tensor", 2.0
        peak_src = f"{src}: bf16_tflops (burst cuBLAS bf16 GEMM; the kernel runs kind::f16 MMAs)"
    else:
        attn_peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        attn_bound, exec_per_useful = "alu", 1.0
        peak_src = "152 SMs x 128 fp32 lanes x 2 FLOP x sm_max_mhz"
    ev_us = attn_ms / max(1, attn_n) * 1e3
    live_us = None if args.hidden else ms_per_step * 1e3 / n_fwd
    if live_us is not None and live_us < ev_us:
        kern_us, kern_src = live_us, ("live: the whole forward's time in the timed region, "
                                      "which bounds the kernel's (events around each launch gave "
                                      f"{ev_us:.2f} us)")
    else:
        kern_us, kern_src = ev_us, ("CUDA events around each launch, "
                                    f"{max(1, min(args.steps, 5))} replays of the step right after "
                                    "the timed region")
    attn_tflops = flops_fwd / (kern_us * 1e-6) / 1e12
    # first stage: fp32 q, k, v read; q-hat and k-hat written as bf16 hi/lo (4 bytes per element)
    # and v-hat as fp16 (2 bytes) for the tensor-core kernel, fp32 for the exact path
    if tc:
        norm_bytes = w.T * w.hd * (4 * (w.nh + 2 * w.nkv) + 4 * (w.nh + w.nkv) + 2 * w.nkv)
    else:
        norm_bytes = w.T * w.hd * 8 * (w.nh + 2 * w.nkv)
    norm_avg_s = norm_ms / max(1, norm_n) / 1e3
    norm_gbs = norm_bytes / norm_avg_s / 1e9 if norm_n else 0.0   # no first-stage launch on the
                                                                    # projection path (fused)
    # What one launch of that size can reach at all: a device-to-device copy moving the same
    # bytes (half read, half written), timed the same way (events around each launch, L2 flushed
    # by a larger write before each).
    copy_ref = None
    if norm_n:
        half = norm_bytes // 8                                   # floats read = floats written
        src_buf = torch.empty(half, dtype=torch.float32, device=dev)
        dst_buf = torch.empty_like(src_buf)
        flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
        ca, cb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(20):
            flush.zero_()
            ca.record()
            dst_buf.copy_(src_buf)
            cb.record()
            cb.synchronize()
            times.append(ca.elapsed_time(cb))
        times.sort()
        cu = times[len(times) // 2] * 1e3
        copy_ref = {"bytes": 2 * half * 4, "us": cu, "gbs": 2 * half * 4 / (cu * 1e-6) / 1e9,
                    "frac": 2 * half * 4 / (cu * 1e-6) / 1e9 / peaks["hbm_gbs"]}
        del src_buf, dst_buf, flush

    # ---------------------------------------------------------------- end to end from host memory
    # Every step's inputs go host -> device and every forward's output device -> host through
    # pinned buffers, inside the timed region.  The transfers are pipelined a step at a time: a
    # step's canvases and cache (one copy per array) upload on one copy stream while the step
    # before it computes, and its 48 outputs download on another while the step after it
    # computes, through two device slots of each.  The compute stream then meets events only at
    # step boundaries: an event recorded or awaited between two forwards would switch off the
    # overlap of one forward's attention kernel with the next forward's first stage
    # (programmatic dependent launch), ~15 us per forward.  The first step's upload and the last
    # step's download have nothing to overlap with; both are inside the timed region.
    e2e = None
    if args.e2e_steps > 0 and not args.hidden:
        keys = [k for k in ("q", "k_canvas", "v_canvas", "q_norm_w", "k_norm_w")
                if canv[0][k] is not None]
        h_in = {k: torch.stack([c[k].cpu() for c in canv]).pin_memory() for k in keys}
        h_kc = kc.cpu().pin_memory() if kc is not None else None
        h_vc = vc.cpu().pin_memory() if vc is not None else None
        h_out = torch.empty((n_fwd, w.T, w.nh * w.hd), dtype=torch.float32).pin_memory()
        d_in = [{k: torch.empty_like(h_in[k], device=dev) for k in keys} for _ in range(2)]
        d_out = [torch.empty_like(h_out, device=dev) for _ in range(2)]
        d_kc = [torch.empty_like(kc) if kc is not None else None for _ in range(2)]
        d_vc = [torch.empty_like(vc) if vc is not None else None for _ in range(2)]
        h2d = sum(t.numel() * 4 for t in h_in.values())
        h2d += 0 if kc is None else (kc.numel() + vc.numel()) * 4
        d2h = h_out.numel() * 4
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        ev_in_ready, ev_done, ev_out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = {"done": [False, False], "out": [False, False]}
        e2e_graphs = []

        def upload(slot):
            # a step's inputs into `slot`, once the step that last read it has finished
            with torch.cuda.stream(s_in):
                if used["done"][slot]:
                    s_in.wait_event(ev_done[slot])
                for k in keys:
                    d_in[slot][k].copy_(h_in[k], non_blocking=True)
                if kc is not None:
                    d_kc[slot].copy_(h_kc, non_blocking=True)
                    d_vc[slot].copy_(h_vc, non_blocking=True)
                ev_in_ready[slot].record(s_in)

        def compute(slot):
            # one step on the inputs of `slot`: the cache conversion, then the 48 forwards
            if kc is not None:
                plan.cache_prepare(d_kc[slot], d_vc[slot])
            x = d_in[slot]
            for i in range(n_fwd):
                plan.forward(x["q"][i], x["k_canvas"][i], x["v_canvas"][i], None, None,
                             x["q_norm_w"][i] if "q_norm_w" in x else None,
                             x["k_norm_w"][i] if "k_norm_w" in x else None, None,
                             d_out[slot][i])

        # each slot's step is captured once into a CUDA graph and replayed, as in the timed
        # region above (the events stay outside the graphs, at step boundaries): enqueuing the
        # forwards one by one cost the host ~45 us each, nearly what they take on the device
        run_compute = []
        for slot in range(2):
            if args.no_graph:
                run_compute.append(lambda slot=slot: compute(slot))
            else:
                g_ = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_):
                    compute(slot)
                run_compute.append(g_.replay)
                e2e_graphs.append(g_)

        def e2e_run(n_steps):
            upload(0)
            for st in range(n_steps):
                slot = st % 2
                if st + 1 < n_steps:
                    upload(slot ^ 1)                # the next step's inputs, during this step
                stream.wait_event(ev_in_ready[slot])
                if used["out"][slot]:
                    stream.wait_event(ev_out_free[slot])
                run_compute[slot]()
                ev_done[slot].record(stream)
                used["done"][slot] = True
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[slot])
                    h_out.copy_(d_out[slot], non_blocking=True)
                    ev_out_free[slot].record(s_out)
                used["out"][slot] = True
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)

        e2e_run(2)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h0 = time.perf_counter()
        e2e_run(args.e2e_steps)
        host_ms = (time.perf_counter() - h0) * 1e3 / args.e2e_steps
        e1.record(stream)
        torch.cuda.synchronize()
        if plan.sync_status() != B.DG_OK:
            raise RuntimeError("device wait timed out in the end-to-end run")
        # the outputs copied back to the host by the last end-to-end step: first and last forward
        if rank == 0:
            checked["e2e"] = [check_rows(w, 0, h_out[0], args.path),
                              check_rows(w, n_fwd - 1, h_out[n_fwd - 1], args.path)]
        del run_compute, e2e_graphs
        ems, e2e_flops = replicas.aggregate(e0.elapsed_time(e1), flops_step * args.e2e_steps,
                                            dev if world > 1 else None)
        e2e = {"value": replicas.throughput(ems, e2e_flops) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ems / args.e2e_steps, "host_enqueue_ms_per_step": host_ms,
               "steps": args.e2e_steps,
               "cuda_graph": not args.no_graph,
               "overlap": "a step's canvases and cache upload while the step before it "
                          "computes and its outputs download while the step after it computes "
                          "(two device slots of each, events at step boundaries only); the "
                          "first upload and the last download are timed unoverlapped"}

    launches_per_step = (1 if w.ctx > 0 else 0) + n_fwd * (plan.get(B.DG_INFO_LAUNCHES)
                                                           + (1 if args.hidden else 0)
                                                           + (3 if args.layer else 0))
    plan.close()

    # ---------------------------------------------------------------- the other workloads
    side = None
    if not args.no_side and not args.hidden and world == 1:
        side = side_workloads(B, dev, args, attn_peak, peaks)

    # the capture is of the default run's kernel (the auto schedule, the instantiation without
    # the o_proj operand split)
    traffic = (attn_traffic() if tc and w.name == "denoise48_ctx8k" and not args.hidden
               and not args.splits else None)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16x3+f16" if args.path == "tc" else "f32", "data": "synthetic",
        "config": workload_config(w),
        "run": {"path": args.path, "splits": splits, "cuda_graph": not args.no_graph,
                "inputs_resident": True},
        "us_per_denoise_step": ms_per_step * 1e3 / n_fwd,
        "canvas_steps_per_s": n_fwd * args.steps * world / (ms / 1e3),
        "roofline": {"bound": attn_bound, "achieved": attn_tflops, "peak": attn_peak,
                     "unit": "TFLOP/s", "frac": attn_tflops / attn_peak,
                     "traffic": traffic,
                     # DRAM rate: the captured bytes per launch over the kernel time above
                     "dram_gbs": traffic / (kern_us * 1e-6) / 1e9 if traffic else None,
                     "kernel": "attn_tc_kernel" if tc else "attn_fp32_kernel",
                     "peak_source": peak_src,
                     "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"] if tc else None,
                     "kernel_us": kern_us, "kernel_us_source": kern_src,
                     "event_us_per_launch": ev_us, "launches": attn_n,
                     "useful_flop_per_launch": flops_fwd,
                     "executed_mma": None if not tc else {
                         "tflops": attn_tflops * exec_per_useful,
                         "frac": attn_tflops * exec_per_useful / attn_peak,
                         "note": "MMA work the tensor pipe executes: Q.K^T as three bf16 products "
                                 "(hi.hi + hi.lo + lo.hi) and P.V as one fp16 product, two units "
                                 "per useful one; the scheme's ceiling is 0.5 of the peak in "
                                 "useful FLOPs"},
                     "tf32_nominal": None if not tc else {
                         "peak": attn_peak * NOMINAL_TF32_OVER_BF16,
                         "frac": attn_tflops / (attn_peak * NOMINAL_TF32_OVER_BF16),
                         "note": "useful FLOPs against a TF32 rate of the measured bf16 burst "
                                 "x the nominal tf32/bf16 ratio (1.1/2.25): the basis the target "
                                 "is stated on; these MMAs do not run at that rate"}},
        "norm_rope": {"bound": "hbm", "achieved": norm_gbs, "peak": peaks["hbm_gbs"],
                      "unit": "GB/s", "frac": norm_gbs / peaks["hbm_gbs"],
                      "avg_launch_us": norm_avg_s * 1e6, "bytes_per_launch": norm_bytes,
                      "bytes": "fp32 q, k, v read; bf16 hi/lo q-hat, k-hat and fp16 v-hat "
                               "written" if tc else "fp32 q, k, v read and written",
                      "same_size_copy": copy_ref},
        "stage_ms_per_step": {k: v / rec_steps for k, v in (("norm_rope", norm_ms),
                              ("attention", attn_ms), ("combine", comb_ms), ("cache", cache_ms))},
        "gpu_launches": launches_per_step * args.steps,
        # every check that ran passed (a failed one raises): the timed output always, the
        # end-to-end outputs when that run was made
        "checked": (checked["timed"] is not None and (checked["e2e"] is not None or e2e is None)
                    if not args.hidden else False),
        "check": checked,
        "configs": side,
        "projection": None if not args.hidden else {
            "H": args.hidden, "bound": "tensor",
            "useful_gflop_per_launch": 2 * w.T * args.hidden * (w.nh + 2 * w.nkv) * w.hd / 1e9,
            "avg_launch_us": proj_ms / max(1, proj_n) * 1e3,
            "achieved": 2 * w.T * args.hidden * (w.nh + 2 * w.nkv) * w.hd
                        / (proj_ms / max(1, proj_n) / 1e3) / 1e12,
            "unit": "TFLOP/s", "peak": attn_peak,
            "frac": 2 * w.T * args.hidden * (w.nh + 2 * w.nkv) * w.hd
                    / (proj_ms / max(1, proj_n) / 1e3) / 1e12 / attn_peak,
            "note": "input norm + q/k/v projections with the first stage fused (two launches), "
                    "useful fp32-GEMM FLOPs against the bf16 burst peak (the GEMM runs three "
                    "bf16 products); the step's value then includes this work"},
        "oproj": None if not args.layer else {
            "H": args.hidden, "bound": "tensor",
            "useful_gflop_per_launch": 2 * w.T * args.hidden * w.nh * w.hd / 1e9,
            "avg_launch_us": oproj_ms / max(1, oproj_n) * 1e3,
            "achieved": 2 * w.T * args.hidden * w.nh * w.hd / (oproj_ms / max(1, oproj_n) / 1e3) / 1e12,
            "unit": "TFLOP/s", "peak": attn_peak,
            "frac": 2 * w.T * args.hidden * w.nh * w.hd / (oproj_ms / max(1, oproj_n) / 1e3) / 1e12
                    / attn_peak,
            "note": "o_proj GEMM + post-attention norm and residual add (two launches; the "
                    "attention kernel wrote the GEMM's bf16 operand split, else a third launch "
                    "makes it), useful fp32-GEMM FLOPs against the bf16 burst peak"},
        "layer_us_per_forward": ms_per_step * 1e3 / n_fwd if args.layer else None,
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        f, s, threads, desc = oracle_sample(w, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle", "sample": desc}
        f1, s1, _, desc1 = oracle_sample(w, args.cpu_budget_s / 4, threads=1)
        line["cpu_baseline"]["one_core"] = {"value": f1 / s1 / 1e12, "unit": "TFLOP/s",
                                            "sample": desc1}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
