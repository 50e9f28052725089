"""Benchmark of the owner-side Muon / AdamW step (one JSON line on stdout).

A step is one pass of the whole hot path over the workload: the Muon step
(momentum, Newton-Schulz on every matrix, weight decay + update, bf16 copy)
and the AdamW step of the AdamW-route tensors, with every input already
resident in HBM.  Default workload: the Llama-3-8B-shaped set (224 Muon
matrices, 6.98e9 elements, plus 1.05e9 AdamW elements).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

value = dense Newton-Schulz TFLOP per step (all ranks) / step time, so the
unit is TFLOP/s of the whole step; ms_per_step is the step time itself.
Under torchrun (N > 1) the default is the owner-partitioned step of one
model over the N ranks (strong scaling: every tensor stepped once, by its
owner, with the collectives of the pages' routes); ``--mode replicas`` runs
an independent copy per rank instead (weak scaling).  The slowest rank's
time counts.  ``--impl reference`` times the float64
CPU oracle on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024  # GB300 L2

# Sources of the CTA-pair NS kernel and of the tile lists it runs (plan.cu
# builds and balances them, step.cu picks one per launch): DRAM traffic
# measured by ncu is reported only while all of them are unchanged since the
# capture.
KERNEL_SOURCES = ("k_ns_tc2.cu", "ns_epilogue.cuh", "ptx.cuh", "internal.h", "plan.cu", "step.cu")


def kernel_source_sha():
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "matrix_optimizer_step_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


METRIC = "Muon step ms & NS TFLOP/s (% bf16 TC peak), Llama-3-8B-shaped matrix set"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_burst": d["bf16_tflops"],
                "bf16_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_burst": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


def _workload_desc(wl):
    return (f"{wl.name}: {len(wl.matrices)} Muon tensors, {wl.muon_numel / 1e9:.3f}e9 elements, "
            f"{len(wl.vectors)} AdamW tensors, {wl.adamw_numel / 1e9:.3f}e9 elements")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        try:
            sm = [float(r[1]) for r in rows]
            mx = max(float(r[2]) for r in rows)
        except ValueError:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- CPU legs
def _oracle_sample(wl):
    """Bounded sample of the workload for the float64 oracle: the named
    Muon matrices (with their own inputs) and a 4M-element AdamW slice."""
    from matrix_optimizer_step_gb300 import workloads as W

    # Llama-3-8B: layer 0's k (the p = 1024 class) and gate (14336 x 4096,
    # the class that carries 80 % of the flops); the other p = 4096 classes
    # (q, o 4096 x 4096; up; down 4096 x 14336) take gate's measured rate.
    # About 10 s of host work per sample on 16 Arm cores.
    picks = {"llama3_8b": ["layers.0.k", "layers.0.gate"],
             "llama3_8b_layer": ["layers.0.k"],
             "moe_experts": [], "many_small": [s.name for s in wl.matrices[:48]],
             "gpt2_small": [s.name for s in wl.matrices[:12]],
             "single_256x512": [s.name for s in wl.matrices]}[wl.name]
    mats = []
    for i, spec in enumerate(wl.matrices):
        if spec.name in picks:
            W0 = W.master_init(spec, i).double().numpy()
            G = W.muon_grad(wl, spec, i).float().double().numpy()
            mats.append((spec, W0, G))
    if wl.name == "moe_experts":  # two expert slices of the first w1
        spec = wl.matrices[0]
        W0 = W.master_init(spec, 0)[:2].double().numpy()
        G = W.muon_grad(wl, spec, 0)[:2].float().double().numpy()
        mats.append((spec, W0, G))
    adam = None
    if wl.vectors:
        spec = max(wl.vectors, key=lambda v: v.numel)
        n = min(4 << 20, spec.numel)
        idx = wl.vectors.index(spec)
        w = W.vector_init(spec, idx)[:n].double().numpy()
        g = W.vector_grad(spec, idx)[:n].float().double().numpy()
        adam = (n, w, g)
    return mats, adam


def _oracle_time(wl, sample):
    """Run the oracle on the sample once; return (seconds, sample NS flops,
    extrapolated full-step seconds)."""
    import numpy as np

    from matrix_optimizer_step_gb300 import workloads as W
    from oracle import adamw as oadamw
    from oracle import muon as omuon

    h = wl.hyper
    mats, adam = sample
    flops = 0
    rate = {}  # (p, q) -> seconds per dense NS flop, from the sampled matrices of that class
    t_muon = 0.0
    for spec, W0, G in mats:
        t0 = time.perf_counter()
        omuon.muon_step(W0, np.zeros_like(W0), G, h["lr"], h["momentum"], h["wd"], h["ns_steps"],
                        h["a"], h["b"], h["c"])
        dt = time.perf_counter() - t0
        t_muon += dt
        m, n = spec.mn
        f = W.ns_flops(m, n, h["ns_steps"]) * (W0.size // (m * n))
        flops += f
        key = (min(m, n), max(m, n))
        s0, f0 = rate.get(key, (0.0, 0))
        rate[key] = (s0 + dt, f0 + f)
    t_adam = 0.0
    if adam is not None:
        n, w, g = adam
        t1 = time.perf_counter()
        oadamw.adamw_step(w, np.zeros(n), np.zeros(n), g, h["adam_lr"], h["beta1"], h["beta2"],
                          h["adam_eps"], h["adam_wd"], 1)
        t_adam = time.perf_counter() - t1
    # Each matrix of the workload at its own class's measured rate where the
    # sample holds that class, else at the rate of the sampled class with
    # the same p (the Gram size), else at the sample's overall rate.
    overall = t_muon / max(flops, 1)
    est = 0.0
    for spec in wl.matrices:
        m, n = spec.mn
        key = (min(m, n), max(m, n))
        f = W.ns_flops(m, n, h["ns_steps"]) * spec.n_slices
        if key in rate:
            r = rate[key][0] / rate[key][1]
        else:
            same_p = [k for k in rate if k[0] == key[0]]
            r = (sum(rate[k][0] for k in same_p) / sum(rate[k][1] for k in same_p)) if same_p else overall
        est += f * r
    if adam is not None:
        est += t_adam * wl.adamw_numel / adam[0]
    return t_muon + t_adam, flops, est


def _sample_desc(wl, sample):
    mats, adam = sample
    names = ", ".join(f"{s.name}{'[0:2]' if wl.name == 'moe_experts' else ''}" for s, _, _ in mats[:6])
    more = f" (+{len(mats) - 6} more)" if len(mats) > 6 else ""
    ad = f"; AdamW on {adam[0]} elements" if adam else ""
    return (f"float64 oracle Muon step on {len(mats)} matrices ({names}{more}){ad}; full-step time "
            f"extrapolated per shape class by NS flops at the sampled class's rate (Muon) and by element "
            f"count (AdamW)")


def _clock_normalized(achieved, peak, clk):
    """NS throughput per GHz of the SM clock sampled during the timed region,
    beside the measured sustained peak per GHz of the clock sampled while
    that peak was measured: separates kernel gains from power-cap luck."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not achieved or not clk or not clk.get("sm_mhz") or not os.path.exists(p):
        return None
    ref_mhz = json.load(open(p)).get("clocks_under_load", {}).get("sm_mhz_median")
    if not ref_mhz:
        return None
    a = achieved / (clk["sm_mhz"] / 1e3)
    b = peak / (ref_mhz / 1e3)
    return {"achieved_tflops_per_ghz": a, "peak_tflops_per_ghz": b, "frac": a / b,
            "sm_mhz": clk["sm_mhz"], "peak_sm_mhz": ref_mhz}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def reduce_max_over_ranks(value, dist, device):
    """Slowest rank's value (every rank gets it); identity without a process group."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- main legs
def run_reference(args, wl, rank, world):
    if rank != 0:
        return
    sample = _oracle_sample(wl)
    # Warm-up steps (untimed) only warm the host BLAS threads and caches: the
    # smallest sampled matrix does that as well as the whole sample.
    warm = (sorted(sample[0], key=lambda t: t[1].size)[:1], sample[1])
    for _ in range(args.warmup):
        _oracle_time(wl, warm)
    ests, secs = [], []
    for _ in range(args.steps):
        s, flops, est = _oracle_time(wl, sample)
        ests.append(est)
        secs.append(s)
    from matrix_optimizer_step_gb300 import workloads as W

    total = W.workload_ns_flops(wl)
    ms = 1000.0 * statistics.median(ests)
    value = total / (ms / 1000.0) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_desc(wl), "ns_steps": wl.hyper["ns_steps"]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": _sample_desc(wl, sample),
                         "sample_seconds_per_step": statistics.median(secs)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, wl, rank, world, local_rank):
    import torch

    import matrix_optimizer_step_gb300 as mos
    from matrix_optimizer_step_gb300 import workloads as W

    dist = None
    if world > 1:
        import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    mos.load_library()
    for kv in args.tuning:
        k, v = kv.split("=")
        mos.dmuon_set_tuning(int(k), int(v))
    h = wl.hyper
    mat = W.materialize(wl, dev)
    step = mos.OwnerStep(local_rank)
    step.set_muon(mat.masters, mat.momenta, mat.grads, mat.params)
    if wl.vectors:
        step.set_adamw(mat.v_masters, mat.v_exp_avg, mat.v_exp_avg_sq, mat.v_grads, mat.v_params)
    stream = torch.cuda.current_stream()
    t_counter = [0]

    muon_kw = dict(lr=h["lr"], momentum=h["momentum"], wd=h["wd"], ns_steps=h["ns_steps"], a=h["a"],
                   b=h["b"], c=h["c"], nesterov=h["nesterov"], fp32_ns=h["fp32_ns"])

    def one_step():
        adam_kw = None
        if wl.vectors:
            t_counter[0] += 1
            adam_kw = dict(lr=h["adam_lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["adam_eps"],
                           wd=h["adam_wd"], step=t_counter[0])
        if args.overlap_adamw:
            step.step(muon_kw, adam_kw, stream=stream)
        else:
            step.muon_step(stream=stream, **muon_kw)
            if adam_kw is not None:
                step.adamw_step(stream=stream, **adam_kw)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        one_step()
    step.sync(stream)

    # ---------------- timed region: K steps, device events on the stream
    clocks = ClockSampler(local_rank)
    clocks.start()
    step.profile(True)
    step.profile_read()
    launches0 = step.kernel_launches()
    # State smaller than a few L2 sizes would stay cached from one step to
    # the next: then every step is timed on its own and L2 is flushed (a
    # write of twice its size) between steps, outside the timed spans.
    state_bytes = sum(t.numel() * t.element_size() for t in mat.flats.values())
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if state_bytes < 4 * L2_BYTES else None
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if flush is None:
        e0.record(stream)
        for _ in range(args.steps):
            one_step()
        e1.record(stream)
        torch.cuda.synchronize()
        total_ms = e0.elapsed_time(e1)
    else:
        total_ms = 0.0
        for _ in range(args.steps):
            flush.fill_(1)
            e0.record(stream)
            one_step()
            e1.record(stream)
            torch.cuda.synchronize()
            total_ms += e0.elapsed_time(e1)
    barrier()
    launches = step.kernel_launches() - launches0
    prof = step.profile_read()
    step.profile(False)
    clk = clocks.stop()
    step.sync(stream)
    ms = reduce_max_over_ranks(total_ms / args.steps, dist, dev)
    l2_note = ("inputs larger than L2 (no flush needed)" if flush is None else
               "L2 flushed between steps (each step timed on its own)")
    del flush

    # ---------------- end to end: host grads in, host bf16 params out.
    # Through dmuon_step_host: every step copies this step's gradients in
    # from page-locked host memory and the bf16 parameters out, group by
    # group, overlapped with the other groups' compute.  No overlap across
    # steps (the next step's gradients would depend on these parameters).
    e2e_steps = max(1, min(args.steps, 3))
    g_flat, p_flat = mat.flats["grad"], mat.flats["param"]
    host_g = torch.empty(g_flat.shape, dtype=g_flat.dtype, pin_memory=True)
    host_p = torch.empty(p_flat.shape, dtype=p_flat.dtype, pin_memory=True)
    host_g.copy_(g_flat)

    def host_views(flat_host, flat_dev, views):
        base = flat_dev.data_ptr()
        out = []
        for v in views:
            o = (v.data_ptr() - base) // v.element_size()
            out.append(flat_host[o:o + v.numel()].view(v.shape))
        return out

    step.set_host_io(host_views(host_g, g_flat, mat.grads), host_views(host_p, p_flat, mat.params),
                     host_views(host_g, g_flat, mat.v_grads) if wl.vectors else None,
                     host_views(host_p, p_flat, mat.v_params) if wl.vectors else None)

    def e2e_step():
        adam_kw = None
        if wl.vectors:
            t_counter[0] += 1
            adam_kw = dict(lr=h["adam_lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["adam_eps"],
                           wd=h["adam_wd"], step=t_counter[0])
        step.step_host(muon_kw, adam_kw, n_groups=args.e2e_groups, stream=stream)

    e2e_step()
    step.sync(stream)
    barrier()
    torch.cuda.synchronize()
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = reduce_max_over_ranks(x0.elapsed_time(x1) / e2e_steps, dist, dev)
    h2d = g_flat.numel() * g_flat.element_size()
    d2h = p_flat.numel() * p_flat.element_size()
    # One more host-buffer step with the library's timeline on: when the
    # gradient copies, each group's compute and the parameter copies ended.
    step.profile(True)
    e2e_step()
    tl = step.host_timeline()
    step.profile_read()
    step.profile(False)
    step.sync(stream)
    # The host link's own rate in this run (one plain copy each way), which
    # bounds e2e from below once the copies are the longer side.
    link = {}
    for name, fn, nbytes in (("h2d_gbs", lambda: g_flat.copy_(host_g, non_blocking=True), h2d),
                             ("d2h_gbs", lambda: host_p.copy_(p_flat, non_blocking=True), d2h)):
        torch.cuda.synchronize()
        x0.record(stream)
        fn()
        x1.record(stream)
        torch.cuda.synchronize()
        link[name] = nbytes / (x0.elapsed_time(x1) / 1e3) / 1e9
    # Both directions at once (the pipelined step overlaps them).
    side = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    x0.record(stream)
    side.wait_event(x0)
    g_flat.copy_(host_g, non_blocking=True)
    with torch.cuda.stream(side):
        host_p.copy_(p_flat, non_blocking=True)
    stream.wait_stream(side)
    x1.record(stream)
    torch.cuda.synchronize()
    link["both_ways_gbs"] = (h2d + d2h) / (x0.elapsed_time(x1) / 1e3) / 1e9
    del host_g, host_p
    # The end-to-end time's own bound: the longest of the gradient copies,
    # the parameter copies and the device-only step, plus what the pipeline
    # cannot hide -- the first group's gradients before any compute and the
    # last group's parameters after it (both taken from the timeline).
    e2e_detail = None
    if tl is not None and tl["groups"]:
        first_in = tl["groups"][0][0]
        last_out = tl["end"] - tl["groups"][-1][1]
        bound = max(h2d / (link["h2d_gbs"] * 1e9) * 1e3, d2h / (link["d2h_gbs"] * 1e9) * 1e3,
                    (h2d + d2h) / (link["both_ways_gbs"] * 1e9) * 1e3, ms) + first_in + last_out
        e2e_detail = {
            "lower_bound_ms": bound, "frac_of_bound": bound / e2e_ms,
            "timeline_ms": {"h2d_done": tl["h2d_done"], "compute_done": tl["groups"][-1][1], "end": tl["end"],
                            "first_group_h2d": first_in, "last_group_d2h": last_out,
                            "compute_waiting_for_h2d": sum(max(0.0, g[0] - (tl["groups"][i - 1][1] if i else 0.0))
                                                           for i, g in enumerate(tl["groups"]))},
            "groups": len(tl["groups"]),
            "per_group_ms": [[round(x, 2) for x in g] for g in tl["groups"]],
        }

    if rank != 0:
        return
    peaks = _peaks()
    ns_flops = W.workload_ns_flops(wl)
    ns_ms = sum(prof[k][0] for k in ("ns_gram", "ns_poly", "ns_combine")) / args.steps
    ns_launches = sum(prof[k][1] for k in ("ns_gram", "ns_poly", "ns_combine"))
    ns_tflops = ns_flops / (ns_ms / 1e3) / 1e12 if ns_ms > 0 else None
    # Roofline on the algorithmic flops of the symmetric iteration (upper
    # triangles of X X^T and A A, i.e. p(p+1)/2 dot products each), not the
    # dense count, so the fraction is not inflated.  The kernels compute the
    # diagonal 256-blocks in full, so they execute slightly more than this.
    ns_alg = W.workload_ns_flops_algorithmic(wl) if not h["fp32_ns"] else ns_flops
    ns_alg_tflops = ns_alg / (ns_ms / 1e3) / 1e12 if ns_ms > 0 else None
    # Streaming kernels: bytes of the passes that actually ran as their own
    # launches (the update runs inside the last NS product on the bf16 path).
    ew_parts = {"momentum": W.momentum_bytes(wl), "adamw": W.adamw_bytes(wl)}
    if prof["update"][1] > 0:
        ew_parts["update"] = W.update_bytes(wl)
    ew_bytes = sum(ew_parts.values())
    ew_ms = sum(prof[k][0] for k in list(ew_parts) + ["norm"]) / args.steps
    ew_gbs = ew_bytes / (ew_ms / 1e3) / 1e9 if ew_ms > 0 else None
    ew_detail = {k: {"ms": prof[k][0] / args.steps,
                     "GB/s": (v / (prof[k][0] / args.steps / 1e3) / 1e9) if prof[k][0] > 0 else None}
                 for k, v in ew_parts.items()}
    # The same kernels on the algorithmic bytes per element of the scope
    # table (momentum 12 with bf16 grads, update 12, AdamW 28): the X0 low
    # half the momentum pass also writes is not counted as work.
    ew_alg = {"momentum": W.momentum_bytes_algorithmic(wl), "adamw": W.adamw_bytes(wl)}
    if "update" in ew_parts:
        ew_alg["update"] = W.update_bytes(wl)
    ew_alg_gbs = sum(ew_alg.values()) / (ew_ms / 1e3) / 1e9 if ew_ms > 0 else None
    for k, v in ew_alg.items():
        ew_detail[k]["GB/s_algorithmic"] = (v / (prof[k][0] / args.steps / 1e3) / 1e9) if prof[k][0] > 0 else None
        ew_detail[k]["frac_algorithmic"] = (ew_detail[k]["GB/s_algorithmic"] / peaks["hbm_gbs"]
                                            if ew_detail[k]["GB/s_algorithmic"] else None)
    peak = peaks["bf16_sustained"]
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "ns_tc_traffic.json")
    if os.path.exists(tpath):
        try:
            tj = json.load(open(tpath))
            if tj.get("kernel_sha256") == kernel_source_sha() and tj.get("workload") == wl.name:
                traffic = tj.get("bytes_per_step")
        except (OSError, ValueError, KeyError):
            traffic = None
    line = {
        "metric": METRIC, "value": world * ns_flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": _workload_desc(wl), "ns_steps": h["ns_steps"],
                   "ns_operands": "fp32 in NS mode" if h["fp32_ns"] else "bf16 operands, fp32 accumulate",
                   "state": "fp32 master/momentum/AdamW moments, bf16 grads and params",
                   "l2": l2_note, "parallelism": f"replicas x{world}",
                   "adamw": "side stream beside the Muon step" if args.overlap_adamw else "after the Muon step"},
        "flops_basis": "dense_count",
        "ns_tflops_dense_count": ns_tflops,
        "ns_tflops_algorithmic": ns_alg_tflops,
        "ns_tflop_per_step": {"dense_count": ns_flops / 1e12, "algorithmic": ns_alg / 1e12},
        "ns_dense_count_frac_of_bf16_sustained": (ns_tflops / peak) if ns_tflops else None,
        "roofline": {"bound": "tensor", "kernel": "ns_tc2_kernel (all NS phases, algorithmic flops)",
                     "achieved": ns_alg_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": (ns_alg_tflops / peak) if ns_alg_tflops else None,
                     "frac_of_burst": (ns_alg_tflops / peaks["bf16_burst"]) if ns_alg_tflops else None,
                     "peak_src": f"{peaks['src']} bf16 sustained",
                     "traffic": traffic, "launches_per_step": ns_launches / args.steps,
                     "clock_normalized": _clock_normalized(ns_alg_tflops, peak, clk)},
        "elementwise": {"bound": "hbm", "achieved": ew_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": (ew_gbs / peaks["hbm_gbs"]) if ew_gbs else None,
                        "bytes_per_step": ew_bytes, "achieved_algorithmic": ew_alg_gbs,
                        "frac_algorithmic": (ew_alg_gbs / peaks["hbm_gbs"]) if ew_alg_gbs else None,
                        "bytes_per_step_algorithmic": sum(ew_alg.values()), "kernels": ew_detail},
        "kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
        "gpu_launches": launches,
        "e2e": {"value": world * ns_flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "api": "dmuon_step_host", "n_groups": args.e2e_groups,
                "host_link": link, "attribution": e2e_detail},
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        sample = _oracle_sample(wl)
        secs, flops, est = _oracle_time(wl, sample)
        line["cpu_baseline"] = {"value": ns_flops / est / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
                                "kind": "oracle", "sample": _sample_desc(wl, sample),
                                "sample_seconds": secs, "est_ms_per_step": est * 1e3}
    print(json.dumps(line), flush=True)
    step.close()

# ------------------------------------------------ owner-partitioned (N > 1)
SHARDED_NAMES = ("embed_tokens", "word_embeddings", "wte", "lm_head")


def _route(spec):
    """Route of an AdamW-side tensor by the pages' policy: embedding and
    output tables "sharded_adamw", everything else "adamw"."""
    return "sharded_adamw" if any(k in spec.name for k in SHARDED_NAMES) else "adamw"


def run_owner(args, wl, rank, world, local_rank, dist):
    """One optimizer step of the whole model over `world` ranks, the pages'
    way: every Muon / small-AdamW tensor stepped once, by its owner, after
    the mean gradient is reduced to it; parameters broadcast from owners;
    embedding-like tables sharded (reduce_scatter / all_gather).  Total work
    is one model's step whatever the rank count (strong scaling)."""
    import torch

    import matrix_optimizer_step_gb300 as mos
    from matrix_optimizer_step_gb300 import workloads as W
    from matrix_optimizer_step_gb300.owner_dist import DistributedOwnerStep, OwnerLayout

    dev_index = local_rank % torch.cuda.device_count()
    torch.cuda.set_device(dev_index)
    dev = torch.device("cuda", dev_index)
    mos.load_library()
    for kv in args.tuning:
        k, v = kv.split("=")
        mos.dmuon_set_tuning(int(k), int(v))
    h = wl.hyper
    adam_idx = [j for j, v in enumerate(wl.vectors) if _route(v) == "adamw"]
    shard_idx = [j for j, v in enumerate(wl.vectors) if _route(v) == "sharded_adamw"]
    L = OwnerLayout.build([s.shape for s in wl.matrices], [wl.vectors[j].numel for j in adam_idx],
                          [wl.vectors[j].numel for j in shard_idx], world, ns_steps=h["ns_steps"])
    ds = DistributedOwnerStep(L, device=dev)
    order = [("m", i) for i in range(len(wl.matrices))] + [("v", j) for j in adam_idx] + [("v", j) for j in shard_idx]
    for t, (kind, i) in enumerate(order):
        w = W.master_init(wl.matrices[i], i, dev) if kind == "m" else W.vector_init(wl.vectors[i], i, dev)
        ds.load_weight(t, w)
        del w
    # This rank's gradients (each data-parallel rank has its own).
    for t, (kind, i) in enumerate(order):
        g = (W.muon_grad(wl, wl.matrices[i], i, step=rank, device=dev) if kind == "m"
             else W.vector_grad(wl.vectors[i], i, step=rank, device=dev))
        ds.grads()[t].copy_(g.reshape(ds.grads()[t].shape))
        del g
    g_save = (ds.grad_flat.clone(), ds.sp_grad_flat.clone())  # the gradients every step starts from
    muon_kw = dict(lr=h["lr"], momentum=h["momentum"], wd=h["wd"], ns_steps=h["ns_steps"], a=h["a"], b=h["b"],
                   c=h["c"], nesterov=h["nesterov"], fp32_ns=h["fp32_ns"])
    t_counter = [0]
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    phase_ms = [0.0, 0.0, 0.0]

    def one_step(timed):
        t_counter[0] += 1
        adam_kw = dict(lr=h["adam_lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["adam_eps"], wd=h["adam_wd"],
                       step=t_counter[0])
        # The gradients of a fresh backward pass (a reduce leaves the
        # non-owners' copies undefined).
        ds.grad_flat.copy_(g_save[0])
        ds.sp_grad_flat.copy_(g_save[1])
        ev[0].record(stream)
        ds.reduce_grads()
        ev[1].record(stream)
        ds.local_step(muon_kw, adam_kw, stream=stream)
        ev[2].record(stream)
        ds.publish_params()
        ev[3].record(stream)
        if timed:
            torch.cuda.synchronize()
            for k in range(3):
                phase_ms[k] += ev[k].elapsed_time(ev[k + 1])

    for _ in range(args.warmup):
        one_step(False)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev_index)
    clocks.start()
    ds.stepper.profile(True)
    ds.stepper.profile_read()
    launches0 = ds.stepper.kernel_launches()
    dist.barrier()
    torch.cuda.synchronize()
    total_ms = 0.0
    for _ in range(args.steps):
        one_step(True)
        total_ms += sum(ev[k].elapsed_time(ev[k + 1]) for k in range(3))
    torch.cuda.synchronize()
    dist.barrier()
    launches = ds.stepper.kernel_launches() - launches0
    prof = ds.stepper.profile_read()
    ds.stepper.profile(False)
    clk = clocks.stop()
    ms = reduce_max_over_ranks(total_ms / args.steps, dist, dev)
    ns_ms = sum(prof[k][0] for k in ("ns_gram", "ns_poly", "ns_combine")) / args.steps
    mine_muon = [i for i in L.owned(rank) if i < len(wl.matrices)]
    own_alg = sum(W.ns_flops_algorithmic(*wl.matrices[i].mn, h["ns_steps"]) * wl.matrices[i].n_slices
                  for i in mine_muon)
    own_tflops = own_alg / (ns_ms / 1e3) / 1e12 if ns_ms > 0 else 0.0
    stats = torch.tensor([ns_ms, phase_ms[0] / args.steps, phase_ms[1] / args.steps, phase_ms[2] / args.steps,
                          own_tflops, float(launches)], dtype=torch.float64,
                         device=dev if args.dist_backend == "nccl" else "cpu")  # gloo gathers host tensors
    gathered = [torch.empty_like(stats) for _ in range(world)]
    dist.all_gather(gathered, stats)
    per_rank = [g.tolist() for g in gathered]

    # End to end: this rank's gradients in from page-locked host memory, the
    # step, the bf16 parameters out (copies and step one after the other).
    # One page-locked buffer per flat serves both directions (the parameters
    # come back where the gradients came from), halving the pinned host
    # memory of N ranks on one host; later steps then read the previous
    # step's parameters as gradients, which changes no timing.
    host_g = torch.empty(ds.grad_flat.shape, dtype=ds.grad_flat.dtype, pin_memory=True)
    host_sg = torch.empty(ds.sp_grad_flat.shape, dtype=ds.sp_grad_flat.dtype, pin_memory=True)
    host_p, host_sp = host_g, host_sg
    host_g.copy_(g_save[0])
    host_sg.copy_(g_save[1])
    e2e_steps = max(1, min(args.steps, 3))
    dist.barrier()
    torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(e2e_steps):
        t_counter[0] += 1
        ds.grad_flat.copy_(host_g, non_blocking=True)
        ds.sp_grad_flat.copy_(host_sg, non_blocking=True)
        ds.step(muon_kw, dict(lr=h["adam_lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["adam_eps"],
                              wd=h["adam_wd"], step=t_counter[0]), stream=stream)
        host_p.copy_(ds.param_flat, non_blocking=True)
        host_sp.copy_(ds.sp_param_flat, non_blocking=True)
    x1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    e2e_ms = reduce_max_over_ranks(x0.elapsed_time(x1) / e2e_steps, dist, dev)
    h2d = world * (host_g.numel() * host_g.element_size() + host_sg.numel() * host_sg.element_size())
    d2h = world * (host_p.numel() + host_sp.numel()) * 2
    ds.stepper.sync()
    if rank != 0:
        ds.close()
        return
    peaks = _peaks()
    ns_flops = W.workload_ns_flops(wl)
    peak = peaks["bf16_sustained"]
    ach = min(r[4] for r in per_rank)
    line = {
        "metric": METRIC, "value": ns_flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": _workload_desc(wl), "ns_steps": h["ns_steps"],
                   "ns_operands": "bf16 operands, fp32 accumulate",
                   "state": "fp32 master/momentum/AdamW moments on owners only, bf16 grads and params on every rank",
                   "l2": "inputs larger than L2 (no flush needed)",
                   "parallelism": f"owner x{world}: mean grads reduced to owners, owners step, bf16 params "
                                  f"broadcast; embedding tables reduce_scatter / all_gather",
                   "backend": args.dist_backend},
        "flops_basis": "dense_count",
        "roofline": {"bound": "tensor", "kernel": "ns_tc2_kernel (owned tensors' NS phases, algorithmic flops; "
                                                  "slowest rank)",
                     "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak if ach else None,
                     "peak_src": f"{peaks['src']} bf16 sustained", "traffic": None},
        "owner": {"per_rank": [{"ns_ms": r[0], "reduce_ms": r[1], "step_ms": r[2], "publish_ms": r[3],
                                "ns_tflops_algorithmic": r[4], "launches": int(r[5])} for r in per_rank],
                  "owned_elements": [sum(math.prod(L.muon_shapes[i]) if i < len(L.muon_shapes)
                                         else L.adamw_numels[i - len(L.muon_shapes)] for i in L.owned(r))
                                     for r in range(world)]},
        "gpu_launches": int(sum(r[5] for r in per_rank)),
        "e2e": {"value": ns_flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "DistributedOwnerStep.step with host copies before and after"},
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    ds.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="llama3_8b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-groups", type=int, default=12,
                    help="groups of the host-buffer step (copies of one group overlap the others' compute)")
    ap.add_argument("--overlap-adamw", action="store_true",
                    help="run the AdamW step on a side stream beside the Muon step (OwnerStep.step); "
                         "per-kernel AdamW times then include waiting for SMs")
    ap.add_argument("--mode", choices=("owner", "replicas"), default=None,
                    help="with --gpus N > 1: the owner-partitioned step of one model (default), or N "
                         "independent replicas of the one-GPU step; --mode owner under torchrun with one "
                         "rank runs the owner step on a process group of one")
    ap.add_argument("--dist-backend", choices=("nccl", "gloo"), default="nccl",
                    help="process-group backend for N > 1 (gloo only to check the code path)")
    ap.add_argument("--tuning", action="append", default=[],
                    help="KEY=VALUE passed to dmuon_set_tuning before the run")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from matrix_optimizer_step_gb300 import workloads as W

    wl = W.workload(args.workload)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return
    # The owner-partitioned step: the default with several ranks; with one
    # rank only when asked for under torchrun (a group of one).
    owner = args.mode == "owner" or (args.mode is None and world > 1)
    if owner and world == 1 and "MASTER_ADDR" not in os.environ:
        ap.error("--mode owner with one rank needs torchrun (a process group of one)")
    grouped = world > 1 or owner
    if grouped:
        import torch.distributed as dist

        dist.init_process_group(args.dist_backend)
    try:
        if owner:
            run_owner(args, wl, rank, world, local_rank, dist)
        else:
            run_ours(args, wl, rank, world, local_rank)
    finally:
        if grouped:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
