#!/usr/bin/env python3
"""Benchmark of the block-sparse matmul hot path on GB300.

One step = fprop + bprop + updat of the hidden-4096, block-32, 50%-dense
layout (128 x 128 Bernoulli(0.5) blocks), bf16 activations in (N, C) layout,
at minibatch N = 1024 and N = 64 (six passes).  The metric is effective
TFLOP/s = 2 * N * nnz * bs^2 per pass, summed over the step, divided by the
device time of the step.

Streams: the minibatch-1024 and minibatch-64 problems are independent, so a step
runs the three minibatch-64 passes on a second stream, forked from and joined
back into the timing stream inside the step: they fill the SMs that the
dense-tile kernels of the minibatch-1024 passes leave idle.

Timing: W warm-up steps, then exactly K timed steps.  Four input/output sets
(each ~83 MB, together > 2x the 129 MB L2) rotate between steps, so every step
reads cold inputs.  Steps are enqueued in chunks of 50 behind a short device
sleep so that the host never starves the GPU inside a chunk.  CUDA events on
the timing stream bracket every chunk of back-to-back steps (an event between
steps would keep a step's first kernel from overlapping the previous step's
last one under programmatic dependent launch, which back-to-back training steps
do); the reported device time is the sum of the chunk intervals, the sleeps
outside them.  A second pass over the same K steps runs the passes on one
stream and brackets every kernel with events, which gives each kernel's own
duration for the per-pass table and the roofline object.

With --gpus N under torchrun every rank holds its own minibatch rows (a global minibatch of N
times as many rows, weak scaling) and the replicated weight; each weight gradient is summed over
the ranks by one NCCL all-reduce inside the timed step (block_sparse_matrix_gb300.dp).

--impl reference times the float64 CPU oracle (the only other implementation
of the method here) on a bounded sample of the same workload.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_matrix_gb300 import dp, workloads as wk  # noqa: E402

METRIC = "effective TFLOP/s per pass (fprop/bprop/updat) and % of roofline on 1 GB300"
WORKLOAD = ("hidden C=K=4096, block_size=32, 128x128 Bernoulli(0.5) layout, bf16 inputs with fp32 accumulate, "
            "feature_axis=1 (N,C); one step = fprop+bprop+updat at N=1024 and at N=64")
NSETS = 4
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws, device):
    """The largest value of x over the ranks of the default process group (x itself at
    world size 1): the job's time is that of its slowest replica."""
    if ws <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ws, step_flops, steps, dev_ms):
    """Whole-job effective TFLOP/s: every replica does step_flops per step (weak scaling),
    and the job takes the slowest replica's dev_ms for `steps` steps."""
    return ws * step_flops * steps / (dev_ms * 1e-3) / 1e12


# ---- pass bookkeeping -------------------------------------------------------------------

def pass_list(nnz, bs, C, K, Ns, e=2):
    """(name, N, effective flops, algorithmic bytes) per pass of one step."""
    out = []
    for N in Ns:
        f = wk.effective_flops(N, nnz, bs)
        wbytes = nnz * bs * bs * e
        out.append(("fprop_n%d" % N, N, f, (N * C + N * K) * e + wbytes))
        out.append(("bprop_n%d" % N, N, f, (N * C + N * K) * e + wbytes))
        out.append(("updat_n%d" % N, N, f, (N * C + N * K) * e + nnz * bs * bs * 4))
    return out


def roof_time(flops, bytes_, peaks):
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = bytes_ / (peaks["hbm_gbs"] * 1e9)
    return max(t_tc, t_hbm), ("tensor" if t_tc >= t_hbm else "hbm")


# ---- clocks ------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- our implementation --------------------------------------------------------------------

def traffic_for(kernel_pass):
    """(read, write) DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else (None, None)).  ncu counts DRAM traffic inside the
    kernel's own duration: the kernel's outputs are written into the 129 MB L2 and reach DRAM
    after the kernel ends, so the write figure is not the kernel's write-back."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        d = json.load(f)
    if d.get("src_sha") != source_sha():
        return None, None
    e = d.get("passes", {}).get(kernel_pass)
    if not isinstance(e, dict):
        return None, None
    return e.get("read"), e.get("write")


def source_sha():
    """Hash of the sources of the step's kernels: every file in csrc/ but the normalisations,
    the projections, the SIMT and the block-size 16/8 kernels, none of which the step runs."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_sparse_matrix_gb300", "csrc")
    skip = ("bsmm_norm.cu", "bsmm_wnorm.cu", "bsmm_proj.cu", "bsmm_simt.cu", "bsmm_sp.cu")
    for name in sorted(n for n in os.listdir(csrc) if n not in skip):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def run_ours(args):
    from block_sparse_matrix_gb300 import bsmm
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    wl = wk.CONFIGS["h4096_b32_p50_n1024"]
    Ns = [1024, 64]
    inp = wk.make_inputs(wl)
    L, bs, C, K = inp.layout, wl.bs, wl.C, wl.K
    m = bsmm.BlocksparseMatMul(L, block_size=bs, feature_axis=1)
    nnz = m.nnz
    passes = pass_list(nnz, bs, C, K, Ns)
    if args.only:
        passes = [p for p in passes if p[0] == args.only]
        if not passes:
            raise SystemExit("--only must name one of fprop_n1024 bprop_n1024 updat_n1024 fprop_n64 bprop_n64 updat_n64")
    step_flops = sum(p[2] for p in passes)

    # Rotating device sets: inputs (x, dy per N, w) and outputs (y, dx per N, dw per N).
    sets = []
    for s in range(NSETS):
        d = {"w": (inp.w if s == 0 else wk.normals(inp.w.shape, 9000 + s, float(np.sqrt(wl.w_var)),
                                                    wl.dtype)).to(dev)}
        for N in Ns:
            d["x%d" % N] = wk.normals((N, C), 9100 + 10 * s + N % 7, 1.0, wl.dtype).to(dev)
            d["dy%d" % N] = wk.normals((N, K), 9200 + 10 * s + N % 7, 1.0, wl.dtype).to(dev)
            d["y%d" % N] = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
            d["dx%d" % N] = torch.empty((N, C), dtype=torch.bfloat16, device=dev)
            d["dw%d" % N] = torch.empty((nnz, bs, bs), dtype=torch.float32, device=dev)
        sets.append(d)
    stream = torch.cuda.current_stream()

    def launch_pass(name, d):
        kind, n = name.split("_n")
        N = int(n)
        if kind == "fprop":
            bsmm.bsmm_fprop(m.handle, d["x%d" % N], d["w"], d["y%d" % N], N)
        elif kind == "bprop":
            bsmm.bsmm_bprop(m.handle, d["dy%d" % N], d["w"], d["dx%d" % N], N)
        else:
            bsmm.bsmm_updat(m.handle, d["x%d" % N], d["dy%d" % N], d["dw%d" % N], N)

    def exchange(name, d):
        # Data parallel over the minibatch: every rank holds its own N rows of a global minibatch of
        # N * world rows and the replicated weight; the weight gradient is summed over the ranks
        # (one NCCL all-reduce per weight gradient; none on one GPU).
        if ws > 1 and name.startswith("updat"):
            dp.allreduce_dw(d["dw%s" % name.split("_n")[1]])

    side = torch.cuda.Stream(device=dev)
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
    big = [p for p in passes if p[1] == max(Ns)]
    small = [p for p in passes if p[1] != max(Ns)]

    def step(i):
        # The two minibatches are independent problems: the small one's passes (and their weight
        # gradient all-reduce) run on the side stream, forked from and joined back into the
        # current stream inside the step.
        d = sets[i % NSETS]
        cur = torch.cuda.current_stream()
        if small and big:
            ev_fork.record(cur)
            side.wait_event(ev_fork)
            with torch.cuda.stream(side):
                for p in small:
                    launch_pass(p[0], d)
                    exchange(p[0], d)
            for p in big:
                launch_pass(p[0], d)
                exchange(p[0], d)
            ev_join.record(side)
            cur.wait_event(ev_join)
        else:
            for p in passes:
                launch_pass(p[0], d)
                exchange(p[0], d)

    # Warm-up (W steps), then count our launches per step.
    warm = max(3, args.warmup)
    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    m.sync_status()
    c0 = bsmm.launch_count()
    step(0)
    torch.cuda.synchronize()
    launches_per_step = bsmm.launch_count() - c0

    # Host enqueue time per step -> device sleep long enough to cover a chunk.
    t0 = time.perf_counter()
    for i in range(20):
        step(i)
    host_step_s = (time.perf_counter() - t0) / 20
    torch.cuda.synchronize()
    chunk = 50
    sleep_cycles = int(host_step_s * 1.3 * chunk * 2.1e9) + 100000   # cycles at <= 2.1 GHz

    K_steps = args.steps

    def timed(per_pass):
        # Steps are queued in chunks behind a device sleep so the host never starves the GPU.
        # Without per_pass, events bracket each chunk of back-to-back steps (streams as in a real
        # training loop); with per_pass, the passes run on one stream and events bracket every
        # kernel, which gives each kernel's own duration.
        ev_chunk = []
        ev_pass = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in passes]
                   for _ in range(K_steps)] if per_pass else None
        for c0 in range(0, K_steps, chunk):
            torch.cuda._sleep(sleep_cycles)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(c0, min(K_steps, c0 + chunk)):
                d = sets[i % NSETS]
                if not per_pass:
                    step(i)
                    continue
                for j, p in enumerate(passes):
                    ev_pass[i][j][0].record(stream)
                    launch_pass(p[0], d)
                    ev_pass[i][j][1].record(stream)
                    exchange(p[0], d)
            b.record(stream)
            ev_chunk.append((a, b))
        return ev_chunk, ev_pass

    sampler = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    ev_chunk, _ = timed(False)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    if ws > 1:
        torch.distributed.barrier()
    _, ev_pass = timed(True)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    m.sync_status()

    dev_ms = sum(a.elapsed_time(b) for a, b in ev_chunk)
    pass_us = {}
    for j, p in enumerate(passes):
        pass_us[p[0]] = 1000.0 * sum(ev_pass[i][j][0].elapsed_time(ev_pass[i][j][1]) for i in range(K_steps)) / K_steps
    dev_ms = max_over_ranks(dev_ms, ws, dev)
    ms_per_step = dev_ms / K_steps
    value = job_value(ws, step_flops, K_steps, dev_ms)

    peaks, peak_src = load_peaks()
    per_pass = {}
    for name, N, f, b in passes:
        t = pass_us[name] * 1e-6
        tr, bound = roof_time(f, b, peaks)
        per_pass[name] = {"us": round(pass_us[name], 3), "tflops": round(f / t / 1e12, 2),
                          "gbs": round(b / t / 1e9, 1), "roofline_us": round(tr * 1e6, 3), "bound": bound,
                          "roofline_frac": round(tr / t, 4)}
    dom = max(passes, key=lambda p: pass_us[p[0]])
    name, N, f, b = dom
    t = pass_us[name] * 1e-6
    tr, bound = roof_time(f, b, peaks)
    if bound == "tensor":
        achieved, peak, unit = f / t / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = b / t / 1e9, peaks["hbm_gbs"], "GB/s"
    rd, wr = traffic_for(name)
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4),
                "traffic": (rd + wr) if rd is not None and wr is not None else None,
                "dram_read_bytes": rd, "dram_write_bytes": wr,
                "dram_write_note": "ncu counts DRAM bytes inside the kernel's duration; outputs are written into "
                                   "L2 and written back to DRAM after the kernel, so the write field does not "
                                   "measure this kernel's write-back",
                "kernel": name, "algorithmic_bytes": b, "flops": f, "peak_source": peak_src + " (burst)"}

    e2e = run_e2e(m, inp, Ns, passes, dev, args) if (rank == 0 and not args.only) else None
    configs = run_configs(dev, peaks, args.config_reps) if (rank == 0 and not args.only and
                                                             args.config_reps > 0) else None
    cpu = (run_cpu_baseline(wl, inp, Ns, budget_s=args.cpu_budget)
           if (rank == 0 and ws == 1 and args.cpu_budget > 0) else None)

    if configs is not None:
        # the same kernel launched back to back over rotating inputs (the configs timing): how it runs
        # inside a stream of passes, without the launch floor a kernel timed alone carries
        cname = "h4096_b32_p50_n%d" % N
        pname = name.split("_n")[0]
        st = configs.get(cname, {}).get("passes", {}).get(pname, {}).get("us_stream")
        if st:
            a2 = (f if bound == "tensor" else b) / (st * 1e-6) / (1e12 if bound == "tensor" else 1e9)
            roofline["achieved_back_to_back"] = round(a2, 2)
            roofline["frac_back_to_back"] = round(a2 / peak, 4)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws, "steps": K_steps,
                "warmup": warm, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normals)",
                "config": {"workload": WORKLOAD, "nnz": nnz, "l2": "4 rotating input/output sets, ~330 MB > 2x L2",
                           "streams": "minibatch-64 passes on a second stream, forked and joined inside each step",
                           "timing": "CUDA events around chunks of %d back-to-back steps; sleeps between chunks "
                                     "are outside the timed intervals" % chunk,
                           "parallelism": ("data parallel over the minibatch: %d rows per GPU, weight gradients "
                                           "all-reduced over NCCL inside the step" % max(Ns)) if ws > 1
                           else "single GPU"},
                "passes": per_pass, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "configs": configs,
                "clocks": clocks, "gpu_launches": launches_per_step * K_steps,
                "wall_s_timed_region": round(wall1 - wall0, 3)}
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_e2e(m, inp, Ns, passes, dev, args):
    """The same step through the public API from pinned HOST buffers: every step uploads its
    inputs, runs the six passes and downloads its results, all inside the timed region.  Steps
    are pipelined over three streams (uploads, passes, downloads) with two device buffer sets
    ordered by events, so step i+1's uploads and step i-1's downloads overlap step i's passes."""
    from block_sparse_matrix_gb300 import bsmm
    wl = wk.CONFIGS["h4096_b32_p50_n1024"]
    C, K, bs, nnz = wl.C, wl.K, wl.bs, m.nnz
    host = {"w": inp.w.pin_memory()}
    for N in Ns:
        host["x%d" % N] = wk.normals((N, C), 9300 + N, 1.0, wl.dtype).pin_memory()
        host["dy%d" % N] = wk.normals((N, K), 9400 + N, 1.0, wl.dtype).pin_memory()
        for k, shape, dt in (("y", (N, K), torch.bfloat16), ("dx", (N, C), torch.bfloat16),
                             ("dw", (nnz, bs, bs), torch.float32)):
            host["%s%d" % (k, N)] = torch.empty(shape, dtype=dt).pin_memory()
    devb = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    ins = ["w"] + ["x%d" % N for N in Ns] + ["dy%d" % N for N in Ns]
    outs = ["%s%d" % (k, N) for N in Ns for k in ("y", "dx", "dw")]
    h2d = sum(host[k].numel() * host[k].element_size() for k in ins)
    d2h = sum(host[k].numel() * host[k].element_size() for k in outs)
    steps = max(10, min(args.steps, 200))
    s_up, s_cmp, s_dn = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_dn = [torch.cuda.Event() for _ in range(2)]

    def one(i):
        b = i % 2
        d = devb[b]
        with torch.cuda.stream(s_up):
            if i >= 2:
                s_up.wait_event(ev_cmp[b])          # step i-2's passes have read this input set
            for k in ins:
                d[k].copy_(host[k], non_blocking=True)
            ev_up[b].record(s_up)
        s_cmp.wait_event(ev_up[b])
        if i >= 2:
            s_cmp.wait_event(ev_dn[b])              # step i-2's results have left this output set
        for name, N, _, _ in passes:
            kind = name.split("_n")[0]
            if kind == "fprop":
                bsmm.bsmm_fprop(m.handle, d["x%d" % N], d["w"], d["y%d" % N], N, stream=s_cmp)
            elif kind == "bprop":
                bsmm.bsmm_bprop(m.handle, d["dy%d" % N], d["w"], d["dx%d" % N], N, stream=s_cmp)
            else:
                bsmm.bsmm_updat(m.handle, d["x%d" % N], d["dy%d" % N], d["dw%d" % N], N, stream=s_cmp)
        ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_dn):
            s_dn.wait_event(ev_cmp[b])
            for k in outs:
                host[k].copy_(d[k], non_blocking=True)
            ev_dn[b].record(s_dn)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    for i in range(steps):
        one(i)
    e.record(s_dn)                                   # after the last step's downloads
    torch.cuda.synchronize()
    m.sync_status()
    ms = a.elapsed_time(e) / steps
    flops = sum(p[2] for p in passes)
    return {"value": round(flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 4), "steps": steps,
            "pipelined": "uploads, passes and downloads on three streams, two device buffer sets"}


# ---- every benchmark configuration, pass by pass ---------------------------------------------

# Derived fp32 FFMA peak for the fp32 configuration (no tensor cores): 152 SMs x 128 FMA/clk x
# 2 FLOP x 2.07 GHz (the unit counts and the maximum SM clock of a GB300).
FFMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def config_passes(wl, nnz):
    """(pass name, flops, algorithmic bytes, callable builder key) of one workload: fprop, bprop
    and updat at its minibatch, and for a workload with timesteps the per-step fprop/bprop and the
    grouped weight gradient of `group` steps accumulated into float32 dW."""
    e = 4 if wl.dtype == "f32" else 2
    N, C, K, bs = wl.N, wl.C, wl.K, wl.bs
    f = wk.effective_flops(N, nnz, bs)
    act = (N * C + N * K) * e
    out = [("fprop", f, act + nnz * bs * bs * e), ("bprop", f, act + nnz * bs * bs * e),
           ("updat", f, act + nnz * bs * bs * 4)]
    if wl.steps > 1:
        G = wl.group
        out.append(("updat_grouped_g%d" % G, G * f, G * act + 2 * nnz * bs * bs * 4))
    return out


def cold_times(fn, flush, reps):
    """Device microseconds of fn() launched alone, cold, reps times: each launch follows a 256 MB
    read-only sweep that evicts the L2, and every sweep, event and launch is queued behind one
    device sleep that outlasts the host's enqueue time, so the start event fires when the sweep
    ends with the launch already queued (host latency is not counted).  Median over reps."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(5):
        flush.sum()
        fn()
    host_s = (time.perf_counter() - t0) / 5
    torch.cuda.synchronize()
    torch.cuda._sleep(int(host_s * 1.5 * reps * 2.1e9) + 200000)     # cycles at <= 2.1 GHz
    evs = []
    for _ in range(reps):
        flush.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs) * 1000.0


def stream_times(fn, nsets, launches):
    """Device microseconds per launch of fn(i) launched `launches` times back to back on one
    stream (programmatic dependent launch lets each launch overlap the previous one's tail),
    rotating over nsets input/output sets whose total exceeds twice the L2, so every launch
    reads cold inputs.  Queued behind a device sleep that outlasts the host's enqueue time."""
    for i in range(nsets):
        fn(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(launches):
        fn(i % nsets)
    host_s = (time.perf_counter() - t0) / launches
    torch.cuda.synchronize()
    torch.cuda._sleep(int(host_s * 1.5 * launches * 2.1e9) + 200000)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(launches):
        fn(i % nsets)
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1000.0 / launches


def config_sets(wl, m, inp, dev, min_bytes=300 << 20, max_sets=32):
    """Copies of a configuration's inputs and outputs on the device, enough of them that their
    total exceeds min_bytes (more than twice the 129 MB L2)."""
    def one():
        d = {"x": inp.x.to(dev), "w": inp.w.to(dev), "dy": inp.dy.to(dev)}
        d["y"] = torch.empty(m.o_shape(wl.N), dtype=d["x"].dtype, device=dev)
        d["dx"] = torch.empty(m.i_shape(wl.N), dtype=d["x"].dtype, device=dev)
        d["dw"] = torch.zeros(m.w_shape, dtype=torch.float32, device=dev)
        if wl.steps > 1:
            d["xs"] = [a.to(dev) for a in inp.xs]
            d["dys"] = [a.to(dev) for a in inp.dys]
        return d
    sets = [one()]
    per = sum(t.numel() * t.element_size() for v in sets[0].values() for t in (v if isinstance(v, list) else [v]))
    n = min(max_sets, max(2, -(-min_bytes // per)))
    sets += [one() for _ in range(n - 1)]
    return sets


def recurrent_layer(wl, dev, flush, reps):
    """The recurrent layer's training pass as a user runs it, in backpropagation-through-time
    order: `steps` fprops through one weight (t = 0, 1, ...), then the bprops in reverse
    (t = steps-1, ..., 0); each group of `group` steps' weight gradient is accumulated into one
    float32 dW on a side stream as soon as the backward pass has produced that group's last dy
    (the group of the latest steps first), so it overlaps the remaining bprops; the side stream is
    joined at the end.  Launched eagerly, and captured once in a CUDA graph and replayed.  Device
    microseconds per layer (median over reps, each after the L2 sweep, queued behind a device
    sleep), with effective TFLOP/s."""
    from block_sparse_matrix_gb300 import bsmm
    inp = wk.make_inputs(wl)
    m = bsmm.BlocksparseMatMul(inp.layout, block_size=wl.bs, feature_axis=wl.feature_axis)
    T, G, N = wl.steps, wl.group, wl.N
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        w = inp.w.to(dev)
        xs = [a.to(dev) for a in inp.xs]
        dys = [a.to(dev) for a in inp.dys]
        ys = [torch.empty(m.o_shape(N), dtype=w.dtype, device=dev) for _ in range(T)]
        dxs = [torch.empty(m.i_shape(N), dtype=w.dtype, device=dev) for _ in range(T)]
        dw = torch.empty(m.w_shape, dtype=torch.float32, device=dev)

        side = torch.cuda.Stream(device=dev)
        groups = list(range(0, T, G))[::-1]             # the latest steps' group completes first

        def layer():
            cur = torch.cuda.current_stream()
            for t in range(T):
                m.fprop(xs[t], w, ys[t])
            for t in reversed(range(T)):
                m.bprop(dys[t], w, dxs[t])
                if t in groups:                          # every dy of the group t .. t+G-1 is known
                    ev = torch.cuda.Event()
                    ev.record(cur)
                    side.wait_event(ev)
                    with torch.cuda.stream(side):
                        m.updat_grouped(xs[t:t + G], dys[t:t + G], dw=dw, accumulate=t != groups[0])
            ev = torch.cuda.Event()
            ev.record(side)
            cur.wait_event(ev)

        layer()
        eager = cold_times(layer, flush, reps)
        g = torch.cuda.CUDAGraph()
    s.synchronize()
    with torch.cuda.graph(g, stream=s):
        layer()
    with torch.cuda.stream(s):
        graph = cold_times(g.replay, flush, reps)
    s.synchronize()
    m.sync_status()
    f = 2 * T * wk.effective_flops(N, m.nnz, wl.bs) + T * wk.effective_flops(N, m.nnz, wl.bs)
    m.close()
    return {"what": "%d fprops, then %d bprops in reverse step order, each group of %d steps' weight "
                    "gradient accumulated into float32 dW on a side stream once its dys are known "
                    "(overlapping the remaining bprops); %d launches" % (T, T, G, 2 * T + (T + G - 1) // G),
            "eager_us": round(eager, 3), "graph_us": round(graph, 3),
            "tflops_eager": round(f / (eager * 1e-6) / 1e12, 2), "tflops_graph": round(f / (graph * 1e-6) / 1e12, 2)}


def launch_floor(dev, flush, reps):
    """Fixed cost of a launch, timed the two ways the passes are: an empty kernel of 192 CTAs
    alone between events after the L2 sweep, and back to back; with and without a
    tensor-memory allocation (a kernel that contains tcgen05 instructions costs more to launch)."""
    from block_sparse_matrix_gb300 import bsmm
    h = bsmm.bsmm_create(np.ones((1, 1), np.uint8), 32, 1)
    try:
        out = {}
        for key, tm in (("tensor_memory_kernel", True), ("plain_kernel", False)):
            fn = lambda i=0: bsmm.bsmm_selftest_empty_launch(h, 192, tm)
            out[key] = {"alone_us": round(cold_times(fn, flush, reps), 3),
                        "stream_us": round(stream_times(fn, 1, 200), 3)}
        bsmm.bsmm_sync_status(h)
    finally:
        bsmm.bsmm_destroy(h)
    return out


def run_configs(dev, peaks, reps):
    """Each benchmark configuration on its own: every pass timed alone with CUDA events, cold
    (a 256 MB read-only sweep evicts the L2 before each timed launch), median over reps; and
    the same pass launched back to back over rotating input sets larger than the L2."""
    from block_sparse_matrix_gb300 import bsmm
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    out = {}
    for name, wl in wk.CONFIGS.items():
        inp = wk.make_inputs(wl, steps=min(wl.steps, wl.group) if wl.steps > 1 else None)
        m = bsmm.BlocksparseMatMul(inp.layout, block_size=wl.bs, feature_axis=wl.feature_axis)
        sets = config_sets(wl, m, inp, dev)
        calls = {"fprop": lambda i: m.fprop(sets[i]["x"], sets[i]["w"], sets[i]["y"]),
                 "bprop": lambda i: m.bprop(sets[i]["dy"], sets[i]["w"], sets[i]["dx"]),
                 "updat": lambda i: m.updat(sets[i]["x"], sets[i]["dy"], sets[i]["dw"])}
        if wl.steps > 1:
            calls["updat_grouped_g%d" % wl.group] = lambda i: m.updat_grouped(
                sets[i]["xs"], sets[i]["dys"], dw=sets[i]["dw"], accumulate=True)
        res = {}
        for pname, flops, byts in config_passes(wl, m.nnz):
            fn = calls[pname]
            us = cold_times(lambda: fn(0), flush, reps)
            us_stream = stream_times(fn, len(sets), max(40, 4 * len(sets)))
            if wl.dtype == "f32":
                t_c, bound_c = flops / (FFMA_TFLOPS * 1e12), "alu"
            else:
                t_c, bound_c = flops / (peaks["bf16_tflops"] * 1e12), "tensor"
            t_m = byts / (peaks["hbm_gbs"] * 1e9)
            tr = max(t_c, t_m)
            res[pname] = {"us": round(us, 3), "tflops": round(flops / (us * 1e-6) / 1e12, 2),
                          "roofline_us": round(tr * 1e6, 3), "bound": bound_c if t_c >= t_m else "hbm",
                          "roofline_frac": round(tr / (us * 1e-6), 4),
                          "us_stream": round(us_stream, 3), "roofline_frac_stream": round(tr / (us_stream * 1e-6), 4)}
        m.sync_status()
        out[name] = {"shape": "C=%d K=%d bs=%d density=%s N=%d %s fa=%d nnz=%d%s" % (
            wl.C, wl.K, wl.bs, wl.density, wl.N, wl.dtype, wl.feature_axis, m.nnz,
            (" steps=%d group=%d" % (wl.steps, wl.group)) if wl.steps > 1 else ""), "passes": res}
        m.close()
        del sets
        if wl.steps > 1:
            out[name]["layer"] = recurrent_layer(wl, dev, flush, reps)
    out["_launch_floor_us"] = launch_floor(dev, flush, reps)
    del flush
    out["_timing"] = ("us: each pass alone between CUDA events on the launching stream, median of %d, after a "
                      "256 MB read-only sweep that evicts L2, queued behind a device sleep so host enqueue "
                      "time is not counted; us_stream: the pass launched back to back on one stream over "
                      "rotating input/output sets larger than twice the L2 (cold inputs), device time per "
                      "launch; _launch_floor_us: an empty 192-CTA kernel timed both ways (the alone figure "
                      "is part of every pass's us); peaks: %s" % (
                          reps, "tensor = MEASURED_PEAKS bf16_tflops (fp16 the same rate), hbm = hbm_gbs, "
                          "alu = derived fp32 FFMA peak %.1f TFLOP/s" % FFMA_TFLOPS))
    return out


def run_single_pass(args):
    """--pass CONFIG:PASS: one pass of one benchmark configuration, launched warmup + steps times
    (cold: an L2-evicting sweep before each), median microseconds as one JSON line.  For kernel
    profiles of any configuration (ncu -k ... python bench.py --pass h8192_b16_p10:fprop)."""
    name, pname = args.single_pass.split(":")
    dev = torch.device("cuda", 0)
    peaks, _ = load_peaks()
    wl = wk.CONFIGS[name]
    from block_sparse_matrix_gb300 import bsmm
    inp = wk.make_inputs(wl, steps=min(wl.steps, wl.group) if wl.steps > 1 else None)
    m = bsmm.BlocksparseMatMul(inp.layout, block_size=wl.bs, feature_axis=wl.feature_axis)
    x, w, dy = inp.x.to(dev), inp.w.to(dev), inp.dy.to(dev)
    y = torch.empty(m.o_shape(wl.N), dtype=x.dtype, device=dev)
    dx = torch.empty(m.i_shape(wl.N), dtype=x.dtype, device=dev)
    dw = torch.zeros(m.w_shape, dtype=torch.float32, device=dev)
    calls = {"fprop": lambda: m.fprop(x, w, y), "bprop": lambda: m.bprop(dy, w, dx), "updat": lambda: m.updat(x, dy, dw)}
    if wl.steps > 1:
        xs = [a.to(dev) for a in inp.xs]
        dys = [a.to(dev) for a in inp.dys]
        calls["updat_grouped_g%d" % wl.group] = lambda: m.updat_grouped(xs, dys, dw=dw, accumulate=True)
    fn = calls[pname]
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    for _ in range(max(1, args.warmup)):
        fn()
    us = cold_times(fn, flush, args.steps)
    m.sync_status()
    print(json.dumps({"pass": args.single_pass, "us": round(us, 3), "steps": args.steps, "nnz": m.nnz}), flush=True)


# ---- CPU oracle --------------------------------------------------------------------------

def oracle_sample(wl, inp, n_rows, n_blocks, nthreads, N):
    """One bounded sample of the step on the oracle: n_rows minibatch rows of fprop
    and bprop and n_blocks blocks of updat at minibatch N.  Returns (eff. flops, s)."""
    from oracle import oracle as o
    L, bs = inp.layout, wl.bs
    x = inp.x[:N].double().numpy()
    dy = inp.dy[:N].double().numpy()
    w = inp.w.double().numpy()
    t0 = time.perf_counter()
    o.fprop(L, bs, x, w, 1, rows=(0, n_rows), nthreads=nthreads)
    o.bprop(L, bs, dy, w, 1, rows=(0, n_rows), nthreads=nthreads)
    o.updat(L, bs, x, dy, 1, blocks=(0, n_blocks), nthreads=nthreads)
    dt = time.perf_counter() - t0
    nnz = inp.nnz
    flops = 2 * n_rows * nnz * bs * bs * 2 + 2 * N * n_blocks * bs * bs
    return flops, dt


def run_cpu_baseline(wl, inp, Ns, budget_s=10.0):
    from oracle import oracle as o
    o.build()
    nthreads = len(os.sched_getaffinity(0))
    # calibrate on one row / a few blocks, then size the sample to the budget
    f1, t1 = oracle_sample(wl, inp, nthreads, 64, nthreads, 1024)
    scale = max(1, int(budget_s / max(t1, 1e-3)))
    rows = min(1024, nthreads * scale)
    blocks = min(inp.nnz, 64 * scale)
    # repeat the sample until about three quarters of the budget is spent (at most 8 times)
    f = t = 0.0
    reps = 0
    while reps < 8 and (reps == 0 or t < 0.75 * budget_s):
        fi, ti = oracle_sample(wl, inp, rows, blocks, nthreads, 1024)
        f, t, reps = f + fi, t + ti, reps + 1
    return {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": "float64 dense-W oracle at N=1024: %d x (fprop and bprop of %d minibatch rows, updat of %d "
                      "blocks), %.1f s; effective FLOPs 2*rows*nnz*bs^2 per fwd/bwd + 2*N*bs^2 per block" %
                      (reps, rows, blocks, t)}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import oracle as o
    o.build()
    wl = wk.CONFIGS["h4096_b32_p50_n1024"]
    inp = wk.make_inputs(wl)
    nthreads = len(os.sched_getaffinity(0))
    rows, blocks = nthreads, 128
    for _ in range(args.warmup):
        oracle_sample(wl, inp, rows, blocks, nthreads, 1024)
    tot_f = tot_t = 0.0
    for _ in range(args.steps):
        f, t = oracle_sample(wl, inp, rows, blocks, nthreads, 1024)
        tot_f += f
        tot_t += t
    v = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * tot_t / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded normals)",
            "config": {"workload": WORKLOAD, "nnz": inp.nnz},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                             "sample": "per step: fprop+bprop of %d rows and updat of %d blocks at N=1024" %
                                       (rows, blocks)},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _time_launches(fn, steps, warmup):
    """Device microseconds per call of fn(i): chunks of launches queued behind a device sleep
    that covers their enqueueing, so the GPU never waits for the host inside a chunk."""
    for i in range(max(3, warmup)):
        fn(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(20):
        fn(i)
    host_s = (time.perf_counter() - t0) / 20
    torch.cuda.synchronize()
    chunk = 50
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(0, steps, chunk)]
    for c, c0 in enumerate(range(0, steps, chunk)):
        torch.cuda._sleep(int(host_s * 1.5 * chunk * 2.1e9) + 100000)
        ev[c][0].record()
        for i in range(c0, min(steps, c0 + chunk)):
            fn(i)
        ev[c][1].record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(e) for a, e in ev) * 1000 / steps


def run_norm(args):
    """The normalisations and projections around the step, each on its own.
    layer_norm (README "blocksparse.norms") on the step's activation shape, N = 1024 samples of
    C = 4096 bf16 features, in both layouts; 16 rotating input/output sets (256 MB > L2).  Bytes
    per launch = read x + write y + g, b; its gradient (with relu) reads x, y, dy and writes dx
    (+ g, dg, db); one launch there is the partial-sum kernel and the reduction kernel.
    l2_normalize (README "blocksparse.matmul", weight normalisation) of the step's float32 weight
    (hidden 4096, block 32, 50% dense) to bf16, and its gradient (bf16 dy -> float32 dw, dgain);
    8 rotating sets (> L2).  Bytes per launch: read w (+ dy) + write y (or dw) + gain (+ dgain).
    SparseProj gather and scatter between 4096 and 2048 bf16 features at N = 1024, both layouts.
    One JSON line."""
    from block_sparse_matrix_gb300 import bsmm
    dev = torch.device("cuda", 0)
    N, C, sets = 1024, 4096, 16
    peaks, peak_src = load_peaks()
    g = torch.randn(C, device=dev)
    b = torch.randn(C, device=dev)
    out = {}

    def entry(us, byts):
        gbs = byts / us / 1e3
        return {"us": round(us, 3), "gbs": round(gbs, 1), "bytes": byts,
                "roofline_frac": round(gbs / peaks["hbm_gbs"], 4)}

    for axis in (1, 0):
        shape = (N, C) if axis == 1 else (C, N)
        xs = [wk.normals(shape, 500 + i, 1.0, "bf16").to(dev) for i in range(sets)]
        ys = [torch.empty_like(x) for x in xs]
        us = _time_launches(lambda i: bsmm.layer_norm(xs[i % sets], g, b, axis=axis, y=ys[i % sets]),
                            args.steps, args.warmup)
        out["layer_norm_axis%d" % axis] = entry(us, 2 * N * C * 2 + 2 * C * 4)
        # gradient with relu: read x, y, dy, write dx (bf16), read g, write dg, db; the workspace of
        # per-CTA partial sums is written and read back on top (not counted)
        dys = [wk.normals(shape, 600 + i, 1.0, "bf16").to(dev) for i in range(sets)]
        dxs = [torch.empty_like(x) for x in xs]
        us = _time_launches(lambda i: bsmm.layer_norm_grad(xs[i % sets], g, dys[i % sets], y=ys[i % sets],
                                                           axis=axis, relu=True, dx=dxs[i % sets]),
                            args.steps, args.warmup)
        out["layer_norm_grad_axis%d" % axis] = entry(us, 4 * N * C * 2 + 3 * C * 4)
        del xs, ys, dys, dxs

    wl = wk.CONFIGS["h4096_b32_p50_n1024"]
    lay = wk.make_layout(wl.R, wl.S, wl.layout_kind, wl.density, wl.force_diag, 1000 * wl.seed_ns)
    m = bsmm.BlocksparseMatMul(lay, block_size=wl.bs, feature_axis=wl.feature_axis)
    wsets = 8
    ws = [wk.normals(m.w_shape, 700 + i, 0.02, "f32").to(dev) for i in range(wsets)]
    ys = [torch.empty(m.w_shape, dtype=torch.bfloat16, device=dev) for _ in range(wsets)]
    gain = torch.rand(m.K, device=dev) + 0.5
    us = _time_launches(lambda i: m.l2_normalize(ws[i % wsets], gain, y=ys[i % wsets]), args.steps, args.warmup)
    el = m.nnz * wl.bs * wl.bs
    out["l2_normalize"] = entry(us, el * (4 + 2) + m.K * 4)
    dws = [torch.empty(m.w_shape, dtype=torch.float32, device=dev) for _ in range(wsets)]
    dgain = torch.empty(m.K, device=dev)
    us = _time_launches(lambda i: m.l2_normalize_grad(ws[i % wsets], ys[i % wsets], gain, dw=dws[i % wsets],
                                                      dgain=dgain), args.steps, args.warmup)
    out["l2_normalize_grad"] = entry(us, el * (4 + 2 + 4) + 2 * m.K * 4)
    nnz = m.nnz
    m.close()
    del ws, ys, dws

    # SparseProj (README "blocksparse.matmul"): runs of 32 features every 64 of the 4096 hidden
    # features (nproj 2048), N = 1024 bf16 samples; bytes = read + write of the moved elements
    # (scatter writes every dense element).
    for axis in (1, 0):
        sp = bsmm.SparseProj(C, nproj=2048, proj_stride=64, block_size=32, feature_axis=axis)
        dense = (N, C) if axis == 1 else (C, N)
        sparse = (N, sp.nproj) if axis == 1 else (sp.nproj, N)
        xs = [wk.normals(dense, 800 + i, 1.0, "bf16").to(dev) for i in range(sets)]
        ss = [torch.empty(sparse, dtype=torch.bfloat16, device=dev) for _ in range(sets)]
        us = _time_launches(lambda i: sp.gather(xs[i % sets], out=ss[i % sets]), args.steps, args.warmup)
        out["sparse_proj_gather_axis%d" % axis] = entry(us, 2 * N * sp.nproj * 2)
        us = _time_launches(lambda i: sp.scatter(ss[i % sets], out=xs[i % sets]), args.steps, args.warmup)
        out["sparse_proj_scatter_axis%d" % axis] = entry(us, N * sp.nproj * 2 + N * C * 2)
        sp.close()
        del xs, ss
    print(json.dumps({"metric": "normalisation and projection GB/s (algorithmic bytes) on 1 GB300",
                      "unit": "GB/s",
                      "value": round(min(v["gbs"] for v in out.values()), 1), "dtype": "bf16",
                      "config": {"workload": "layer_norm and its gradient: N=1024 x C=4096 bf16, 16 rotating sets; "
                                             "l2_normalize: hidden 4096, block 32, 50%% dense, %d blocks, "
                                             "float32 w -> bf16, 8 rotating sets; SparseProj: N=1024 x "
                                             "4096 -> 2048 features (runs of 32 every 64), bf16, 16 rotating "
                                             "sets" % nnz},
                      "peak": peaks["hbm_gbs"], "peak_source": peak_src, "passes": out}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of CPU time for the oracle baseline sample (0 skips it)")
    ap.add_argument("--only", default="",
                    help="time a single pass (e.g. fprop_n1024) instead of the whole step; for kernel profiling")
    ap.add_argument("--config-reps", type=int, default=20,
                    help="timed launches per pass for the per-configuration table (0 skips it)")
    ap.add_argument("--pass", dest="single_pass", default="",
                    help="CONFIG:PASS -- time one pass of one configuration (e.g. h8192_b16_p10:fprop), for profiles")
    ap.add_argument("--norm", action="store_true",
                    help="time layer_norm, l2_normalize (and its gradient) and SparseProj instead of the step")
    args = ap.parse_args()
    if args.single_pass:
        run_single_pass(args)
    elif args.norm:
        run_norm(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
