#!/usr/bin/env python
"""Benchmark of the SAF hybrid causal attention layer on GB300.

One step = forward + backward of one 124M-shaped hybrid attention layer
(B=8, H=12 with 3 frozen heads, T=4096, d_h=64, bf16) through libsaf's C ABI:
the static pre-pass, the fused persistent forward, the backward pre-pass,
the dynamic-head backward, the frozen heads' dV and the dQ post-pass.

Printed (rank 0, one JSON line): useful TFLOP/s of the whole job (useful
FLOPs count 4 d T^2/2 per dynamic head and 2 d T^2/2 per frozen head in the
forward, 8 d T^2/2 and 2 d T^2/2 in the backward), tokens/s, the fraction of
the measured bf16 peak, the dominant kernel's roofline, an end-to-end figure
with host buffers, the float64 oracle's throughput on the host cores, the
SM clocks seen during the timed region, and secondary figures for the other
workloads (1B layer with alpha/rho gradients, the calibration reduction,
the static-ratio sweep).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl saf|reference]

With N > 1 the script runs under torchrun, one rank per GPU; every rank runs
its own replica of the layer (the layer has no cross-GPU exchange), so the
scaling is weak and the value sums all ranks' work over the slowest rank's
time.  ``--impl reference`` times the float64 CPU oracle on this host instead
(rank 0 only).
"""

from __future__ import annotations

import argparse
from dataclasses import replace
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dynamic_causal_attention_gb300.synthetic import (  # noqa: E402
    ATTN_CONFIGS, CALIB_CONFIG, PREFILL_SWEEP, attn_inputs, prefill_inputs,
    static_heads_for_ratio, sweep_config)

METRIC = "hybrid attn fwd+bwd useful TFLOP/s & tokens/s, % of GB300 bf16 tensor peak"
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------- work model
def useful_flops(cfg, grads=None):
    """(fwd, bwd) useful FLOPs of one layer step."""
    grads = cfg.want_param_grads if grads is None else grads
    u = cfg.d_h * cfg.T * cfg.T / 2.0
    hs = len(cfg.static_heads)
    hd = cfg.H - hs
    fwd = cfg.B * (4 * u * hd + 2 * u * hs)
    bwd = cfg.B * (8 * u * hd + (4 if grads else 2) * u * hs)
    return fwd, bwd


def kernel_flops(cfg, name, grads=None):
    """Useful FLOPs one launch of a kernel performs (for the roofline)."""
    grads = cfg.want_param_grads if grads is None else grads
    u = cfg.d_h * cfg.T * cfg.T / 2.0
    hs = len(cfg.static_heads)
    hd = cfg.H - hs
    return {
        "hybrid_fwd": cfg.B * (4 * u * hd + 2 * u * hs),
        "bwd_dynamic": cfg.B * 8 * u * hd,
        "static_dv": cfg.B * 2 * u * hs,
        "param_grad": cfg.B * 2 * u * hs if grads else 0.0,
    }.get(name)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


def bf16_peak(peaks, region_s):
    """The bf16 denominator for a kernel timed inside a region of region_s
    seconds: the burst figure (a GEMM timed alone) for regions under a
    second, the sustained one (a seconds-long GEMM loop under the power cap)
    for longer ones.  Returns (TFLOP/s, description)."""
    if region_s < 1.0:
        return peaks["bf16_tflops"], (f"{peaks['source']} burst bf16 (timed region "
                                      f"{region_s:.3f} s < 1 s)")
    return peaks["bf16_tflops_sustained"], (f"{peaks['source']} sustained bf16 (timed region "
                                            f"{region_s:.1f} s)")


def roofline_of(cfg, kernels, region_s, peaks, sm_mhz=None):
    """The roofline object of the dominant kernel of a traced step loop."""
    dom = max(kernels, key=lambda n: kernels[n]["ms_total"]) if kernels else None
    if not dom or not kernel_flops(cfg, dom):
        return None
    avg_ms = kernels[dom]["ms_total"] / kernels[dom]["launches"]
    ach = kernel_flops(cfg, dom) / (avg_ms / 1e3) / 1e12
    peak, kind = bf16_peak(peaks, region_s)
    return {"kernel": dom, "bound": "tensor", "achieved": round(ach, 1), "peak": peak,
            "unit": "TFLOP/s", "frac": round(ach / peak, 4), "peak_kind": kind,
            "frac_of_burst_peak": round(ach / peaks["bf16_tflops"], 4),
            "frac_of_sustained_peak": round(ach / peaks["bf16_tflops_sustained"], 4),
            "sm_mhz_median": sm_mhz, "timed_region_s": round(region_s, 4),
            "flop_per_launch": kernel_flops(cfg, dom),
            "traffic": ncu_traffic(dom, cfg.name)}


# Source files that define each timed kernel: a recorded DRAM-traffic figure
# counts only while these are unchanged.
KERNEL_SOURCES = {
    "hybrid_fwd": ("attn_fwd.cu", "attn_common.cuh", "ptx.cuh", "attn_kernels.h"),
    "static_dv": ("attn_fwd.cu", "attn_common.cuh", "ptx.cuh", "attn_kernels.h"),
    "bwd_dynamic": ("attn_bwd.cu", "attn_common.cuh", "ptx.cuh", "attn_kernels.h"),
    "param_grad": ("attn_bwd.cu", "attn_common.cuh", "ptx.cuh", "attn_kernels.h"),
}


_COMMENT_RE = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def source_hash(kernel):
    """Hash of the kernel's source files with comments and blank space
    removed, so that a comment-only edit keeps a recorded figure valid."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dynamic_causal_attention_gb300", "csrc")
    for f in KERNEL_SOURCES.get(kernel, ()):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            code = _COMMENT_RE.sub("", fh.read())
        h.update(f.encode())
        h.update("\n".join(ln.strip() for ln in code.splitlines() if ln.strip()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch from the committed ncu record
    (profiles/dram_traffic.txt: workload, kernel, bytes, source hash), if it
    was taken on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 4 and not line.startswith("#") and parts[0] == workload \
                        and parts[1] == kernel and parts[3] == source_hash(kernel):
                    return float(parts[2])
    except OSError:
        pass
    return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- dist
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The largest x over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(local_ms, steps, flop_per_step, world):
    """Whole-job useful TFLOP/s of `world` replicas that each ran `steps`
    steps: every rank's work over the slowest rank's time.  Returns
    (TFLOP/s, ms per step of the slowest rank)."""
    ms = max_over_ranks(local_ms, world)
    per = ms / steps
    return world * flop_per_step / (per / 1e3) / 1e12, per


# ---------------------------------------------------------------- saf arm
class LayerRun:
    """Device-resident inputs and outputs of one layer workload."""

    def __init__(self, cfg, grads=None):
        import torch
        from dynamic_causal_attention_gb300 import api
        self.cfg = cfg
        self.grads = cfg.want_param_grads if grads is None else grads
        inp = attn_inputs(cfg)
        self.host = inp
        dev = torch.device("cuda")
        bf = torch.bfloat16
        self.q, self.k, self.v, self.do = (torch.from_numpy(inp[n]).to(dev, bf)
                                           for n in ("Q", "K", "V", "dO"))
        self.alpha = torch.from_numpy(inp["alpha"]).to(dev)
        self.rho = torch.from_numpy(inp["rho"]).to(dev)
        self.layer = api.HybridAttention(cfg.B, cfg.H, cfg.T, cfg.d_h, cfg.head_is_static,
                                         want_param_grads=self.grads)
        shp = (cfg.B, cfg.H, cfg.T, cfg.d_h)
        self.out = torch.empty(shp, dtype=bf, device=dev)
        self.lse = torch.empty(shp[:3], dtype=torch.float32, device=dev)
        self.gq, self.gk, self.gv = (torch.empty(shp, dtype=bf, device=dev) for _ in range(3))
        self.ga = self.gr = None
        if self.grads:
            self.ga = torch.empty((cfg.H, cfg.T), dtype=torch.float32, device=dev)
            self.gr = torch.empty((cfg.H, cfg.T), dtype=torch.float32, device=dev)
        self.launches = 0

    def step(self, q=None, k=None, v=None, do=None, alpha=None, rho=None, grads=None):
        from dynamic_causal_attention_gb300 import _binding as B
        q = self.q if q is None else q
        k = self.k if k is None else k
        v = self.v if v is None else v
        do = self.do if do is None else do
        alpha = self.alpha if alpha is None else alpha
        rho = self.rho if rho is None else rho
        self.layer.forward(q, k, v, alpha, rho, out=self.out, lse=self.lse)
        n = B.saf_last_launch_count()
        if grads is None:
            grads = (self.gq, self.gk, self.gv, self.ga, self.gr)
        self.layer.backward(q, k, v, self.out, self.lse, do, alpha, rho,
                            want_param_grads=self.grads, grads=grads)
        self.launches += n + B.saf_last_launch_count()

    def input_bytes(self):
        return sum(t.numel() * t.element_size() for t in (self.q, self.k, self.v, self.do))


def time_steps(run, steps, warmup, world, trace=False, sampler=None, graph=False):
    """Time `steps` steps on the device (CUDA events on the launching stream,
    synchronised on both sides).  With `graph`, one step (the same C-ABI
    calls on the same resident buffers) is captured once in a CUDA graph
    after the warm-up and the timed loop replays it, as a training loop that
    keeps its buffers would; run.launches then counts the captured step's
    launches once per replay."""
    import torch
    from dynamic_causal_attention_gb300 import _binding as B
    for _ in range(warmup):
        run.step()
    torch.cuda.synchronize()
    g = None
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            before = run.launches
            with torch.cuda.graph(g, stream=side):
                run.step()
            per_step = run.launches - before
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
    barrier(world)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if trace:
        B.saf_trace_enable(1)
    run.launches = 0
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    if g is not None:
        for _ in range(steps):
            g.replay()
        run.launches = per_step * steps
    else:
        for _ in range(steps):
            run.step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    clocks = sampler.stop() if sampler else None
    kernels = {}
    if trace:
        for i in range(B.saf_trace_count()):
            st, name, kms = B.saf_trace_get(i)
            if st == 0:
                k = kernels.setdefault(name, {"launches": 0, "ms_total": 0.0})
                k["launches"] += 1
                k["ms_total"] += kms
        B.saf_trace_enable(0)
    return ms, clocks, kernels


def e2e_steps(run, steps):
    """Whole steps through the public API with host buffers: every step copies
    its inputs from pinned host memory to the device, runs forward and
    backward, and copies its results (the gradients) back to pinned host
    memory.  The copies run on two copy streams against double-buffered
    device inputs and outputs, so step t+1's inputs travel and step t's
    results return while step t computes, as a training loop would overlap
    them; every step's copies fall inside the timed region."""
    import torch
    dev_in = [[run.q, run.k, run.v, run.do, run.alpha, run.rho]]
    dev_in.append([torch.empty_like(t) for t in dev_in[0]])
    outs0 = [run.gq, run.gk, run.gv, run.ga, run.gr]
    dev_out = [outs0, [None if t is None else torch.empty_like(t) for t in outs0]]
    host_in = [t.to("cpu").pin_memory() for t in dev_in[0]]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs0 if t is not None]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    cs = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    def run_steps(n):
        for t in range(n):
            one(t)

    def one(t):
        s = t % 2
        up.wait_event(in_free[s])            # step t-2 has finished reading set s
        with torch.cuda.stream(up):
            for d, h in zip(dev_in[s], host_in):
                d.copy_(h, non_blocking=True)
        ready[s].record(up)
        cs.wait_event(ready[s])
        cs.wait_event(out_free[s])           # step t-2's results have left set s
        q, k, v, do, alpha, rho = dev_in[s]
        run.step(q, k, v, do, alpha, rho, grads=tuple(dev_out[s]))
        in_free[s].record(cs)
        done[s].record(cs)
        down.wait_event(done[s])
        with torch.cuda.stream(down):
            for h, d in zip(host_out, [x for x in dev_out[s] if x is not None]):
                h.copy_(d, non_blocking=True)
        out_free[s].record(down)

    run_steps(2)                      # warm-up: streams and pinned transfers
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run_steps(steps)
    torch.cuda.synchronize()
    return (time.perf_counter() - t0) * 1e3 / steps, h2d, d2h


def calib_secondary(peaks, n_samples=None):
    """The calibration reduction at its full size: 64 sequences x 144 heads x
    T = 1024 fp32 probabilities (38.65 GB, generated on the device outside
    timing), accumulated in 12 per-layer calls, then finalized.  n_samples
    replaces the 64 sequences (a smaller case for profiling)."""
    import torch
    from dynamic_causal_attention_gb300 import api
    from dynamic_causal_attention_gb300.synthetic import calib_probabilities
    c = CALIB_CONFIG
    if n_samples:
        c = replace(c, N=int(n_samples))
    A = calib_probabilities(c.N, c.num_heads, c.T, d_h=c.d_h, device="cuda")
    layers = [A[:, l * c.H:(l + 1) * c.H].contiguous() for l in range(c.L)]
    del A
    torch.cuda.empty_cache()
    cal = api.Calibration(c.num_heads, c.T)
    k = api.num_select(c.r, c.num_heads)
    A_hat = torch.empty((c.num_heads, c.T, c.T), dtype=torch.float32, device="cuda")
    s_var = torch.empty(c.num_heads, dtype=torch.float32, device="cuda")
    sel = torch.empty(k, dtype=torch.int32, device="cuda")
    from dynamic_causal_attention_gb300 import _binding as B

    def once():
        cal.reset()
        for l, a in enumerate(layers):
            cal.accumulate(a, head_begin=l * c.H)
        st = B.saf_calib_finalize(cal.handle, k, A_hat.data_ptr(), s_var.data_ptr(),
                                  sel.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0

    for _ in range(2):
        once()
    torch.cuda.synchronize()
    B.saf_trace_enable(1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    e0.record()
    for _ in range(reps):
        once()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    acc_ms = 0.0
    n_acc = 0
    for i in range(B.saf_trace_count()):
        st, name, kms = B.saf_trace_get(i)
        if name == "calib_accumulate":
            acc_ms += kms
            n_acc += 1
    B.saf_trace_enable(0)
    tri = c.T * (c.T + 1) // 2
    read_bytes = c.N * c.num_heads * tri * 4
    state_bytes = 2 * c.num_heads * tri * 4
    alg_bytes = read_bytes + c.num_heads * c.T * c.T * 4
    acc_gbs = (read_bytes + state_bytes) / (acc_ms / n_acc * c.L / 1e3) / 1e9 if n_acc else None
    out = {
        "workload": f"calibration N={c.N}, {c.num_heads} heads, T={c.T}, k={k} (12 per-layer "
                    "accumulate calls + finalize)",
        "ms": round(ms, 3),
        "algorithmic_bytes": alg_bytes,
        "GB_per_s": round(alg_bytes / (ms / 1e3) / 1e9, 1),
        "frac_of_hbm": round(alg_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 3),
        "accumulate_GB_per_s": round(acc_gbs, 1) if acc_gbs else None,
        "accumulate_frac_of_hbm": round(acc_gbs / peaks["hbm_gbs"], 3) if acc_gbs else None,
        "selected_first": [int(x) for x in sel[:8].cpu()],
    }
    cal.close()

    # forward-KL selector: the same samples, with the entropy sums tracked
    cal_kl = api.Calibration(c.num_heads, c.T, track_kl=True)

    def once_kl():
        cal_kl.reset()
        for l, a in enumerate(layers):
            cal_kl.accumulate(a, head_begin=l * c.H)
        return cal_kl.finalize_kl(k)

    once_kl()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(3):
        s_kl, sel_kl = once_kl()
    e1.record()
    torch.cuda.synchronize()
    kl_ms = e0.elapsed_time(e1) / 3
    out["kl_selector"] = {
        "ms": round(kl_ms, 3),
        "GB_per_s": round(read_bytes / (kl_ms / 1e3) / 1e9, 1),
        "frac_of_hbm": round(read_bytes / (kl_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 3),
        "note": "accumulate with the entropy sums + finalize_kl; GB/s counts the samples read",
        "selected_first": [int(x) for x in sel_kl[:8].cpu()],
    }
    cal_kl.close()

    # compact fit of alpha/rho to the mean pattern, candidates in variance order
    order = torch.argsort(s_var).to(torch.int32)
    api.fit_compact(A_hat, order, k)
    torch.cuda.synchronize()
    e0.record()
    alpha, rho, kl, fsel = api.fit_compact(A_hat, order, k)
    e1.record()
    torch.cuda.synchronize()
    fit_ms = e0.elapsed_time(e1)
    kl_h = kl.cpu()
    out["compact_fit"] = {
        "ms": round(fit_ms, 3),
        "workload": f"alpha/rho fit, 400 Adam steps per candidate, T={c.T}, "
                    f"{c.num_heads} candidates in variance order, k={k}, KL gate 0.2 nat",
        "selected": int(fsel.numel()),
        "kl_of_first_candidates": [round(float(x), 4) for x in kl_h[:8]],
    }
    del layers, A_hat
    torch.cuda.empty_cache()
    # the reduction's own figures last in the block, so that the end of the
    # output line (the calibration block, then the 1B layer's) holds them
    for name in ("ms", "algorithmic_bytes", "GB_per_s", "frac_of_hbm", "accumulate_GB_per_s",
                 "accumulate_frac_of_hbm"):
        out[name] = out.pop(name)
    return out


def sharp_secondary(peaks):
    """The sharp-mean pattern: calibration fed logits (N=16 sequences x 144
    heads x T = 1024, generated on the device outside timing), then the
    causal softmax of each row of their mean."""
    import torch
    from dynamic_causal_attention_gb300 import api
    from dynamic_causal_attention_gb300.synthetic import calib_probabilities
    c = CALIB_CONFIG
    N = 16
    X = calib_probabilities(N, c.num_heads, c.T, d_h=c.d_h, device="cuda", want_logits=True)
    layers = [X[:, l * c.H:(l + 1) * c.H].contiguous() for l in range(c.L)]
    del X
    torch.cuda.empty_cache()
    cal = api.Calibration(c.num_heads, c.T)

    def once():
        cal.reset()
        for l, a in enumerate(layers):
            cal.accumulate(a, head_begin=l * c.H)
        return cal.finalize_sharp()

    once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        pat = once()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 3
    tri = c.T * (c.T + 1) // 2
    alg = N * c.num_heads * tri * 4 + c.num_heads * c.T * c.T * 4
    out = {"workload": f"sharp mean: N={N} logit samples, {c.num_heads} heads, T={c.T} "
                       "(12 per-layer accumulate calls + finalize_sharp)",
           "ms": round(ms, 3),
           "GB_per_s": round(alg / (ms / 1e3) / 1e9, 1),
           "frac_of_hbm": round(alg / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 3),
           "row_sum_max_err": float((pat.sum(-1) - 1).abs().max())}
    cal.close()
    del layers, pat
    torch.cuda.empty_cache()
    return out


def gqa_secondary(peaks, steps=20, warmup=3):
    """The 124M-shaped layer with grouped K/V: 12 query heads over 4 K/V heads
    (3 frozen query heads), forward + backward through the C ABI."""
    import torch
    from dynamic_causal_attention_gb300 import api
    cfg = ATTN_CONFIGS["124m"]
    B, H, T, d, Hkv = cfg.B, cfg.H, cfg.T, cfg.d_h, 4
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    bf = torch.bfloat16
    rnd = lambda *shp: torch.randn(shp, generator=g, device="cuda").to(bf)
    q, do = rnd(B, H, T, d), rnd(B, H, T, d)
    k, v = rnd(B, Hkv, T, d), rnd(B, Hkv, T, d)
    inp = attn_inputs(cfg, B=1, H=H, T=T, d_h=8)  # alpha, rho only
    alpha = torch.from_numpy(inp["alpha"]).cuda()
    rho = torch.from_numpy(inp["rho"]).cuda()
    layer = api.HybridAttention(B, H, T, d, cfg.head_is_static, H_kv=Hkv)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), None, None)

    def step():
        layer.forward(q, k, v, alpha, rho, out=out, lse=lse)
        layer.backward(q, k, v, out, lse, do, alpha, rho, grads=grads)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    st, site = layer.device_status()
    per = e0.elapsed_time(e1) / steps
    f, b = useful_flops(cfg)
    tf = (f + b) / (per / 1e3) / 1e12
    res = {"workload": f"124m with grouped K/V: B={B} H={H} H_kv={Hkv} T={T} d_h={d} "
                       f"static={list(cfg.static_heads)}",
           "ms_per_step": round(per, 4), "TFLOP_per_s": round(tf, 1),
           "frac_of_bf16_peak": round(tf / bf16_peak(peaks, per * steps / 1e3)[0], 3),
           "device_status": int(st)}
    del layer, q, k, v, do, out, lse, grads
    torch.cuda.empty_cache()
    return res


def layer_secondary(cfg, steps, warmup, peaks, roofline=False, cpu_s=0.0):
    run = LayerRun(cfg)
    ms, _, _ = time_steps(run, steps, warmup, 1, trace=False, graph=True)
    ms_traced, _, kernels = time_steps(run, steps, 3, 1, trace=True)
    f, b = useful_flops(cfg)
    per = ms / steps
    tf = (f + b) / (per / 1e3) / 1e12
    res = {"workload": f"{cfg.name}: B={cfg.B} H={cfg.H} T={cfg.T} d_h={cfg.d_h} "
                       f"static={list(cfg.static_heads)} grads={cfg.want_param_grads}",
           "launch": "one step captured in a CUDA graph, replayed",
           "ms_per_step": round(per, 4), "TFLOP_per_s": round(tf, 1),
           "tokens_per_s": round(cfg.B * cfg.T / (per / 1e3)),
           "frac_of_bf16_peak": round(tf / bf16_peak(peaks, ms / 1e3)[0], 3),
           "kernels_ms_per_step": {k: round(v["ms_total"] / steps, 4) for k, v in kernels.items()}}
    if roofline:
        res["roofline"] = roofline_of(cfg, kernels, ms_traced / 1e3, peaks)
    del run
    if cpu_s > 0:
        res["cpu_baseline"] = cpu_baseline(cfg, budget_s=cpu_s)
    return res


def prefill_secondary(peaks):
    """Forward-only causal prefill: the 124M head shape at batch 64 over
    T = 512..16K with 0%, 25% and 50% of heads frozen, and batch 1 at
    T = 4096.  Reports ms per forward and the speed ratio against 0%."""
    import torch
    from dynamic_causal_attention_gb300 import api
    P = PREFILL_SWEEP
    H, d = P["H"], P["d_h"]

    def time_fwd(B, T, r, reps):
        mask = np.zeros(H, dtype=np.uint8)
        for h in static_heads_for_ratio(H, r):
            mask[h] = 1
        q, k, v, alpha, rho = prefill_inputs(B, H, T, d)
        layer = api.HybridAttention(B, H, T, d, mask)
        out = torch.empty_like(v)
        lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
        for _ in range(2):
            layer.forward(q, k, v, alpha, rho, out=out, lse=lse)
        torch.cuda.synchronize()
        # one forward (the frozen-head pre-pass and the fused kernel) captured
        # in a CUDA graph and replayed
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                layer.forward(q, k, v, alpha, rho, out=out, lse=lse)
        torch.cuda.synchronize()
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        u = d * T * T / 2.0
        hs = int(mask.sum())
        flop = B * (4 * u * (H - hs) + 2 * u * hs)
        del q, k, v, out, lse, layer, g
        torch.cuda.empty_cache()
        return ms, flop / (ms / 1e3) / 1e12

    res = {}
    for T in P["T"]:
        row = {}
        base = None
        for r in P["ratios"]:
            ms, tf = time_fwd(P["B"], T, r, 5 if T >= 8192 else 10)
            base = ms if r == 0.0 else base
            row[f"r={r:g}"] = {"ms": round(ms, 4), "TFLOP_per_s": round(tf, 1),
                               "speedup_vs_r0": round(base / ms, 3)}
        res[f"T={T}"] = row
    b1 = {}
    base = None
    for r in P["ratios"]:
        ms, tf = time_fwd(1, P["batch1_T"], r, 50)
        base = ms if r == 0.0 else base
        b1[f"r={r:g}"] = {"ms": round(ms, 4), "speedup_vs_r0": round(base / ms, 3)}
    res[f"batch1_T={P['batch1_T']}"] = b1
    return {"workload": f"causal prefill, forward only, B={P['B']} H={H} d_h={d}",
            "launch": "one forward captured in a CUDA graph, replayed", "sweep": res}


# ---------------------------------------------------------------- oracle leg
def oracle_sample(inp, cfg, s, rows_per_block=1024):
    """One bounded sample of the layer for the float64 oracle: query rows
    [i0, i0 + rows) of head (s mod H) of sequence 0, forward and backward
    (the rows' share of every gradient).  Returns its useful FLOPs."""
    import oracle
    T, d = cfg.T, cfg.d_h
    h = s % cfg.H
    nblk = T // rows_per_block
    blk = (s // cfg.H) % nblk
    rows = np.arange(blk * rows_per_block, (blk + 1) * rows_per_block)
    keys = float(np.sum(rows + 1))          # causal (i, j) pairs in the block
    if h in cfg.static_heads:
        oracle.static_head_fwd_rows(inp["alpha"][h], inp["rho"][h], inp["V"][0, h], rows)
        oracle.static_head_bwd_rows(inp["alpha"][h], inp["rho"][h], inp["V"][0, h],
                                    inp["dO"][0, h], rows)
        return keys * d * (2 + 2)
    oracle.dynamic_head_fwd_rows(inp["Q"][0, h], inp["K"][0, h], inp["V"][0, h], rows)
    oracle.dynamic_head_bwd_rows(inp["Q"][0, h], inp["K"][0, h], inp["V"][0, h],
                                 inp["dO"][0, h], rows)
    return keys * d * (4 + 8)


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(cfg, budget_s=15.0):
    inp = attn_inputs(cfg, B=1)
    t0 = time.perf_counter()
    flops, s = 0.0, 0
    while time.perf_counter() - t0 < budget_s and s < 4 * cfg.H:
        flops += oracle_sample(inp, cfg, s)
        s += 1
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores(),
            "kind": "oracle",
            "sample": f"{s} blocks of 1024 query rows (heads cycled, sequence 0) of the "
                      f"{cfg.name} layer, fwd+bwd in float64 NumPy, {dt:.1f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = ATTN_CONFIGS["124m"]
    inp = attn_inputs(cfg, B=1)
    # about 0.4 s per 1024-row block on a few host cores: shrink the block so
    # that the whole run stays within a few minutes
    rows = 1024
    while rows > 128 and (args.steps + args.warmup) * 0.4 * rows / 1024 > 150:
        rows //= 2
    for s in range(args.warmup):
        oracle_sample(inp, cfg, s, rows)
    t0 = time.perf_counter()
    flops = 0.0
    for s in range(args.steps):
        flops += oracle_sample(inp, cfg, args.warmup + s, rows)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"per step: {rows} query rows of one head (heads cycled, sequence 0) of the 124M "
              "layer, fwd+bwd, float64 NumPy oracle on the host cores")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "124M-shaped hybrid layer fwd+bwd (bounded row-block samples)",
                   "B": cfg.B, "H": cfg.H, "T": cfg.T, "d_h": cfg.d_h,
                   "static_heads": list(cfg.static_heads)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------- main arm
def sweep_secondary(peaks, args=None):
    sweep = {}
    for r in (0.0, 0.125, 0.25, 0.5, 1.0):
        s = layer_secondary(sweep_config(r), 20, 3, peaks)
        sweep[f"r={r:g}"] = {k: s[k] for k in ("ms_per_step", "TFLOP_per_s", "tokens_per_s",
                                              "frac_of_bf16_peak")}
    return sweep


SECONDARY = {
    "prefill": lambda peaks, args: prefill_secondary(peaks),
    "static_ratio_sweep_124m": lambda peaks, args: sweep_secondary(peaks),
    "gqa_124m": lambda peaks, args: gqa_secondary(peaks),
    "sharp_mean": lambda peaks, args: sharp_secondary(peaks),
    "calibration": lambda peaks, args: calib_secondary(peaks, args.calib_samples),
    "1b": lambda peaks, args: layer_secondary(ATTN_CONFIGS["1b"], 30, 3, peaks, roofline=True,
                                              cpu_s=0.0 if args.no_cpu else 8.0),
}


def run_only(args):
    """One secondary workload alone (for profiling it): prints its JSON."""
    import torch
    torch.cuda.set_device(0)
    peaks = load_peaks()
    print(json.dumps({args.only: SECONDARY[args.only](peaks, args)}))


def run_saf(args):
    import torch
    world, rank, local = dist_setup(args.gpus)
    peaks = load_peaks()
    cfg = ATTN_CONFIGS[args.workload]
    run = LayerRun(cfg)
    sampler = ClockSampler(local) if rank == 0 else None
    # The headline loop replays one step captured in a CUDA graph, without
    # the kernel trace (its two events per launch cost about 4% of a 124M
    # step); a second timed loop of the same K steps, eager and traced, gives
    # each kernel's time for the roofline.
    ms, clocks, _ = time_steps(run, args.steps, args.warmup, world, trace=False,
                               sampler=sampler, graph=True)
    f, b = useful_flops(cfg)
    value, per = job_throughput(ms, args.steps, f + b, world)
    launches = run.launches
    ms_traced, _, kernels = time_steps(run, args.steps, 3, world, trace=True)

    # dominant kernel of the traced loop, against the bf16 peak that fits
    # the length of its timed region (burst under a second)
    region_s = max_over_ranks(ms_traced, world) / 1e3
    roofline = roofline_of(cfg, kernels, region_s, peaks,
                           clocks.get("sm_mhz") if clocks else None)
    total = sum(k["ms_total"] for k in kernels.values()) or 1.0
    for k in kernels.values():
        k["share"] = round(k["ms_total"] / total, 4)
        k["ms_total"] = round(k["ms_total"], 3)
    peak, _ = bf16_peak(peaks, region_s)

    e2e = None
    if rank == 0:
        e_ms, h2d, d2h = e2e_steps(run, max(5, min(args.steps, 50)))
        e2e = {"value": round(world * (f + b) / (e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e_ms, 3),
               "copies": "every step's H2D inputs and D2H gradients, on two copy streams "
                         "overlapping the compute of the neighbouring steps",
               "api": "dynamic_causal_attention_gb300.api.HybridAttention (C ABI)"}
    in_bytes = run.input_bytes()
    del run
    torch.cuda.empty_cache()

    # Secondary workloads, in the order they appear in the line: the long
    # prefill table first, the calibration reduction and the 1B layer last,
    # so that the end of the output holds them.
    secondary = {}
    if rank == 0 and not args.quick:
        secondary = {name: SECONDARY[name](peaks, args) for name in SECONDARY}
    barrier(world)
    if rank != 0:
        return
    cpu = None if (world > 1 or args.no_cpu) else cpu_baseline(cfg)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{cfg.name}-shaped hybrid attention layer fwd+bwd",
            "B": cfg.B, "H": cfg.H, "T": cfg.T, "d_h": cfg.d_h,
            "static_heads": list(cfg.static_heads), "param_grads": cfg.want_param_grads,
            "useful_flop_per_step": f + b, "tokens_per_step": cfg.B * cfg.T,
            "parallelism": f"replicas x{world}",
            "l2": f"no flush: the step's bf16 Q/K/V/dO inputs ({in_bytes / 2**20:.0f} MiB) "
                  f"exceed the 129 MB L2",
            "launch": "one step captured in a CUDA graph, replayed K times",
        },
        "tokens_per_s": round(world * cfg.B * cfg.T / (per / 1e3)),
        "frac_of_bf16_peak": round(value / world / peak, 4),
        "frac_of_bf16_peak_sustained": round(value / world / peaks["bf16_tflops_sustained"], 4),
        "ms_per_step_traced": round(max_over_ranks(ms_traced, world) / args.steps, 4),
        "peaks": peaks,
        "roofline": roofline,
        "kernels": kernels,
        "gpu_launches": launches,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "secondary": secondary,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["saf", "reference"], default="saf")
    ap.add_argument("--workload", default="124m", choices=["124m", "1b"])
    ap.add_argument("--quick", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline")
    ap.add_argument("--calib-samples", type=int, default=None,
                    help="sequences of the calibration workload (default 64; fewer to profile)")
    ap.add_argument("--only", choices=sorted(SECONDARY),
                    help="run one secondary workload alone and print its figures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_saf(args)


if __name__ == "__main__":
    main()
