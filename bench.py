#!/usr/bin/env python
"""Sparse attention forward throughput: TFLOP/s over useful (allowed) pairs.

FLOPs = 4 * D * P, P the number of allowed (query, key) pairs over all
batches and heads (one multiply-add of q.k and one of p*v per pair and
dimension).  Default workload: bf16 B1 H16 N131072 D128, window 512/512,
128 uniform-random global tokens (the long-sequence case).  Inputs are
seeded synthetic iid N(0, 1) tensors, larger than L2; the timed region holds
only the library call (inputs resident in HBM).  The "e2e" figure times the
host-memory entry point (lg_attn_fwd_host: q/k/v in pinned host memory copied
in and out/lse copied back by the library, overlapped with the kernels per
group of heads) inside the timed region; ETC and fp32 copy around the device
call instead.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Under torchrun each rank runs one replica of the workload on its own GPU
(no data exchange); the time is the max over ranks and the value the work of
all ranks over that time.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import os

# The CPU oracle runs one single-threaded process per host core (a spawned
# pool); set before numpy loads its BLAS, so every worker inherits it.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_long_sequence_window_gb300 import workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
E2E_GROUPS = 16         # head groups of the host-memory entry point (copies overlap kernels)
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def useful_pairs(lg, w: workloads.Workload) -> int:
    if w.is_longnet:
        return w.B * sum(lg.longnet_count_pairs(w.N, w.seg_w, w.seg_r, w.causal, h) for h in range(w.H))
    if w.is_etc:
        return w.B * w.H * lg.etc_count_pairs(w.N, w.etc_G, w.radius)
    g = workloads.global_positions(w)
    per_head = {}
    total = 0
    for d in w.dilations():
        if d not in per_head:
            per_head[d] = lg.count_pairs(w.N, w.w_left, w.w_right, d, w.causal, g)
        total += per_head[d]
    return w.B * total


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                return json.load(f), "measured"
        except Exception:
            pass
    return {}, "fallback"


# ---------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 200 ms) taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.proc = None
        self.path = tempfile.mktemp(suffix=".csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if uuid:
            cmd[1:1] = ["-i", uuid]
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1])); mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------- inputs

def device_inputs(w, dev, torch):
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def rnd(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(dt)

    t = {n: rnd(w.B, w.H, w.N, w.D) for n in ("q", "k", "v")}
    if w.is_etc:
        for n in ("q_g", "k_g", "v_g"):
            t[n] = rnd(w.B, w.H, w.etc_G, w.D)
        t["g"] = None
    elif w.is_longnet:
        t["g"] = None
    else:
        g = workloads.global_positions(w)
        t["g"] = torch.from_numpy(g).to(dev) if g.size else None
    return t


def make_call(lg, w, t, torch):
    """Returns f() that runs one forward pass with preallocated outputs and workspace."""
    dev = t["q"].device
    if w.is_etc and w.name.startswith("etc_struct"):
        st = workloads.make_etc_structure(w)
        codes = {n: torch.from_numpy(st[n]).to(dev) for n in ("code_l2l", "code_l2g", "code_g2l", "code_g2g")}
        rel = st["rel_k"].to(dev)
        B, H, L, D, G = w.B, w.H, w.N, w.D, w.etc_G
        out_l, out_g = torch.empty_like(t["q"]), torch.empty_like(t["q_g"])
        lse_l = torch.empty(B, H, L, device=dev); lse_g = torch.empty(B, H, G, device=dev)
        ws = torch.empty(lg.etc_struct_attn_fwd_workspace_size(B, H, L, G, D, w.radius, rel.shape[1]),
                         dtype=torch.uint8, device=dev)

        def f():
            lg.etc_struct_attn_fwd(t["q"], t["k"], t["v"], t["q_g"], t["k_g"], t["v_g"], w.radius, rel, **codes,
                                   out_l=out_l, out_g=out_g, lse_l=lse_l, lse_g=lse_g, workspace=ws)
        t.update(codes)
        return f, (out_l, out_g, lse_l, lse_g), ws
    if w.is_longnet:
        out = torch.empty_like(t["q"])
        lse = torch.empty(w.B, w.H, w.N, device=dev)
        ws = torch.empty(lg.longnet_attn_fwd_workspace_size(w.B, w.H, w.N, w.D, w.seg_w, w.seg_r),
                         dtype=torch.uint8, device=dev)

        def f():
            lg.longnet_attn_fwd(t["q"], t["k"], t["v"], w.seg_w, w.seg_r, w.causal, out=out, lse=lse, workspace=ws)
        return f, (out, lse), ws
    if w.is_etc:
        B, H, L, D, G = w.B, w.H, w.N, w.D, w.etc_G
        out_l, out_g = torch.empty_like(t["q"]), torch.empty_like(t["q_g"])
        lse_l = torch.empty(B, H, L, device=dev); lse_g = torch.empty(B, H, G, device=dev)
        ws = torch.empty(lg.etc_attn_fwd_workspace_size(B, H, L, G, D, 1 if w.dtype == "bf16" else 0),
                         dtype=torch.uint8, device=dev)

        def f():
            lg.etc_attn_fwd(t["q"], t["k"], t["v"], t["q_g"], t["k_g"], t["v_g"], w.radius,
                            out_l=out_l, out_g=out_g, lse_l=lse_l, lse_g=lse_g, workspace=ws)
        outs = (out_l, out_g, lse_l, lse_g)
    else:
        out = torch.empty_like(t["q"])
        lse = torch.empty(w.B, w.H, w.N, device=dev)
        ng = 0 if t["g"] is None else t["g"].numel()
        ws = torch.empty(max(256, lg.attn_fwd_workspace_size(w.B, w.H, w.N, w.D, ng, 1 if w.dtype == "bf16" else 0)),
                         dtype=torch.uint8, device=dev)

        def f():
            lg.attn_fwd(t["q"], t["k"], t["v"], w.w_left, w.w_right, w.dilations(), w.causal, t["g"],
                        out=out, lse=lse, workspace=ws)
        outs = (out, lse)
    return f, outs, ws


def launches_per_call(w):
    if w.is_etc and w.name.startswith("etc_struct"):
        return 3  # code packing + q . a^K + attention
    if w.is_longnet:
        # per pattern: unit table + tensor-core kernel (+ gather for the packed layout); then the mix
        packed = sum(1 for a, r in zip(w.seg_w, w.seg_r) if not (r <= 8 and a % r == 0))
        return 2 * len(w.seg_w) + packed + 1
    if w.dtype == "f32":
        return 1  # one CUDA-core kernel (it also checks the global list)
    if w.is_etc:
        return 3  # unit table + tensor-core kernel + merge
    dil = [d for d in set(w.dilations()) if d != 1]
    groups = max(1, -(-len(dil) // 3))
    has_g = bool(w.global_positions) or w.n_random_global > 0
    # per dilation group: unit table + tensor-core kernel; globals: prep + merge
    return 2 * groups + (2 if has_g else 0)


# ---------------------------------------------------------------------- rank bookkeeping

def max_over_ranks(value: float, dist, device) -> float:
    """The maximum of `value` over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica, timed by the slowest rank."""
    return flops_per_step * steps * world / (max_ms / 1e3) / 1e12


# ---------------------------------------------------------------------- native arm

def time_steps(torch, f, steps, flush):
    """Per-step CUDA-event times (ms) on the current stream; L2 flushed between steps if asked.

    The flush writes a buffer of twice the L2 size and then reads another one
    of the same size: the write evicts every line the previous step left in
    L2, and the read writes those dirty lines back before the timed region, so
    a step starts with no input in L2 and no write-back of the flush data to
    pay for.
    """
    stream = torch.cuda.current_stream()
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if flush else None
    reader = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if flush else None
    times = []
    for _ in range(steps):
        if scratch is not None:
            scratch.zero_()
            reader.sum()
        a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
        a.record(stream); f(); b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def run_native(args, rank, world):
    import torch
    import sparse_long_sequence_window_gb300 as lg
    lg.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = workloads.PRESETS[args.workload]
    t = device_inputs(w, dev, torch)
    f, outs, ws = make_call(lg, w, t, torch)
    pairs = useful_pairs(lg, w)
    flops = 4.0 * w.D * pairs
    in_bytes = sum(x.numel() * x.element_size() for k, x in t.items() if x is not None)
    flush = in_bytes < 2 * L2_BYTES

    for _ in range(args.warmup):
        f()
    torch.cuda.synchronize()
    st = lg.query_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {lg.status_string(st)}")

    props = torch.cuda.get_device_properties(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(uuid)
    lg.profile_begin()
    step_ms = time_steps(torch, f, args.steps, flush)
    kernel_ms, kernel_launches = lg.profile_end()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(float(sum(step_ms)), dist, dev)
    value = job_throughput(flops, args.steps, world, total_ms)

    # ---- end to end through the public API: pinned host inputs -> device -> call -> host outputs
    e2e = None
    host = {k: (x.cpu().pin_memory() if x is not None else None) for k, x in t.items()}
    host_out = [o.cpu().pin_memory() for o in outs]
    e2e_steps = max(1, min(args.steps, 10))
    stream = torch.cuda.current_stream()
    h2d = sum(x.numel() * x.element_size() for x in host.values() if x is not None)
    d2h = sum(o.numel() * o.element_size() for o in host_out)
    e_times = []
    if not w.is_etc and not w.is_longnet and w.dtype == "bf16":
        # lg_attn_fwd_host: the library copies q/k/v in and out/lse back itself,
        # overlapping the copies of one group of heads with the kernels of another.
        g_host = host.pop("g", None)
        h2d = sum(x.numel() * x.element_size() for x in host.values())
        staging = (t["q"], t["k"], t["v"]) + tuple(outs)

        def e2e_call():
            if g_host is not None:
                t["g"].copy_(g_host, non_blocking=True)
            lg.attn_fwd_host(host["q"], host["k"], host["v"], w.w_left, w.w_right, w.dilations(), w.causal,
                             t["g"], out_h=host_out[0], lse_h=host_out[1], staging=staging, workspace=ws,
                             n_groups=E2E_GROUPS)
        if g_host is not None:
            h2d += g_host.numel() * g_host.element_size()
    else:
        def e2e_call():
            for k_, x in host.items():
                if x is not None:
                    t[k_].copy_(x, non_blocking=True)
            f()
            for ho, o in zip(host_out, outs):
                ho.copy_(o, non_blocking=True)
    e2e_call()
    torch.cuda.synchronize()
    for _ in range(e2e_steps):
        a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_call()
        b.record(stream)
        b.synchronize()
        e_times.append(a.elapsed_time(b))
    e_ms = max_over_ranks(float(sum(e_times)), dist, dev)
    e2e = {"value": job_throughput(flops, e2e_steps, world, e_ms), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}

    # ---- roofline of the dominant kernel (the tensor-core attention kernel does every useful FLOP)
    peaks, peak_kind = measured_peaks()
    if w.dtype == "bf16":
        peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS)) if peaks else FALLBACK_BF16_TFLOPS
        kernel_per_step = kernel_ms / max(1, args.steps)
        achieved = flops / (kernel_per_step / 1e3) / 1e12
        traffic = committed_traffic(w)
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 4), "traffic": traffic,
                    "peak_source": f"bf16_tflops of {peak_kind}", "kernel": "tc_attn_kernel",
                    "kernel_ms_per_launch": round(kernel_ms / max(1, kernel_launches), 4),
                    "launches": kernel_launches}
        # The kernel runs back to back for the whole timed region, under the power cap: the
        # cuBLAS figure measured the same way (seconds of back-to-back GEMMs) sits beside it.
        if peaks and "bf16_tflops_sustained" in peaks:
            sus = float(peaks["bf16_tflops_sustained"])
            roofline["peak_sustained"] = sus
            roofline["frac_sustained"] = round(achieved / sus, 4)
    else:
        roofline = None

    backward = None
    if not args.no_bwd:
        backward = bench_backward(lg, torch, w, t, outs, flush, args.bwd_steps, peaks, peak_kind)

    per_config = None
    if rank == 0 and world == 1 and not args.no_sweep:
        sweep.no_bwd = args.no_bwd
        per_config = sweep(lg, torch, dev)

    line = {
        "metric": "sparse attn fwd TFLOP/s (in-band pairs) & % bf16 tensor peak, N=512-128K",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic iid N(0,1), seeded",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "useful_pairs": pairs, "useful_flops_per_step": flops,
                   "l2": "flushed between steps (write, then read, 2x L2)" if flush else "inputs larger than L2",
                   "parallelism": f"replicas x{world}"},
        "pct_bf16_peak": round(100 * value / world / (roofline["peak"] if roofline else FALLBACK_BF16_TFLOPS), 2),
        "e2e": e2e,
        "gpu_launches": launches_per_call(w) * args.steps,
        "roofline": roofline,
        "backward": backward,
        "clocks": clk,
        "step_ms_median": round(statistics.median(step_ms), 5),
    }
    if per_config:
        line["per_config"] = per_config
        line["linear_in_n_slope"] = linear_in_n_slope(per_config)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_seconds)
    if dist:
        dist.destroy_process_group()
    return line


def bench_backward(lg, torch, w, t, outs, flush, steps, peaks, peak_kind):
    """The backward pass of the same workload (lg_attn_bwd / lg_etc_attn_bwd) after one forward.

    Useful FLOPs: 8 * D per allowed pair (the contractions dP = dO V^T, dV =
    P^T dO, dK = dS^T Q, dQ = dS K; the recomputed S = Q K^T is not counted).
    The time is the whole library call (prep, tensor-core kernels, reduce),
    CUDA events on the current stream, L2 flushed between steps when the
    inputs fit in it.
    """
    if w.dtype != "bf16" or w.is_longnet or w.name.startswith("etc_struct"):   # no backward for these
        return None
    gen = torch.Generator(device=t["q"].device)
    gen.manual_seed(w.seed + 7919)
    dout = torch.randn(t["q"].shape, generator=gen, device=t["q"].device, dtype=torch.float32).to(torch.bfloat16)
    pairs = useful_pairs(lg, w)
    flops = 8.0 * w.D * pairs
    if w.is_etc:
        out_l, out_g, lse_l, lse_g = outs
        dout_g = torch.randn(t["q_g"].shape, generator=gen, device=t["q"].device, dtype=torch.float32).to(torch.bfloat16)
        ws = torch.empty(lg.etc_attn_bwd_workspace_size(w.B, w.H, w.N, w.etc_G, w.D, 1), dtype=torch.uint8,
                         device=t["q"].device)

        def f():
            lg.etc_attn_bwd(t["q"], t["k"], t["v"], t["q_g"], t["k_g"], t["v_g"], out_l, out_g, lse_l, lse_g,
                            dout, dout_g, w.radius, workspace=ws)
    else:
        out, lse = outs
        ng = 0 if t["g"] is None else t["g"].numel()
        ws = torch.empty(lg.attn_bwd_workspace_size(w.B, w.H, w.N, w.D, ng, 1), dtype=torch.uint8,
                         device=t["q"].device)
        grads = [torch.empty_like(t["q"]) for _ in range(3)]

        def f():
            lg.attn_bwd(t["q"], t["k"], t["v"], out, lse, dout, w.w_left, w.w_right, w.dilations(), w.causal,
                        t["g"], dq=grads[0], dk=grads[1], dv=grads[2], workspace=ws)
    for _ in range(3):
        f()
    torch.cuda.synchronize()
    st = lg.query_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after the backward warm-up: {lg.status_string(st)}")
    ms = time_steps(torch, f, steps, flush)
    med = statistics.median(ms)
    achieved = flops / (med / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS)) if peaks else FALLBACK_BF16_TFLOPS
    res = {"metric": "sparse attn bwd TFLOP/s (8*D per allowed pair)", "value": round(achieved, 2),
           "unit": "TFLOP/s", "ms_per_call": round(med, 4), "steps": steps,
           "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(achieved / peak, 4), "peak_source": f"bf16_tflops of {peak_kind}",
                        "kernel": "whole backward call (bwd_kv_kernel + bwd_q_kernel dominate)"}}
    del ws, dout
    return res


def sweep(lg, torch, dev):
    """Every preset, briefly: TFLOP/s and ms per call (runtime against N for the long-scale trio)."""
    res = {}
    for name, w in workloads.PRESETS.items():
        t = device_inputs(w, dev, torch)
        f, outs, ws = make_call(lg, w, t, torch)
        flops = 4.0 * w.D * useful_pairs(lg, w)
        in_bytes = sum(x.numel() * x.element_size() for x in t.values() if x is not None)
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        steps = 30 if w.N >= 100000 else 100
        ms = time_steps(torch, f, steps, in_bytes < 2 * L2_BYTES)
        st = lg.query_status(ws)
        med = statistics.median(ms)
        res[name] = {"tflops": round(flops / (med / 1e3) / 1e12, 2), "ms": round(med, 5),
                     "status": lg.status_string(st)}
        if w.dtype == "bf16" and not getattr(sweep, "no_bwd", False):
            b = bench_backward(lg, torch, w, t, outs, in_bytes < 2 * L2_BYTES, 10 if w.N >= 100000 else 30, {}, "")
            if b is not None:
                res[name]["bwd_tflops"] = b["value"]
                res[name]["bwd_ms"] = b["ms_per_call"]
        del t, f, outs, ws
        torch.cuda.empty_cache()
    return res


def kernel_source_digest():
    """Hash of the tensor-core kernel's sources with comments and blank lines removed."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("lg_tc.cu", "lg_internal.h", "lg_ptx.cuh"):
        text = open(os.path.join(ROOT, "sparse_long_sequence_window_gb300", "csrc", name)).read()
        for line in text.splitlines():
            code = re.sub(r"//.*", "", line).rstrip()
            if code.strip():
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def committed_traffic(w):
    """DRAM bytes per launch from a committed ncu capture of the current kernel sources, else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        import hashlib
        with open(path) as f:
            rec = json.load(f)
        digest = kernel_source_digest()
        ent = rec.get(w.name)
        if ent and ent.get("kernel_sha") == digest:
            return ent.get("dram_bytes_per_launch")
    except Exception:
        return None
    return None


# ---------------------------------------------------------------------- CPU oracle

def cpu_inputs(w, seed=1234):
    """One head's inputs for the CPU oracle (drawn once per run)."""
    rng = np.random.default_rng(seed)
    D, N = w.D, w.N
    if w.is_etc:
        G = w.etc_G
        return [rng.standard_normal((1, 1, n, D), dtype=np.float32) for n in (N, N, N, G, G, G)]
    return [rng.standard_normal((1, 1, N, D), dtype=np.float32) for _ in range(3)]


def cpu_sample(w, budget_s, seed=1234, arrs=None):
    """Runs the CPU oracle on uniformly sampled rows of one head for about budget_s seconds.

    Returns (useful FLOPs computed, seconds, rows).
    """
    from oracle import lg_oracle
    rng = np.random.default_rng(seed)
    D, N = w.D, w.N
    if arrs is None:
        arrs = cpu_inputs(w, seed)
    if w.is_etc:
        G = w.etc_G
        flops = 0.0; rows = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            i = int(rng.integers(0, N))
            lg_oracle.etc_attn_fwd_rows(*arrs, w.radius, [i])
            lo, hi = max(0, i - w.radius), min(N - 1, i + w.radius)
            flops += 4.0 * D * ((hi - lo + 1) + G)
            rows += 1
        return flops, time.perf_counter() - t0, rows
    if w.is_longnet:
        q, k, v = arrs
        flops = 0.0; rows = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            i = int(rng.integers(0, N))
            lg_oracle.longnet_attn_fwd_rows(q, k, v, w.seg_w, w.seg_r, w.causal, [i])
            for sw, sr in zip(w.seg_w, w.seg_r):   # head 0: offset 0
                kept = lg_oracle.longnet_rows(N, sw, sr, 0, i // sw)
                if (kept == i).any():
                    flops += 4.0 * D * int((kept <= i).sum() if w.causal else kept.size)
            rows += 1
        return flops, time.perf_counter() - t0, rows
    g = workloads.global_positions(w)
    gflags = np.zeros(N, bool); gflags[g] = True
    q, k, v = arrs
    d = w.dilations()[0]
    flops = 0.0; rows = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        i = int(rng.integers(0, N))
        lg_oracle.attn_fwd_rows(q, k, v, w.w_left, w.w_right, [d], w.causal, g, [i])
        n_keys = int(lg_oracle.allowed_row(i, N, w.w_left, w.w_right, d, w.causal, gflags).sum())
        flops += 4.0 * D * n_keys
        rows += 1
    return flops, time.perf_counter() - t0, rows


# The oracle over all host cores: one spawned worker process per core (spawn,
# not fork: the parent may already hold a CUDA context), each single-threaded,
# each drawing the same one-head inputs once and evaluating its own uniformly
# drawn rows.  The throughput is the sum of the workers' useful FLOPs over the
# wall time of the parallel section.
_WORKER = {}


def _pool_init(preset):
    w = workloads.PRESETS[preset]
    _WORKER["w"] = w
    _WORKER["arrs"] = cpu_inputs(w)


def _pool_task(args):
    budget_s, seed = args
    return cpu_sample(_WORKER["w"], budget_s, seed=seed, arrs=_WORKER["arrs"])


class OraclePool:
    def __init__(self, preset, workers=None):
        import multiprocessing as mp
        self.workers = max(1, workers or os.cpu_count() or 1)
        self.pool = mp.get_context("spawn").Pool(self.workers, initializer=_pool_init, initargs=(preset,))
        # every worker has its inputs before anything is timed
        self.pool.map(_pool_task, [(0.0, i) for i in range(self.workers)], chunksize=1)

    def sample(self, budget_s, seed):
        """Useful FLOPs, wall seconds and rows of one parallel sample of about budget_s seconds."""
        t0 = time.perf_counter()
        res = self.pool.map(_pool_task, [(budget_s, seed * 1000 + i) for i in range(self.workers)], chunksize=1)
        secs = time.perf_counter() - t0
        return sum(r[0] for r in res), secs, sum(r[2] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(preset, budget_s=15.0):
    w = workloads.PRESETS[preset]
    pool = OraclePool(preset)
    try:
        flops, secs, rows = pool.sample(budget_s, seed=1)
    finally:
        pool.close()
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": pool.workers, "kind": "oracle",
            "host_cpu_count": os.cpu_count(),
            "sample": f"{rows} uniformly drawn query rows of one head of {w.name}, fp64 numpy, "
                      f"{secs:.1f} s wall on {pool.workers} single-threaded worker processes"}


def linear_in_n_slope(per_config):
    """Least-squares slope of log(ms per call) against log(N) over the long-scale sweep (1 = linear)."""
    pts = [(workloads.PRESETS[n].N, per_config[n]["ms"]) for n in ("long_8k", "long_32k", "long_128k")
           if n in per_config]
    if len(pts) < 2:
        return None
    x = np.log([p[0] for p in pts]); y = np.log([p[1] for p in pts])
    slope = float(np.polyfit(x, y, 1)[0])
    return {"slope": round(slope, 4), "points_N_ms": [[int(a), b] for a, b in pts],
            "workload": "long_scale bf16 B1 H16 D128 w512/512 G=128 random"}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step a bounded sample of the workload's rows."""
    w = workloads.PRESETS[args.workload]
    per_step = max(0.05, min(10.0, 150.0 / max(1, args.steps + args.warmup)))  # whole run about 2.5 min
    pool = OraclePool(args.workload)
    try:
        for i in range(args.warmup):
            pool.sample(per_step, seed=90 + i)
        total_f, total_s, total_rows = 0.0, 0.0, 0
        for s in range(args.steps):
            fl, sec, rows = pool.sample(per_step, seed=1000 + s)
            total_f += fl; total_s += sec; total_rows += rows
    finally:
        pool.close()
    value = total_f / total_s / 1e12
    sample = (f"{total_rows} uniformly drawn query rows of one head of {w.name} over {args.steps} steps "
              f"of ~{per_step:.1f} s each, fp64 numpy, {pool.workers} single-threaded worker processes")
    return {
        "impl": "reference",
        "metric": "sparse attn fwd TFLOP/s (in-band pairs) & % bf16 tensor peak, N=512-128K",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic iid N(0,1), seeded",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": pool.workers, "kind": "oracle",
                         "host_cpu_count": os.cpu_count(), "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="long_128k", choices=sorted(workloads.PRESETS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward-pass measurement")
    ap.add_argument("--bwd-steps", type=int, default=10)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    line = run_native(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
