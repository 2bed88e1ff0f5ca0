#!/usr/bin/env python
"""Benchmark of the fused attention hot path on GB300.

One step = one forward + backward pass (every step of the path: TMA staging, tile
skipping, Q K^T, masking, online softmax, P V, epilogue; Delta, the backward main
kernel, the dQ finalize) over the dense causal head_dim-512 workload
B=2, Hq=32, Hkv=4, S=4096, scale 1/sqrt(512), seeded N(0,1) bf16 inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. `value` is whole-job fwd+bwd TFLOP/s with inputs resident in
HBM (causal-aware count: 4*D per unmasked (query, key) pair forward, 10*D backward);
`e2e` is the same metric through the C ABI with host buffers (pinned host -> device
copies of q, k, v, dO and device -> host copies of o, lse, dQ, dK, dV of every step inside
the timed region; the copies of neighbouring steps overlap the compute on two copy
streams, with two device buffer sets). Inputs (q, dO: 268 MB each) are larger than L2, so no flush is needed between
steps. `roofline` is for the kernel with the largest device time, timed live with CUDA
events bracketing each launch. `extra` holds the sliding-window (d256, W=1024),
varlen (d512) and paged-decode (HBM GB/s) measurements. `cpu_baseline` is the fp64
oracle timed on the host cores over a causal prefix of the same workload.

Under torchrun (N > 1) every rank runs its own replica on its own batch (the
workload shards by batch / head group with no exchange): "scaling": "weak".
`--impl reference` times the fp64 oracle (the reference arm for this path) on a
bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd+bwd TFLOP/s (d512 causal, d256 SWA) % BF16 peak; decode HBM GB/s"
WORKLOAD = {"workload": "dense causal attention fwd+bwd, head_dim 512, GQA 8:1",
            "B": 2, "Hq": 32, "Hkv": 4, "S": 4096, "D": 512, "causal": True, "window": 0,
            "scale": "1/sqrt(512)", "inputs": "seeded N(0,1) bf16", "l2": "inputs larger than L2 (no flush)"}
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# dram bytes per launch (ncu: dram__bytes_read.sum + dram__bytes_write.sum) for kernels whose
# counters were captured, keyed by kernel; valid only while the kernel's own sources hash the same.
# bwd_main_d512: captured at B=1 (half the workload, same per-cluster work) and doubled.
KERNEL_SOURCES = {"bwd_main_d512": ["attn_bwd.cu", "ptx.cuh", "attn_internal.h"],
                  "fwd_d512": ["attn_fwd.cu", "ptx.cuh", "attn_internal.h"]}
TRAFFIC = {"bwd_main_d512": {"bytes": 2 * (2.675791e9 + 1.553483e9), "src": "4aa4b8e941023f1f"}}


def pairs_causal(S: int, W: int = 0) -> int:
    if W <= 0 or W >= S:
        return S * (S + 1) // 2
    return W * (W + 1) // 2 + (S - W) * W


def kernel_sources_hash(files) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_flash_gqa_gb300", "csrc")
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


# ----------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks/throttle sampling every 200 ms; keeps samples inside [t0, t1]."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [v for t, v in self.samples if any(a <= t <= b for a, b in self.windows)]
        if not inside:
            inside = [v for _, v in self.samples]
        def num(x):
            try:
                return float(x.split()[0])
            except Exception:
                return None
        sm = [num(v[0]) for v in inside if len(v) >= 8 and num(v[0]) is not None]
        mx = [num(v[1]) for v in inside if len(v) >= 8 and num(v[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for v in inside if len(v) >= 8 for i in range(4) if v[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ----------------------------------------------------------------------------------------------
def dist_setup(n_gpus: int):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        pg = dist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank_step: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job rate: every rank runs its own replica of the step (weak scaling), the step time
    is the slowest rank's."""
    return flops_per_rank_step * world / (ms_per_step_max * 1e-3) / 1e12


def to_dev(bits, pin=False):
    import numpy as np
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.cuda()


# ----------------------------------------------------------------------------------------------
def bench_ours(args, rank, world, pg):
    import numpy as np
    import torch

    import __graft_entry__
    import attention_flash_gqa_gb300 as attn
    import synth

    __graft_entry__.build()
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()

    p = synth.dense(args.batch, 32, 4, 4096, 512, 0, seed=1000 + rank, name="dense_d512_causal")
    flops_fwd = 4 * p.D * pairs_causal(p.S) * p.B * p.Hq
    flops_bwd = 10 * p.D * pairs_causal(p.S) * p.B * p.Hq
    flops_step = flops_fwd + flops_bwd

    q, k, v, do = (to_dev(x) for x in (p.q, p.k, p.v, p.do))
    o = torch.empty_like(q)
    lse = torch.empty((p.B, p.Hq, p.S), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(attn.attn_workspace_size(attn.ATTN_OP_BWD, p.B, p.Hq, p.Hkv, p.S, p.D), dtype=torch.uint8,
                     device="cuda")

    def step():
        attn.attn_fwd(q, k, v, o, lse, scale=p.scale)
        attn.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, scale=p.scale, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = attn.attn_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {attn.attn_status_string(st)}")
    finite = bool(torch.isfinite(o.float()).all() and torch.isfinite(dq.float()).all()
                  and torch.isfinite(dk.float()).all() and torch.isfinite(dv.float()).all())

    gpu_id = getattr(props, "uuid", None)
    gpu_id = ("GPU-" + str(gpu_id)) if gpu_id is not None and not str(gpu_id).startswith("GPU-") else str(gpu_id or dev)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.5)

    # ---- device-timed region: inputs resident in HBM ----------------------------------------
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    launches0 = attn.attn_launch_count()
    attn.attn_profile_start()
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(pg)
    prof = attn.attn_profile_stop()
    launches = attn.attn_launch_count() - launches0
    clocks.mark(t0, t1)
    ms_step = ev0.elapsed_time(ev1) / args.steps
    ms_step_max = max_over_ranks(pg, ms_step)
    value = aggregate_tflops(flops_step, world, ms_step_max)

    # ---- dominant kernel roofline --------------------------------------------------------------
    dom = max(prof.items(), key=lambda kv: kv[1][1])
    name, (n_launch, total_ms) = dom
    per_launch = {"fwd_d512": flops_fwd, "bwd_main_d512": flops_bwd}.get(name)
    avg_ms = total_ms / n_launch
    achieved = per_launch / (avg_ms * 1e-3) / 1e12 if per_launch else None
    peak = peaks["bf16_tflops"]
    tr = TRAFFIC.get(name)
    traffic = tr["bytes"] if tr and name in KERNEL_SOURCES and tr.get("src") == kernel_sources_hash(
        KERNEL_SOURCES[name]) else None
    roofline = {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak if achieved else None, "traffic": traffic,
                "peak_source": f"{peak_src} bf16_tflops (burst: the timed region lasts well under the seconds "
                               "the sustained figure was taken over)",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"] if achieved else None,
                "avg_launch_ms": avg_ms,
                "kernels": {kname: {"launches": n, "total_ms": round(t, 4), "share": round(t / sum(
                    x[1] for x in prof.values()), 4)} for kname, (n, t) in prof.items()}}

    # ---- end to end through the C ABI with host buffers ---------------------------------------
    if args.no_e2e:
        extra = None if args.no_extra else bench_extra(args, attn, synth, peaks, peak_src, clocks)
        return finish(args, rank, world, p, attn, value, ms_step_max, roofline, None, launches, clocks, finite,
                      props, peaks, peak_src, extra)
    hq, hk, hv, hdo = (to_dev(x, pin=True) for x in (p.q, p.k, p.v, p.do))
    ho = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    hdq = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    hdk = torch.empty(k.shape, dtype=torch.bfloat16).pin_memory()
    hdv = torch.empty(v.shape, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))
    # Every step copies its inputs host -> device and its results device -> host. The steps
    # are pipelined like an input pipeline would: two device buffer sets, the inputs of step
    # i+1 are copied in on one stream while step i computes, and step i's results are copied
    # out on another stream while step i+1 computes. The timed region runs from the first
    # input copy to the last result copy.
    bufs = [dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv)]
    bufs.append({name: torch.empty_like(t) for name, t in bufs[0].items()})
    ws2 = torch.empty_like(ws)
    wss = [ws, ws2]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    inputs_free = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        for ev in computed + out_done + inputs_free:
            ev.record(stream)
        for i in range(n + 1):
            if i < n:  # inputs of step i
                bs = bufs[i % 2]
                with torch.cuda.stream(s_in):
                    s_in.wait_event(inputs_free[i % 2])
                    for name, h in (("q", hq), ("k", hk), ("v", hv), ("do", hdo)):
                        bs[name].copy_(h, non_blocking=True)
                    in_ready[i % 2].record(s_in)
            if i >= 1:  # compute of step i-1 was enqueued last iteration; copy its results out
                bs = bufs[(i - 1) % 2]
                with torch.cuda.stream(s_out):
                    s_out.wait_event(computed[(i - 1) % 2])
                    for name, h in (("o", ho), ("lse", hlse), ("dq", hdq), ("dk", hdk), ("dv", hdv)):
                        h.copy_(bs[name], non_blocking=True)
                    out_done[(i - 1) % 2].record(s_out)
            if i < n:  # compute of step i
                bs = bufs[i % 2]
                stream.wait_event(in_ready[i % 2])
                stream.wait_event(out_done[i % 2])  # step i-2's results have left this buffer set
                attn.attn_fwd(bs["q"], bs["k"], bs["v"], bs["o"], bs["lse"], scale=p.scale)
                attn.attn_bwd(bs["q"], bs["k"], bs["v"], bs["o"], bs["lse"], bs["do"], bs["dq"], bs["dk"], bs["dv"],
                              scale=p.scale, workspace=wss[i % 2])
                computed[i % 2].record(stream)
                inputs_free[i % 2].record(stream)
        stream.wait_event(out_done[(n - 1) % 2])

    e2e_run(2)
    torch.cuda.synchronize()
    e_steps = max(3, args.steps // 4)
    barrier(pg)
    torch.cuda.synchronize()
    ev0.record(stream)
    e2e_run(e_steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(pg, ev0.elapsed_time(ev1) / e_steps)
    e2e = {"value": aggregate_tflops(flops_step, world, e_ms), "unit": "TFLOP/s", "ms_per_step": e_ms,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "pipelining": "inputs of step i+1 copied in and results of step i-1 copied out during step i "
                         "(two device buffer sets, separate copy streams)"}
    del hq, hk, hv, hdo, ho, hlse, hdq, hdk, hdv, bufs, ws2, wss
    extra = None if args.no_extra else bench_extra(args, attn, synth, peaks, peak_src, clocks)
    return finish(args, rank, world, p, attn, value, ms_step_max, roofline, e2e, launches, clocks, finite, props,
                  peaks, peak_src, extra)


def finish(args, rank, world, p, attn, value, ms_step_max, roofline, e2e, launches, clocks, finite, props, peaks,
           peak_src, extra):
    clocks.stop()
    st = attn.attn_get_device_status()
    config = {**WORKLOAD, "B": p.B, "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16)", "config": config,
        "frac_of_bf16_peak": {"burst": value / world / peaks["bf16_tflops"],
                              "sustained": value / world / peaks["bf16_tflops_sustained"], "source": peak_src},
        "roofline": roofline, "e2e": e2e, "gpu_launches": launches, "clocks": clocks.summary(),
        "finite": finite, "device_status": attn.attn_status_string(st), "gpu": props.name,
    }
    if extra is not None:
        out["extra"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds, problem=p)
    out["targets"] = targets(value / world, peaks, extra)  # last, so a truncated record keeps its tail
    return out


def targets(d512_tflops, peaks, extra):
    """The three throughput targets of the workload definition, each beside its measured value:
    fractions of the measured burst bf16 peak (prefill / training) and of the measured HBM
    bandwidth (decode)."""
    def entry(value, unit, peak, target):
        if value is None:
            return {"value": None}
        return {"value": round(value, 1), "unit": unit, "frac": round(value / peak, 4), "target_frac": target,
                "met": value / peak >= target}

    ex = extra or {}
    swa = ex.get("swa_d256_w1024", {}).get("value")
    dec = ex.get("decode_paged_d128", {}).get("value")
    return {"peaks": {"bf16_tflops_burst": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"]},
            "d512_causal_fwd_bwd": entry(d512_tflops, "TFLOP/s", peaks["bf16_tflops"], 0.50),
            "swa_d256_w1024_fwd_bwd": entry(swa, "TFLOP/s", peaks["bf16_tflops"], 0.45),
            "decode_paged_d128": entry(dec, "GB/s", peaks["hbm_gbs"], 0.70)}


def bench_extra(args, attn, synth, peaks, peak_src, clocks):
    """Sliding-window d256 fwd+bwd, head_dim 128 / 64 fwd+bwd, varlen d512 fwd+bwd, paged-cache chunked
    prefill d512 (forward),
    merge of results over disjoint key sets (GB/s), paged decode d128 and sliding-window d256 (GB/s)."""
    import numpy as np
    import torch

    res = {}
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(3, args.steps // 4)

    def timed(fn, n):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        t0 = time.time()
        ev0.record(stream)
        for _ in range(n):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        clocks.mark(t0, time.time())
        return ev0.elapsed_time(ev1) / n

    def per_call_ms(fn, n, before=None):
        """Device time of each of n calls, every call bracketed by its own event pair. All calls are
        queued before the first is waited on, so the host's launch overhead overlaps the GPU's
        work and never sits inside a bracket. `before` (e.g. an L2 flush) runs ahead of each
        bracket."""
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        t0 = time.time()
        for e0, e1 in pairs:
            if before is not None:
                before()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        clocks.mark(t0, time.time())
        return [e0.elapsed_time(e1) for e0, e1 in pairs]

    def graph_per_call_ms(fns, n_calls=100, replays=7):
        """Per-call device time of n_calls back-to-back calls captured in one CUDA graph, the calls
        cycling through `fns` (one per KV pool, each pool larger than L2, so no call finds its
        cache in L2). Median over `replays` replays of the graph, divided by n_calls."""
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for f in fns:
                f()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(n_calls):
                fns[i % len(fns)]()
        graph.replay()
        torch.cuda.synchronize()
        t0 = time.time()
        out = []
        for _ in range(replays):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) / n_calls)
        clocks.mark(t0, time.time())
        del graph
        return out

    def per_kernel(fn, n=3):  # a separate, profiled pass: average ms per launch of each kernel
        attn.attn_profile_start()
        for _ in range(n):
            fn()
        prof = attn.attn_profile_stop()
        return {kname: round(t / cnt, 4) for kname, (cnt, t) in prof.items()}

    # sliding window, d256, W=1024, outliers
    p = synth.swa_d256_w1024(seed=7)
    q, k, v, do = (to_dev(x) for x in (p.q, p.k, p.v, p.do))
    o = torch.empty_like(q)
    lse = torch.empty((p.B, p.Hq, p.S), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    swa_step = lambda: (attn.attn_fwd(q, k, v, o, lse, window=p.window, scale=p.scale),
                        attn.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, window=p.window, scale=p.scale))
    ms = timed(swa_step, steps)
    kern_ms = per_kernel(swa_step)
    fl = 14 * p.D * pairs_causal(p.S, p.window) * p.B * p.Hq
    fin = all(bool(torch.isfinite(t.float()).all()) for t in (o, dq, dk, dv))
    res["swa_d256_w1024"] = {"value": fl / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
                             "frac_of_bf16_peak_burst": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                             "frac_of_bf16_peak_sustained": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                             "all_grads_finite": fin, "kernel_ms": kern_ms}
    del q, k, v, do, o, lse, dq, dk, dv

    # head_dim 128 and 64 (Qwen3-class heads), dense causal fwd+bwd
    for name, make in (("dense_d128_causal", synth.dense_d128_causal), ("dense_d64_causal", synth.dense_d64_causal)):
        p = make(seed=7)
        q, k, v, do = (to_dev(x) for x in (p.q, p.k, p.v, p.do))
        o = torch.empty_like(q)
        lse = torch.empty((p.B, p.Hq, p.S), dtype=torch.float32, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        sd_step = lambda: (attn.attn_fwd(q, k, v, o, lse, scale=p.scale),
                           attn.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, scale=p.scale))
        ms = timed(sd_step, steps)
        kern_ms = per_kernel(sd_step)
        fl = 14 * p.D * pairs_causal(p.S) * p.B * p.Hq
        fin = all(bool(torch.isfinite(t.float()).all()) for t in (o, dq, dk, dv))
        res[name] = {"value": fl / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
                     "frac_of_bf16_peak_burst": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                     "frac_of_bf16_peak_sustained": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                     "shape": {"B": p.B, "Hq": p.Hq, "Hkv": p.Hkv, "S": p.S, "D": p.D}, "all_finite": fin,
                     "kernel_ms": kern_ms}
        del q, k, v, do, o, lse, dq, dk, dv

    # varlen d512
    vp = synth.varlen_d512_causal(seed=7)
    q, k, v, do = (to_dev(x) for x in (vp.q, vp.k, vp.v, vp.do))
    cu = torch.from_numpy(vp.cu_seqlens).cuda()
    o = torch.empty_like(q)
    lse = torch.empty((vp.Hq, vp.total_tokens), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    vl_step = lambda: (attn.attn_fwd_varlen(q, k, v, cu, vp.max_seqlen, o, lse, scale=vp.scale),
                       attn.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, scale=vp.scale, cu_seqlens=cu,
                                     max_seqlen=vp.max_seqlen))
    ms = timed(vl_step, steps)
    kern_ms = per_kernel(vl_step)
    fl = 14 * vp.D * vp.Hq * sum(int(L) * (int(L) + 1) // 2 for L in vp.seqlens)
    fin = all(bool(torch.isfinite(t.float()).all()) for t in (o, dq, dk, dv))
    res["varlen_d512_causal"] = {"value": fl / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
                                 "frac_of_bf16_peak_burst": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                                 "frac_of_bf16_peak_sustained": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                                 "all_finite": fin, "seqlens": [int(x) for x in vp.seqlens], "kernel_ms": kern_ms}
    del q, k, v, do, o, lse, dq, dk, dv

    # chunked prefill over a paged cache, d512 (forward only: the new tokens' attention)
    pf = synth.prefill_paged_d512(seed=7)
    qp, kcp, vcp = to_dev(pf.q), to_dev(pf.k_cache), to_dev(pf.v_cache)
    btp = torch.from_numpy(pf.block_table).cuda()
    slp = torch.from_numpy(pf.seq_lens).cuda()
    cuq = torch.from_numpy(pf.cu_q).cuda()
    op = torch.empty_like(qp)
    lp = torch.empty((pf.Hq, pf.total_q), dtype=torch.float32, device="cuda")
    pf_step = lambda: attn.attn_fwd_paged(qp, kcp, vcp, btp, slp, cuq, pf.max_q, op, lp, scale=pf.scale)
    ms = timed(pf_step, max(10, steps))
    kern_ms = per_kernel(pf_step)
    # query i of a request with L cached and n new tokens sees L - n + i + 1 keys
    pairs = sum(int(n) * (int(L) - int(n)) + int(n) * (int(n) + 1) // 2 for L, n in zip(pf.seq_lens, pf.q_lens))
    fl = 4 * pf.D * pf.Hq * pairs
    res["prefill_paged_d512"] = {
        "value": fl / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_call": ms,
        "frac_of_bf16_peak_burst": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
        "frac_of_bf16_peak_sustained": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
        "seq_lens": [int(x) for x in pf.seq_lens], "new_tokens": [int(x) for x in pf.q_lens],
        "all_finite": bool(torch.isfinite(op.float()).all()), "kernel_ms": kern_ms,
        "l2": "inputs larger than L2 (q 134 MB, caches 2 x 84 MB)"}
    del qp, kcp, vcp, op, lp

    # merge of results over disjoint key sets: one rank's combining step of an 8-way ring
    mg = synth.merge_cp8_d512(seed=7)
    mo = to_dev(mg.o_parts)
    ml = torch.from_numpy(mg.lse_parts).cuda()
    om = torch.empty(mo.shape[1:], dtype=torch.bfloat16, device="cuda")
    lm = torch.empty(ml.shape[1:], dtype=torch.float32, device="cuda")
    rows_m = mg.B * mg.S * mg.H
    m_bytes = mg.P * rows_m * (mg.D * 2 + 4) + rows_m * (mg.D * 2 + 4)
    mtimes = per_call_ms(lambda: attn.attn_merge_lse(mo, ml, om, lm), max(20, args.steps) + 3)[3:]
    mmed = statistics.median(mtimes)
    mgbs = m_bytes / (mmed * 1e-3) / 1e9
    res["merge_lse_cp8_d512"] = {"value": mgbs, "unit": "GB/s", "us_per_call_median": mmed * 1e3,
                                 "us_per_call_min": min(mtimes) * 1e3, "bytes_per_call": m_bytes,
                                 "frac_of_hbm_peak": mgbs / peaks["hbm_gbs"], "peak_source": peak_src,
                                 "parts": mg.P, "rows": rows_m, "D": mg.D,
                                 "l2": "inputs larger than L2 (537 MB of parts)"}
    del mo, ml, om, lm

    # paged decode: time the kernel alone, flushing L2 (write > L2) between calls
    pp = synth.decode_paged_d128(seed=7)
    qd, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt = torch.from_numpy(pp.block_table).cuda()
    sl = torch.from_numpy(pp.seq_lens).cuda()
    od = torch.empty_like(qd)
    ld = torch.empty((pp.B, pp.Hq), dtype=torch.float32, device="cuda")
    wsd = torch.zeros(attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, pp.B, pp.Hq, pp.Hkv, 0, pp.D),
                      dtype=torch.uint8, device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    kv_bytes = int(sum(int(L) for L in pp.seq_lens)) * pp.Hkv * pp.D * 2 * 2
    io_bytes = pp.B * pp.Hq * pp.D * 2 * 2 + pp.B * pp.Hq * 4
    flush_l2 = lambda: flush.fill_(1)
    decode_d128 = lambda kcache, vcache: attn.attn_decode_paged(qd, kcache, vcache, bt, sl, od, ld, scale=pp.scale,
                                                                workspace=wsd)
    # (1) CUDA-graph replay of 100 back-to-back calls alternating between two KV pools (268 MB
    # each, more than L2): the serving loop's view, launch costs amortised
    kc2, vc2 = kc.clone(), vc.clone()
    gtimes = graph_per_call_ms([lambda: decode_d128(kc, vc), lambda: decode_d128(kc2, vc2)])
    gmed = statistics.median(gtimes)
    # (2) single calls, each after a 512 MB write that flushes L2 (and leaves it dirty)
    times = per_call_ms(lambda: decode_d128(kc, vc), max(20, args.steps) + 3, flush_l2)[3:]
    med = statistics.median(times)
    gbs = (kv_bytes + io_bytes) / (gmed * 1e-3) / 1e9
    gbs_flushed = (kv_bytes + io_bytes) / (med * 1e-3) / 1e9
    res["decode_paged_d128"] = {"value": gbs, "unit": "GB/s", "us_per_call_median": gmed * 1e3,
                                "us_per_call_min": min(gtimes) * 1e3, "bytes_per_call": kv_bytes + io_bytes,
                                "frac_of_hbm_peak": gbs / peaks["hbm_gbs"], "peak_source": peak_src,
                                "timing": "CUDA graph of 100 calls alternating between two KV pools, each larger than "
                                          "L2; median of 7 replays / 100",
                                "single_call_flushed": {"value": gbs_flushed, "unit": "GB/s", "us_median": med * 1e3,
                                                        "us_min": min(times) * 1e3,
                                                        "frac_of_hbm_peak": gbs_flushed / peaks["hbm_gbs"],
                                                        "timing": "per-call event pairs after a 512 MB L2-flushing "
                                                                  "write, all calls queued ahead"}}
    del qd, kc, vc, kc2, vc2, od, ld, wsd

    # sliding-window decode at head_dim 256 (W = 1024): only the window's keys are read
    ps = synth.decode_paged_swa_d256(seed=7)
    qs, kcs, vcs = to_dev(ps.q), to_dev(ps.k_cache), to_dev(ps.v_cache)
    bts = torch.from_numpy(ps.block_table).cuda()
    sls = torch.from_numpy(ps.seq_lens).cuda()
    os_ = torch.empty_like(qs)
    ls = torch.empty((ps.B, ps.Hq), dtype=torch.float32, device="cuda")
    wss = torch.zeros(attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, ps.B, ps.Hq, ps.Hkv, 0, ps.D),
                      dtype=torch.uint8, device="cuda")
    kv_s = int(sum(min(int(L), ps.window) for L in ps.seq_lens)) * ps.Hkv * ps.D * 2 * 2
    io_s = ps.B * ps.Hq * ps.D * 2 * 2 + ps.B * ps.Hq * 4
    decode_swa = lambda kcache, vcache: attn.attn_decode_paged(qs, kcache, vcache, bts, sls, os_, ls, scale=ps.scale,
                                                               window=ps.window, workspace=wss)
    kcs2, vcs2 = kcs.clone(), vcs.clone()
    gtimes = graph_per_call_ms([lambda: decode_swa(kcs, vcs), lambda: decode_swa(kcs2, vcs2)])
    gmed = statistics.median(gtimes)
    times = per_call_ms(lambda: decode_swa(kcs, vcs), max(20, args.steps) + 3, flush_l2)[3:]
    med = statistics.median(times)
    gbs = (kv_s + io_s) / (gmed * 1e-3) / 1e9
    gbs_flushed = (kv_s + io_s) / (med * 1e-3) / 1e9
    res["decode_paged_swa_d256"] = {"value": gbs, "unit": "GB/s", "us_per_call_median": gmed * 1e3,
                                    "us_per_call_min": min(gtimes) * 1e3, "bytes_per_call": kv_s + io_s,
                                    "frac_of_hbm_peak": gbs / peaks["hbm_gbs"], "peak_source": peak_src,
                                    "window": ps.window,
                                    "timing": "CUDA graph of 100 calls alternating between two KV pools, each larger "
                                              "than L2; median of 7 replays / 100",
                                    "single_call_flushed": {"value": gbs_flushed, "unit": "GB/s", "us_median": med * 1e3,
                                                            "us_min": min(times) * 1e3,
                                                            "frac_of_hbm_peak": gbs_flushed / peaks["hbm_gbs"]}}
    del qs, kcs, vcs, kcs2, vcs2, os_, ls, wss
    return res


class OracleSample:
    """fp64 oracle fwd+bwd on the first `prefix` tokens of every sequence of the workload."""

    def __init__(self, problem=None):
        import oracle
        import synth

        self.orc = oracle.get()
        self.p = problem if problem is not None else synth.dense(2, 32, 4, 4096, 512, 0, seed=1000)
        self.nthreads = oracle.default_threads()

    def run(self, S: int) -> float:
        import numpy as np

        p = self.p
        sub = [np.ascontiguousarray(x[:, :S]) for x in (p.q, p.k, p.v, p.do)]
        t = time.time()
        self.orc.fwd(sub[0], sub[1], sub[2], p.scale, nthreads=self.nthreads)
        self.orc.bwd(*sub, p.scale, nthreads=self.nthreads)
        return time.time() - t

    def pick_prefix(self, budget_s: float) -> int:
        t_small = self.run(256)
        # cost grows as S^2: the prefix that fills the budget, in 128-token multiples, <= 4096
        prefix = int(min(4096, max(128, 256 * (budget_s / max(t_small, 1e-3)) ** 0.5)))
        return max(128, prefix - prefix % 128)

    def flops(self, S: int) -> int:
        p = self.p
        return 14 * p.D * pairs_causal(S) * p.B * p.Hq

    def describe(self, S: int) -> str:
        return (f"fp64 oracle fwd+bwd of the first {S} tokens of every sequence "
                f"(B=2, Hq=32, Hkv=4, D=512, causal), {self.nthreads} threads")


def cpu_baseline(budget_s: float = 20.0, problem=None):
    sample = OracleSample(problem)
    prefix = sample.pick_prefix(budget_s)
    dt = sample.run(prefix)
    return {"value": sample.flops(prefix) / dt / 1e12, "unit": "TFLOP/s", "cores": sample.nthreads,
            "kind": "oracle", "seconds": dt, "sample": sample.describe(prefix)}


def bench_reference(args, rank, world):
    """The reference arm: the fp64 oracle as it stands, on the host cores."""
    if rank != 0:
        return None
    sample = OracleSample()
    total = 150.0  # seconds for the whole run
    prefix = sample.pick_prefix(max(1.0, total / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        sample.run(prefix)
    secs = [sample.run(prefix) for _ in range(args.steps)]
    med = statistics.median(secs)
    value = sample.flops(prefix) / med / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": med * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {**WORKLOAD, "parallelism": "host cores", "sample_tokens": prefix,
                   "sample": f"each step is the causal prefix of the first {prefix} of the S = 4096 tokens"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": sample.nthreads, "kind": "oracle",
                         "sample": sample.describe(prefix) + "; each step one such sample"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def profile_case(args):
    """Run one workload's kernels W + K times and print their device time, for profiler captures
    on a reduced case (no bench line). Cases:
      prefill_paged_d512: the first `--requests` requests of the chunked-prefill workload;
      dense_d128: head_dim 128 forward + backward at batch `--batch`;
      merge_cp8_d512: the 8-part merge;
      decode_swa_d256: the sliding-window head_dim 256 decode;
      decode_d128: the head_dim 128 paged decode (batch 64, Hq 32, Hkv 8);
      swa_d256: the sliding-window head_dim 256 forward + backward at batch `--batch`."""
    import numpy as np
    import torch

    import attention_flash_gqa_gb300 as attn
    import synth

    attn.load_library()
    torch.cuda.set_device(0)
    case = args.profile_case
    extra = {}
    if case == "prefill_paged_d512":
        full = synth.prefill_paged_d512(seed=7)
        n = max(1, min(args.requests, full.B))
        pf = synth.prefill_paged_from_lengths(full.seq_lens[:n], full.q_lens[:n], full.Hq, full.Hkv, full.D, seed=7)
        qp, kc, vc = to_dev(pf.q), to_dev(pf.k_cache), to_dev(pf.v_cache)
        bt, sl, cu = (torch.from_numpy(x).cuda() for x in (pf.block_table, pf.seq_lens, pf.cu_q))
        o = torch.empty_like(qp)
        lse = torch.empty((pf.Hq, pf.total_q), dtype=torch.float32, device="cuda")
        run = lambda: attn.attn_fwd_paged(qp, kc, vc, bt, sl, cu, pf.max_q, o, lse, scale=pf.scale)
        outs = [o]
        extra = {"requests": n, "seq_lens": [int(x) for x in pf.seq_lens]}
    elif case == "dense_d128":
        p = synth.dense(args.batch, 32, 8, 4096, 128, 0, seed=7)
        q, k, v, do = (to_dev(x) for x in (p.q, p.k, p.v, p.do))
        o = torch.empty_like(q)
        lse = torch.empty((p.B, p.Hq, p.S), dtype=torch.float32, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        run = lambda: (attn.attn_fwd(q, k, v, o, lse, scale=p.scale),
                       attn.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, scale=p.scale))
        outs = [o, dq, dk, dv]
        extra = {"B": p.B}
    elif case == "merge_cp8_d512":
        mg = synth.merge_cp8_d512(seed=7)
        mo, ml = to_dev(mg.o_parts), torch.from_numpy(mg.lse_parts).cuda()
        om = torch.empty(mo.shape[1:], dtype=torch.bfloat16, device="cuda")
        lm = torch.empty(ml.shape[1:], dtype=torch.float32, device="cuda")
        run = lambda: attn.attn_merge_lse(mo, ml, om, lm)
        outs = [om]
    elif case == "decode_swa_d256":
        ps = synth.decode_paged_swa_d256(seed=7)
        qs, kcs, vcs = to_dev(ps.q), to_dev(ps.k_cache), to_dev(ps.v_cache)
        bts, sls = torch.from_numpy(ps.block_table).cuda(), torch.from_numpy(ps.seq_lens).cuda()
        os_ = torch.empty_like(qs)
        ls = torch.empty((ps.B, ps.Hq), dtype=torch.float32, device="cuda")
        run = lambda: attn.attn_decode_paged(qs, kcs, vcs, bts, sls, os_, ls, scale=ps.scale, window=ps.window)
        outs = [os_]
    elif case == "swa_d256":
        p = synth.dense(args.batch, 32, 16, 8192, 256, 1024, seed=7, outlier_frac=0.01, outlier_scale=30.0)
        q, k, v, do = (to_dev(x) for x in (p.q, p.k, p.v, p.do))
        o = torch.empty_like(q)
        lse = torch.empty((p.B, p.Hq, p.S), dtype=torch.float32, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        run = lambda: (attn.attn_fwd(q, k, v, o, lse, window=p.window, scale=p.scale),
                       attn.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, window=p.window, scale=p.scale))
        outs = [o, dq, dk, dv]
        extra = {"B": p.B}
    elif case == "decode_d128":
        pd = synth.decode_paged_d128(seed=7)
        qd, kcd, vcd = to_dev(pd.q), to_dev(pd.k_cache), to_dev(pd.v_cache)
        btd, sld = torch.from_numpy(pd.block_table).cuda(), torch.from_numpy(pd.seq_lens).cuda()
        od = torch.empty_like(qd)
        ld = torch.empty((pd.B, pd.Hq), dtype=torch.float32, device="cuda")
        run = lambda: attn.attn_decode_paged(qd, kcd, vcd, btd, sld, od, ld, scale=pd.scale)
        outs = [od]
    else:
        raise SystemExit(f"unknown profile case {case}")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    ev0.record()
    for _ in range(args.steps):
        run()
    ev1.record()
    torch.cuda.synchronize()
    ok = all(bool(torch.isfinite(t.float()).all()) for t in outs) and attn.attn_get_device_status() == 0
    print(json.dumps({"profile_case": case, **extra, "ms_per_call": ev0.elapsed_time(ev1) / args.steps, "ok": ok}),
          flush=True)
    if not ok:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the SWA / varlen / decode measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--batch", type=int, default=2, help="batch of the dense workload (2 = the workload; 1 for "
                                                          "smaller profiler captures)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) leg")
    ap.add_argument("--profile-case", default=None, help="run only this workload's kernel (for profiler captures)")
    ap.add_argument("--requests", type=int, default=8, help="requests of the --profile-case workload")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile_case:
        profile_case(args)
        return
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
        out = bench_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    rank, world, _, pg = dist_setup(args.gpus)
    out = bench_ours(args, rank, world, pg)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
