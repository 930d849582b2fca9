#!/usr/bin/env python
"""Benchmark of the fused exact-attention hot path on one GB300 (or N replicas).

One step = one forward (attn_fwd) and one backward (attn_bwd_preprocess,
attn_bwd_main, attn_bwd_dq_convert: exactly attn_bwd) over the workload's
batch, inputs resident in HBM.  The default workload is B=4, H=16, N=4096,
d=128, causal, bf16, the shape the metric's percentage-of-peak target is
quoted on.  Printed: one JSON line with TFLOP/s of the whole step (FLOPs:
4 B H N^2 d halved for causal forward, 2.5x that for the backward), the
per-pass figures, the dominant kernel's roofline, the end-to-end figure
through the public API with host buffers, the float64 oracle timed on the
host cores, and the SM clocks sampled during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile

import numpy as np
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_attention_58_gb300.workloads import (Workload, dropout_seed, make_packed_inputs,  # noqa: E402
                                                make_workload_inputs, workload)

METRIC = "attention fwd/bwd TFLOP/s and % of GB300 dense bf16 tensor peak"
DEFAULT_WORKLOAD = 3
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------
def pairs_flops_fwd(w: Workload, window: int, Nk: int) -> float:
    """4 d FLOPs per attended (query, key) pair, counted exactly: query i
    stands at key position t = i + Nk - N; key j < Nk is attended when j <= t
    (causal) and t - j < window (and j - t < window unless causal) for a
    window > 0."""
    t = np.arange(w.N, dtype=np.int64) + (Nk - w.N)
    hi = np.minimum(t + 1, Nk) if w.causal else np.full_like(t, Nk)
    lo = np.zeros_like(t)
    if window > 0:
        lo = np.maximum(0, t - window + 1)
        if not w.causal:
            hi = np.minimum(hi, t + window)
    pairs = np.maximum(0, hi - lo).sum()
    return 4.0 * w.B * w.H * w.d * float(pairs)


def varlen_lengths(w: Workload) -> list:
    """Packed-sequence lengths for a workload: uniform integers in [N/8, N]
    (seeded) until the workload's B * N tokens are used up, the last one
    cut to fit."""
    rng = np.random.default_rng(4000 + w.N)
    lens, left = [], w.B * w.N
    while left > 0:
        n = min(int(rng.integers(max(1, w.N // 8), w.N + 1)), left)
        lens.append(n)
        left -= n
    return lens


def fwd_compulsory_bytes(w: Workload) -> int:
    """Q, K, V read and O written once, plus one fp32 LSE per row."""
    es = 2 if w.dtype == "bf16" else 4
    return w.B * w.H * (4 * w.N * w.d * es + w.N * 4)


def bwd_compulsory_bytes(w: Workload) -> int:
    """Q, K, V, O, dO read and dQ, dK, dV written once, plus LSE read."""
    es = 2 if w.dtype == "bf16" else 4
    return w.B * w.H * (8 * w.N * w.d * es + w.N * 4)


def valid_pairs_in_rows(w: Workload, row0: int, nrows: int) -> int:
    """(query, key) pairs a slice of query rows attends to (no key padding)."""
    if not w.causal:
        return nrows * w.N
    return sum(i + 1 for i in range(row0, row0 + nrows))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_PEAK_TFLOPS, 1700.0, FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("attn_fwd_kernel.cuh", "attn_fwd.cu", "attn_bwd_kernel.cuh", "attn_bwd.cu",
                 "ptx.cuh", "philox.cuh", "seq.cuh", "internal.h"):
        with open(os.path.join(ROOT, "exact_attention_58_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec[kernel][workload_name]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = None

    def start(self):
        import torch
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.device_index).uuid)
        except Exception:
            uuid = str(self.device_index)
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={uuid}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.4)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the float64 oracle on the host cores (a bounded sample of the same workload)
# ---------------------------------------------------------------------------
def tmap_encode_us(ptr: int, BH: int, N: int, d: int, reps: int = 20000) -> float:
    """Host time of one cuTensorMapEncodeTiled call of the kind every entry
    point makes per tensor ([B*H, N, d] 16-bit, 128-byte swizzle, 64 x 128
    box), less the cost of a trivial call through the same ctypes path."""
    import ctypes
    drv = ctypes.CDLL("libcuda.so.1")
    enc = drv.cuTensorMapEncodeTiled
    enc.restype = ctypes.c_int
    u64, u32 = ctypes.c_uint64, ctypes.c_uint32
    tmap = (u64 * 16)()
    dims, strides = (u64 * 3)(d, N, BH), (u64 * 2)(d * 2, N * d * 2)
    box, estr = (u32 * 3)(64, 128, 1), (u32 * 3)(1, 1, 1)
    # data type bf16 (9), 3-D, no interleave, 128-byte swizzle (3), L2 256B (3), no OOB NaN
    call = (tmap, 9, 3, ctypes.c_void_p(ptr), dims, strides, box, estr, 0, 3, 3, 0)
    if enc(*call) != 0:
        return float("nan")
    noop = drv.cuDriverGetVersion
    ver = ctypes.c_int()
    t0 = time.perf_counter()
    for _ in range(reps):
        enc(*call)
    t1 = time.perf_counter()
    for _ in range(reps):
        noop(ctypes.byref(ver))
    t2 = time.perf_counter()
    return max(0.0, ((t1 - t0) - (t2 - t1)) / reps * 1e6)


def pinned_copy_gbs(host: list, dev: list, stream, reps: int = 5) -> dict:
    """Raw copy rates between pinned host buffers and device buffers: each
    direction alone, then both at once on two streams."""
    import torch
    other = torch.cuda.Stream()
    nbytes = sum(t.numel() * t.element_size() for t in host)

    def timed(fn_h2d, fn_d2h):
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(reps):
            s.record(stream)
            other.wait_event(s)
            for t_h, t_d in zip(host, dev):
                if fn_h2d:
                    with torch.cuda.stream(stream):
                        t_d.copy_(t_h, non_blocking=True)
                if fn_d2h:
                    with torch.cuda.stream(other):
                        t_h.copy_(t_d, non_blocking=True)
            stream.wait_stream(other)
            e.record(stream)
            torch.cuda.synchronize()
            best = min(best, s.elapsed_time(e))
        return nbytes * (int(fn_h2d) + int(fn_d2h)) / (best * 1e-3) / 1e9

    return {"h2d": round(timed(True, False), 1), "d2h": round(timed(False, True), 1),
            "both_ways_total": round(timed(True, True), 1), "bytes": nbytes}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(inp, w: Workload, heads: int, row0: int, nrows: int, threads: int):
    """Run the oracle's forward+backward on `nrows` query rows of `heads` heads.
    Returns (seconds, algorithmic FLOPs of the sample)."""
    import numpy as np

    import oracle
    hs = [(x // w.H, x % w.H) for x in range(heads)]
    sel = lambda t: np.stack([t[b, h].double().numpy() for b, h in hs])  # noqa: E731
    Q, K, V, dO = sel(inp.q), sel(inp.k), sel(inp.v), sel(inp.do)
    b_idx = [b for b, _ in hs]
    h_idx = [h for _, h in hs]
    kl = [w.N] * heads
    t0 = time.perf_counter()
    oracle.heads_rows_fwd_bwd(Q, K, V, dO, b_idx, h_idx, kl, inp.scale, row0, nrows, w.causal,
                              inp.dropout_p, inp.seed, nthreads=threads)
    dt = time.perf_counter() - t0
    flops = heads * valid_pairs_in_rows(w, row0, nrows) * 14.0 * w.d   # 4d fwd + 10d bwd
    return dt, flops


def calibrate_rows(inp, w, heads, threads, target_s):
    """Rows per head (around N/2) so that one oracle sample of `heads` heads
    takes about target_s seconds."""
    row0 = w.N // 2
    oracle_sample(inp, w, heads, row0, 4, threads)           # warm: threads, pages
    probe = 32
    dt, _ = oracle_sample(inp, w, heads, row0, probe, threads)
    per_row = max(dt / probe, 1e-5)
    return max(1, min(w.N - row0, int(target_s / per_row)))


def cpu_baseline(inp, w, target_s=15.0):
    """The oracle on whole heads (all query rows), one head per core, as many
    rounds of `cores` heads as fit in about target_s seconds."""
    threads = host_cores()
    heads = min(threads, w.B * w.H)
    dt1, fl1 = oracle_sample(inp, w, heads, 0, w.N, threads)   # one round, also a warm-up
    rounds = max(1, min((w.B * w.H) // heads, int(target_s / max(dt1, 1e-3))))
    nh = heads * rounds
    dt, flops = oracle_sample(inp, w, nh, 0, w.N, threads)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"float64 oracle forward+backward of all {w.N} query rows of {nh} of the "
                      f"{w.B * w.H} heads of {w.name} ({threads} threads, OpenMP over heads), "
                      f"{dt:.1f} s; FLOPs counted as 14 d per attended (query, key) pair"}


# ---------------------------------------------------------------------------
# several ranks: independent replicas, timed by the slowest
# ---------------------------------------------------------------------------
def max_over_ranks(x: float, device) -> float:
    """The largest x over the ranks of the default process group (x itself
    when there is none): the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank_step: float, steps: int, elapsed_ms: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of its own replica in
    (at most) elapsed_ms."""
    return world * flops_per_rank_step * steps / (elapsed_ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# reference arm: the oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, w: Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = make_workload_inputs(args.workload)
    threads = host_cores()
    heads = min(threads, w.B * w.H)
    per_step = max(0.5, args.reference_budget_s / (args.steps + args.warmup))
    rows = calibrate_rows(inp, w, heads, threads, per_step)
    row0 = max(0, w.N // 2 - rows // 2)
    for _ in range(args.warmup):
        oracle_sample(inp, w, heads, row0, rows, threads)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = oracle_sample(inp, w, heads, row0, rows, threads)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = (f"each step: float64 oracle forward+backward of query rows [{row0}, {row0 + rows}) "
              f"of {heads} heads of {w.name}, one head per core")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "passes": "fwd+bwd"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "kind": "oracle",
                             "cores": threads, "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, w: Workload):
    import torch
    import torch.distributed as dist

    import exact_attention_58_gb300 as ea

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    ea.library()

    Nk = args.nk if args.nk > 0 else w.N
    # forward-only workloads, and e4m3 inputs (forward only), time the forward alone
    bwd = w.backward and args.dtype != "fp8"
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    half = {"fp16": torch.float16, "fp8": getattr(torch, "float8_e4m3fn", None)}.get(args.dtype)
    lens = None
    if args.varlen:
        # packed sequences: lengths U[N/8, N] until B*N tokens (the workload's
        # token budget); self-attention, the workload's mask and dtype
        lens = varlen_lengths(w)
        inp = make_packed_inputs(lens, lens, w.H, w.d, dtype=half or w.torch_dtype,
                                 sigma=w.sigma, gen_seed=3000 + args.workload, causal=w.causal,
                                 dropout_p=w.dropout_p, dropout_seed_value=dropout_seed(args.workload),
                                 window=args.window)
        q, k, v, do = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.do))
        cu = inp.cu_q.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.H, q.shape[0]), dtype=torch.float32, device=dev)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        ws = torch.empty(ea.attn_bwd_workspace_size(len(lens), w.H, inp.max_q, w.d),
                         dtype=torch.uint8, device=dev)
        kw = dict(causal=w.causal, window=args.window, dropout_p=inp.dropout_p, seed=inp.seed,
                  scale=inp.scale, dev_status=status)
        stages = [
            ("attn_fwd_kernel",
             lambda: ea.attn_fwd_varlen(q, k, v, cu, cu, inp.max_q, inp.max_q, out=o, lse=lse, **kw)),
            ("attn_bwd_varlen (pre+main+convert)",
             lambda: ea.attn_bwd_varlen(q, k, v, o, do, lse, cu, cu, inp.max_q, inp.max_q, dq=dq,
                                        dk=dk, dv=dv, workspace=ws, **kw)),
        ]
    else:
        inp = make_workload_inputs(args.workload, Nk=Nk, d=w.d)
        if half is not None:   # the same draws stored as IEEE half or e4m3
            for name in ("q", "k", "v", "do"):
                t = getattr(inp, name)
                if t is not None:
                    setattr(inp, name, t.to(torch.float32).to(half) if name != "do" or bwd else None)
        q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
        do = inp.do.to(dev) if bwd else None
        kl = inp.key_lens.to(dev) if inp.key_lens is not None else None
        B, H, N, d = q.shape
        o = torch.empty(q.shape, dtype=torch.bfloat16 if args.dtype == "fp8" else q.dtype,
                        device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        if bwd:
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
            ws = torch.empty(ea.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
        kw = dict(causal=w.causal, window=args.window, key_lens=kl, dropout_p=inp.dropout_p,
                  seed=inp.seed, scale=inp.scale)
        stages = [
            ("attn_fwd_kernel", lambda: ea.attn_fwd(q, k, v, out=o, lse=lse, dev_status=status, **kw)),
            ("bwd_pre_kernel", lambda: ea.attn_bwd_preprocess(o, do, lse, ws)),
            ("attn_bwd_kernel",
             lambda: ea.attn_bwd_main(q, k, v, do, dk, dv, ws, dev_status=status, **kw)),
            ("bwd_dq_convert_kernel", lambda: ea.attn_bwd_dq_convert(dq, ws, scale=inp.scale)),
        ]
    if not bwd:
        stages = stages[:1]

    def step(evs=None):
        for i, (_, fn) in enumerate(stages):
            if evs:
                evs[i].record()
            fn()
        if evs:
            evs[len(stages)].record()

    # Inputs that fit in L2 would be served from it on every step; then L2 is
    # flushed (a 256 MiB write) before each step, outside the per-stage
    # events, and the step time is the sum of the stage times.
    qbytes, kbytes = q.numel() * q.element_size(), k.numel() * k.element_size()
    in_bytes = (2 if bwd else 1) * qbytes + 2 * kbytes
    flush = in_bytes <= L2_BYTES
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")

    ns = len(stages)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    start.record()
    for s in range(args.steps):
        if flush:
            flush_buf.zero_()
        step(evs[s])
    end.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")

    elapsed_ms = start.elapsed_time(end)
    per = [[evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(args.steps)] for i in range(ns)]
    if flush:   # the flushes are not part of the step
        elapsed_ms = sum(evs[s][0].elapsed_time(evs[s][ns]) for s in range(args.steps))
    elapsed_ms = max_over_ranks(elapsed_ms, dev)

    exact = args.window > 0 or Nk != w.N or lens is not None
    if lens is not None:   # each packed sequence counted on its own
        flops_fwd = sum(pairs_flops_fwd(dataclasses.replace(w, B=1, N=n), args.window, n)
                        for n in lens if n > 0)
    else:
        flops_fwd = pairs_flops_fwd(w, args.window, Nk) if exact else w.flops_fwd()
    flops_bwd = (2.5 * flops_fwd) if bwd else 0.0
    flops_step = flops_fwd + flops_bwd
    value = job_tflops(world, flops_step, args.steps, elapsed_ms)
    kernel_ms = {name: statistics.mean(x) for (name, _), x in zip(stages, per)}
    fwd_ms = kernel_ms["attn_fwd_kernel"]
    bwd_ms = sum(kernel_ms.values()) - fwd_ms
    peak, peak_sus, hbm, peak_src = load_peaks()
    fwd_tf = flops_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = flops_bwd / (bwd_ms * 1e-3) / 1e12 if bwd else None
    # the backward's dominant launch: the main kernel (with pre and convert
    # when the packed entry point times the three together)
    bwd_main = "attn_bwd_kernel" if "attn_bwd_kernel" in kernel_ms else stages[-1][0]
    main_ms = kernel_ms.get(bwd_main, 0.0)
    main_tf = flops_bwd / (main_ms * 1e-3) / 1e12 if bwd else None
    if bwd and main_ms >= fwd_ms:
        dom, dom_tf, dom_ms = bwd_main, main_tf, main_ms
    else:
        dom, dom_tf, dom_ms = "attn_fwd_kernel", fwd_tf, fwd_ms
    peak_note = f"{peak_src} bf16 dense (burst)"
    if args.dtype == "fp8":   # e4m3 products: the bf16 figure times the nominal 2x ratio
        peak, peak_note = 2.0 * peak, f"{peak_src} bf16 dense (burst) x 2 (nominal fp8/bf16 ratio)"
    roofline = {"bound": "tensor", "kernel": dom, "achieved": dom_tf, "peak": peak,
                "unit": "TFLOP/s", "frac": dom_tf / peak, "traffic": recorded_traffic(dom, w.name),
                "peak_source": peak_note}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- end to end through the public API with pinned host buffers ----
    # Every step copies its inputs from pinned host memory, runs the public
    # calls and copies its results back.  Two sets of device buffers and three
    # streams (host-to-device, compute, device-to-host) let one step's copies
    # overlap another step's compute, as a training or serving loop would.
    e2e = None
    if args.e2e_steps > 0:
        host_in = {"q": inp.q.pin_memory(), "k": inp.k.pin_memory(), "v": inp.v.pin_memory()}
        if bwd:
            host_in["do"] = inp.do.pin_memory()
        if lens is not None:
            host_in["cu"] = inp.cu_q.pin_memory()
        dev0 = {"q": q, "k": k, "v": v, "o": o, "lse": lse}
        if bwd:
            dev0.update(do=do, dq=dq, dk=dk, dv=dv)
        if lens is not None:
            dev0["cu"] = cu
        slots = [dev0, {name: torch.empty_like(t) for name, t in dev0.items()}]
        out_names = ["o", "dq", "dk", "dv"] if bwd else ["o"]
        host_out = {name: torch.empty(dev0[name].shape, dtype=dev0[name].dtype).pin_memory()
                    for name in out_names}

        def api(sl, stream):
            """The public calls of one step on buffer set `sl`."""
            if lens is not None:
                kv = dict(kw, stream=stream)
                ea.attn_fwd_varlen(sl["q"], sl["k"], sl["v"], sl["cu"], sl["cu"], inp.max_q,
                                   inp.max_q, out=sl["o"], lse=sl["lse"], **kv)
                if bwd:
                    ea.attn_bwd_varlen(sl["q"], sl["k"], sl["v"], sl["o"], sl["do"], sl["lse"],
                                       sl["cu"], sl["cu"], inp.max_q, inp.max_q, dq=sl["dq"],
                                       dk=sl["dk"], dv=sl["dv"], workspace=ws, **kv)
                return
            ea.attn_fwd(sl["q"], sl["k"], sl["v"], out=sl["o"], lse=sl["lse"], stream=stream, **kw)
            if bwd:
                ea.attn_bwd(sl["q"], sl["k"], sl["v"], sl["o"], sl["do"], sl["lse"], dq=sl["dq"],
                            dk=sl["dk"], dv=sl["dv"], workspace=ws, stream=stream, **kw)

        h2d, comp, d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
        in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

        def e2e_step(step):
            x = step % 2
            sl = slots[x]
            if step >= 2:
                h2d.wait_event(comp_done[x])     # step - 2 has read these inputs
            with torch.cuda.stream(h2d):
                for name, src in host_in.items():
                    sl[name].copy_(src, non_blocking=True)
                in_ready[x].record(h2d)
            comp.wait_event(in_ready[x])
            if step >= 2:
                comp.wait_event(out_done[x])     # step - 2's results have left
            with torch.cuda.stream(comp):
                api(sl, comp)
                comp_done[x].record(comp)
            d2h.wait_event(comp_done[x])
            with torch.cuda.stream(d2h):
                for name in out_names:
                    host_out[name].copy_(sl[name], non_blocking=True)
                out_done[x].record(d2h)

        for step in range(2):
            e2e_step(step)
        torch.cuda.synchronize()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(h2d)
        for step in range(args.e2e_steps):
            e2e_step(step)
        e_ev.record(d2h)
        torch.cuda.synchronize()
        e_ms = s_ev.elapsed_time(e_ev)
        h2d_bytes = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h_bytes = sum(t.numel() * t.element_size() for t in host_out.values())
        # host side: the time to enqueue one step's public calls (argument
        # checks, tensor-map encodes, launches), one tensor-map encode, and the
        # raw pinned copy rates the pipeline is bounded by
        reps = 50
        t0 = time.perf_counter()
        for _ in range(reps):
            api(slots[0], comp)
        api_us = (time.perf_counter() - t0) / reps * 1e6
        torch.cuda.synchronize()
        pairs = [(host_in[n], slots[1][n]) for n in host_in]
        pairs += [(host_out[n], slots[1][n]) for n in out_names]
        copy_gbs = pinned_copy_gbs([h for h, _ in pairs], [dv for _, dv in pairs], h2d)
        e2e = {"value": flops_step * args.e2e_steps / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "ms_per_step": e_ms / args.e2e_steps,
               "pipeline": "2 buffer sets; copies in, compute, copies out on three streams",
               "host_enqueue_us_per_step": round(api_us, 1),
               "tmap_encode_us": round(tmap_encode_us(q.data_ptr(), w.B * w.H, w.N, w.d), 3)
               if lens is None and w.d <= 256 else None,
               "raw_pinned_copy_gbs": copy_gbs}

    cpu = None
    # the sample is forward+backward of the default (unwindowed) configuration
    if world == 1 and not args.no_cpu_baseline and bwd and not exact:
        cpu = cpu_baseline(inp, w, target_s=args.cpu_seconds)

    l2_note = (f"inputs {in_bytes / 2**20:.0f} MiB <= L2: L2 flushed (256 MiB write) before every step"
               if flush else f"inputs {in_bytes / 2**20:.0f} MiB > L2 {L2_BYTES / 2**20:.0f} MiB, no flush")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.dtype if args.dtype != "default" else ("bf16" if w.dtype == "bf16" else "tf32"),
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "dropout_p": w.dropout_p,
                   "passes": "fwd+bwd" if bwd else "fwd",
                   "window": args.window if args.window > 0 else None,
                   "Nk": Nk if Nk != w.N else None,
                   "varlen": ({"sequences": len(lens), "tokens": sum(lens), "min": min(lens),
                               "max": max(lens)} if lens is not None else None),
                   "global_batch": world * w.B, "seq_len": w.N,
                   "parallelism": f"replicas x{world} (heads independent)",
                   "l2": l2_note},
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf, "fwd_frac_peak": fwd_tf / peak,
        "bwd_frac_peak": bwd_tf / peak if bwd else None, "peak_tflops": peak,
        "kernel_ms": kernel_ms,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (4 if bwd else 1) * args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, help="1-based workload index")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window of this many keys (FLOPs count the attended pairs exactly)")
    ap.add_argument("--nk", type=int, default=0,
                    help="cross-attention: this many keys (queries are the last N positions)")
    ap.add_argument("--headdim", type=int, default=0,
                    help="override the workload's head dim (64, 128 or 256)")
    ap.add_argument("--varlen", action="store_true",
                    help="packed variable-length sequences with the workload's token budget")
    ap.add_argument("--dtype", choices=["default", "fp16", "fp8"], default="default",
                    help="fp16: store the workload's inputs as IEEE half; fp8: as e4m3, forward "
                         "only, O in bf16 (16-bit workloads only)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = workload(args.workload)
    if args.headdim:
        w = dataclasses.replace(w, d=args.headdim, name=f"{w.name}_headdim{args.headdim}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
