#!/usr/bin/env python
"""Benchmark of the quantized-weight projection matmul on one GB300.

A step is one 512-token prefill pass over the LFM2.5-350M projection shapes
(ffn_gate 4608x1024, ffn_down 1024x4608, conv_in 3072x1024, attn_out
1024x1024) with W in f32, Q4_0 and Q8_0: twelve qmm_gemm calls through the C
ABI, on seeded synthetic inputs already resident in HBM.  The headline value is
the step's total algorithmic FLOPs (2*m*k*n per GEMM) over its device time.
Inputs rotate over three copies (about 3 x 115 MB, more than the 129 MB L2), so
every step reads its operands from HBM.

The same run also times the small-batch GEMV (n = 1, 2, 4, 8 on 4608x1024 and
1024x4608, Q4_K and Q8_0), the NVFP4 MoE gate/up GEMV (8 experts x 2 planes of
2048x4096, four rotated weight copies) and the standalone dequant, and reports
their weight-stream GB/s against the measured HBM bandwidth.

``--impl reference`` times the f64 CPU oracle on a bounded sample of the same
workload (this problem has no runnable reference implementation: the pages'
kernels need a graphics stack or are not published).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quant-GEMM TFLOP/s per dtype (n=512 prefill); GEMV GB/s vs HBM peak"
SHAPES = [("ffn_gate", 4608, 1024), ("ffn_down", 1024, 4608), ("conv_in", 3072, 1024), ("attn_out", 1024, 1024)]
DTYPES = ["f32", "q4_0", "q8_0"]
N_TOKENS = 512
COPIES = 3
WORKLOAD = ("LFM2.5-350M 512-token prefill projections (ffn_gate 4608x1024, ffn_down 1024x4608, "
            "conv_in 3072x1024, attn_out 1024x1024), W in f32/q4_0/q8_0, n=512")
# nominal dense tensor-core rates (PFLOP/s): f16/bf16 2.25, tf32 1.1
TF32_OVER_F16 = 1.1 / 2.25
# DRAM bytes (read + write) per launch of the tensor-core GEMM kernel, the
# mean over the step's 12 launches, from one ncu capture of this workload
# (profiles/gemm_tc_kernel_step_dram_traffic.md).  It describes the kernel
# sources it was taken on; if they change, the bench reports null.
GEMM_TRAFFIC_SOURCES = ("gemv_dequant_gemm_gb300/csrc/gemm_tc.cu", "gemv_dequant_gemm_gb300/csrc/decode.cuh",
                        "gemv_dequant_gemm_gb300/csrc/common.cuh")
GEMM_TRAFFIC_SHA16 = "36d66afbb1831adc"
GEMM_TRAFFIC_BYTES = 9.068e6


def _gemm_traffic():
    import hashlib
    h = hashlib.sha256()
    try:
        for f in GEMM_TRAFFIC_SOURCES:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return GEMM_TRAFFIC_BYTES if h.hexdigest()[:16] == GEMM_TRAFFIC_SHA16 else None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def slowest_rank_ms(ms: float, world: int, device: str) -> float:
    """The largest of the ranks' times (the job ends when its slowest rank
    does); a collective, so every rank calls it."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's step time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# oracle (CPU) timing: the cpu_baseline leg and the reference arm
# --------------------------------------------------------------------------

def _oracle_inputs():
    import oracle
    import synth
    ins = []
    for label, m, k in SHAPES:
        x = synth.activations(N_TOKENS, k)
        for fmt in DTYPES:
            w = synth.weights(fmt, m, k, m * oracle.row_bytes(fmt, k))
            ins.append((label, fmt, m, k, w, x))
    return ins


def _oracle_sample(ins, entries_per_gemm, seed=0):
    """Time the oracle on `entries_per_gemm` output entries of each GEMM."""
    import oracle
    rng = np.random.default_rng(seed)
    flops, t = 0.0, 0.0
    for label, fmt, m, k, w, x in ins:
        ni = rng.integers(0, N_TOKENS, entries_per_gemm)
        mj = rng.integers(0, m, entries_per_gemm)
        t0 = time.perf_counter()
        oracle.matmul_entries(fmt, w, x, m, k, N_TOKENS, ni, mj)
        t += time.perf_counter() - t0
        flops += 2.0 * k * entries_per_gemm
    return flops, t


def _oracle_calibrate(ins, budget_s):
    flops, t = _oracle_sample(ins, 64, seed=99)
    per_entry_s = t / (64 * len(ins))
    return max(1, int(budget_s / (per_entry_s * len(ins))))


def _cores():
    import oracle
    return oracle.max_threads()


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    ins = _oracle_inputs()
    budget = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    entries = _oracle_calibrate(ins, budget)
    for _ in range(args.warmup):
        _oracle_sample(ins, entries, seed=1)
    flops, t = 0.0, 0.0
    for s in range(args.steps):
        f, dt = _oracle_sample(ins, entries, seed=100 + s)
        flops += f
        t += dt
    value = flops / t / 1e12
    sample = (f"{entries} random output entries of each of the 12 GEMMs per step "
              f"(2*k flops each, rows decoded per entry), f64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_ours(args):
    import torch

    import gemv_dequant_gemm_gb300 as q
    import oracle
    import synth

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    hbm_gbs, f16_tflops, peak_src = _peaks()
    tf32_tflops = f16_tflops * TF32_OVER_F16

    h = q.qmm_create(local)
    lib = q.load()
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    # ---- prefill workload: COPIES sets of (W, X, dst, workspace) ----
    gemms = []  # per GEMM: dict with host arrays and per-copy device buffers
    copies_n = max(1, args.copies)
    shapes = [s for s in SHAPES if not args.only or s[0] in args.only.split(",")]
    for label, m, k in shapes:
        x_np = synth.activations(N_TOKENS, k)
        for fmt in DTYPES:
            w_np = synth.weights(fmt, m, k, m * q.qmm_row_bytes(fmt, k))
            wsb = q.qmm_gemm_workspace_bytes(fmt, m, k, N_TOKENS)
            copies = []
            for c in range(copies_n):
                copies.append({
                    "w": torch.from_numpy(w_np).cuda(), "x": torch.from_numpy(x_np).cuda(),
                    "dst": torch.empty(N_TOKENS, m, dtype=torch.float32, device="cuda"),
                    "ws": torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda"),
                })
            gemms.append({"label": label, "fmt": fmt, "m": m, "k": k, "wsb": wsb, "w_np": w_np, "x_np": x_np,
                          "copies": copies, "flops": 2.0 * m * k * N_TOKENS})
    flops_step = sum(g["flops"] for g in gemms)
    copy_mb = sum(b.numel() * b.element_size() for g in gemms for b in g["copies"][0].values()) / 1e6
    dt_code = {f: q.DTYPES[f] for f in DTYPES}

    def launch(g, c):
        b = g["copies"][c]
        st = lib.qmm_gemm(h, dt_code[g["fmt"]], b["w"].data_ptr(), b["x"].data_ptr(), b["dst"].data_ptr(),
                          g["m"], g["k"], N_TOKENS, b["ws"].data_ptr() if g["wsb"] else None, g["wsb"], sptr)
        if st:
            raise q.QmmError(st, "qmm_gemm")

    def step(c, evs=None):
        for i, g in enumerate(gemms):
            if evs is not None:
                evs[i][0].record(stream)
            launch(g, c)
            if evs is not None:
                evs[i][1].record(stream)

    # launches of our kernels per step: x->f16 + tensor-core GEMM for packed W, one for f32 W
    # (all launched with programmatic dependent launch, so consecutive calls overlap)
    launches_per_step = sum(1 if g["fmt"] == "f32" else 2 for g in gemms)

    for i in range(args.warmup):
        step(i % copies_n)
    torch.cuda.synchronize()
    if q.qmm_sync_status(h) != 0:
        raise RuntimeError("device status set during warm-up")

    # ---- timed region: K steps, each its 12 GEMMs back to back ----
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.25)
    wall0 = time.perf_counter()
    for s in range(args.steps):
        # keep the GPU busy while the host enqueues the step, so the events
        # below time kernels and not host launch gaps
        torch.cuda._sleep(1_500_000)
        ev_step[s][0].record(stream)
        step(s % copies_n)
        ev_step[s][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    status = q.qmm_sync_status(h)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    # per-GEMM durations: the same steps with an event pair around every call
    # (events serialize the calls, so these are single-call latencies)
    kb = max(3, min(100, args.steps))
    ev_launch = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in gemms]
                 for _ in range(kb)]
    for s in range(kb):
        torch.cuda._sleep(1_500_000)
        step(s % copies_n, ev_launch[s])
    torch.cuda.synchronize()
    launch_ms = np.array([[a.elapsed_time(b) for a, b in row] for row in ev_launch])  # [steps][gemm]
    ms_per_step = slowest_rank_ms(float(np.mean(step_ms)), world, "cuda")
    value = job_tflops(world, flops_step, ms_per_step)

    per_gemm = []
    for i, g in enumerate(gemms):
        us = float(np.mean(launch_ms[:, i])) * 1e3
        peak = tf32_tflops if g["fmt"] == "f32" else f16_tflops
        per_gemm.append({"shape": g["label"], "dtype": g["fmt"], "us": round(us, 3),
                         "tflops": round(g["flops"] / (us * 1e-6) / 1e12, 2),
                         "frac": round(g["flops"] / (us * 1e-6) / 1e12 / peak, 4)})
    per_dtype = {}
    for f in DTYPES:
        idx = [i for i, g in enumerate(gemms) if g["fmt"] == f]
        fl = sum(gemms[i]["flops"] for i in idx)
        tt = sum(float(np.mean(launch_ms[:, i])) for i in idx) * 1e-3
        per_dtype[f] = round(fl / tt / 1e12, 2)
    # dominant kernel: the tensor-core GEMM (qmm_gemm, n=512), all its launches;
    # its peak is the FLOP-weighted harmonic mix of the f16 and tf32 peaks
    tot_t = float(np.sum(np.mean(launch_ms, axis=0))) * 1e-3
    ideal_t = sum(g["flops"] / ((tf32_tflops if g["fmt"] == "f32" else f16_tflops) * 1e12) for g in gemms)
    achieved = flops_step / tot_t / 1e12
    peak_mix = flops_step / ideal_t / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak_mix, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak_mix, 4), "traffic": _gemm_traffic(),
                "traffic_unit": "bytes per gemm_tc_kernel launch (DRAM read + write, ncu)",
                "kernel": "qmm_gemm tensor-core path (x_to_f16 + gemm_tc); per-call event-timed durations",
                "peak_source": f"{peak_src} bf16 dense {f16_tflops} TFLOP/s; tf32 = x{TF32_OVER_F16:.3f} nominal"}

    # ---- e2e: host buffers through the public API ----
    e2e = None
    if not args.no_e2e:
        pinned = []
        for g in gemms:
            pinned.append({"w": torch.from_numpy(g["w_np"]).pin_memory(), "x": torch.from_numpy(g["x_np"]).pin_memory(),
                           "dst": torch.empty(N_TOKENS, g["m"], dtype=torch.float32).pin_memory()})
        h2d = sum(p["w"].numel() * p["w"].element_size() + p["x"].numel() * 4 for p in pinned)
        d2h = sum(p["dst"].numel() * 4 for p in pinned)
        e2e_steps = max(3, min(20, args.steps))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for rep in range(2):  # one untimed pass, then the timed one
            torch.cuda.synchronize()
            ev0.record(stream)
            for s in range(e2e_steps):
                c = s % copies_n
                for g, p in zip(gemms, pinned):
                    b = g["copies"][c]
                    b["w"].copy_(p["w"], non_blocking=True)
                    b["x"].copy_(p["x"], non_blocking=True)
                    launch(g, c)
                    p["dst"].copy_(b["dst"], non_blocking=True)
            ev1.record(stream)
            torch.cuda.synchronize()
        e2e_ms = slowest_rank_ms(ev0.elapsed_time(ev1) / e2e_steps, world, "cuda")
        e2e = {"value": round(job_tflops(world, flops_step, e2e_ms), 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4)}

    # ---- a6-a8: GEMV, MoE, dequant (weight-stream GB/s vs HBM) ----
    sub = None if args.no_sub else run_sub_benches(q, lib, h, torch, synth, stream, hbm_gbs)

    # ---- CPU baseline: the oracle on a bounded sample ----
    cpu = None
    if rank == 0 and not args.no_cpu:
        ins = _oracle_inputs()
        entries = _oracle_calibrate(ins, 15.0)
        f, t = _oracle_sample(ins, entries, seed=7)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
               "sample": f"{entries} random output entries of each of the 12 GEMMs (f64 oracle, {t:.1f} s)"}

    q.qmm_destroy(h)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16/tf32 operands, f32 accumulate",
            "data": "synthetic (seeded LCG / xorshift64 streams)",
            "config": {"workload": WORKLOAD, "n": N_TOKENS, "dtypes": DTYPES,
                       "gemms_per_step": len(gemms), "flops_per_step": flops_step,
                       "l2": f"inputs rotated over {copies_n} copies of {copy_mb:.0f} MB (L2 129 MB)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "per_dtype_tflops": per_dtype, "per_gemm": per_gemm, "roofline": roofline,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk, "timed_wall_s": round(wall, 3), "sub": sub,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _time_calls(torch, stream, calls, reps):
    """Mean device time (ms) per call of calls[i % len(calls)]() over reps
    back-to-back launches: one event pair around the whole run, so that the
    launches overlap as they do in a model's stream (programmatic dependent
    launch) and no per-call event splits them.  A device-side sleep queued
    first keeps the GPU busy while the host enqueues the run."""
    for i in range(min(reps, 3)):
        calls[i % len(calls)]()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(max(2_000_000, 20_000 * reps))
    e0.record(stream)
    for i in range(reps):
        calls[i % len(calls)]()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _moe_v2_sub(q, lib, h, torch, stream, keep, scales, x, y, in_f, n_ff, n_used, n_pairs, wbytes, hbm_gbs):
    sptr = stream.cuda_stream
    mat_bytes = n_ff * q.qmm_row_bytes("nvfp4", in_f)
    keep2, tables2 = [], []
    for c in range(len(keep) // (2 * n_pairs)):
        ptrs = []
        for i in range(2 * n_pairs):
            src = keep[c * 2 * n_pairs + i]
            dst = torch.empty_like(src)
            st = lib.qmm_nvfp4_repack_v2(h, src.data_ptr(), dst.data_ptr(), n_ff, in_f, sptr)
            if st != 0:
                raise RuntimeError(f"qmm_nvfp4_repack_v2 status {st}")
            keep2.append(dst)
            ptrs.append(dst.data_ptr())
        tables2.append(torch.tensor(ptrs + [0] * n_pairs, dtype=torch.int64, device="cuda"))
    calls = [(lambda tb=tb: lib.qmm_moe_gemv(h, q.NVFP4_V2, tb.data_ptr(), scales.data_ptr(), x.data_ptr(),
                                             y.data_ptr(), in_f, n_ff, n_used, 1, sptr)) for tb in tables2]
    if calls[0]() != 0:
        raise RuntimeError("qmm_moe_gemv refused the V2 table")
    ms = _time_calls(torch, stream, calls, 40)
    gbs = wbytes / (ms * 1e-3) / 1e9
    moe_v2 = {"us": round(ms * 1e3, 3), "weight_bytes": wbytes, "weight_gbs": round(gbs, 1),
              "frac_hbm": round(gbs / hbm_gbs, 4)}
    pairs = list(zip(keep, keep2))
    calls = [(lambda s=s_, d=d_: lib.qmm_nvfp4_repack_v2(h, s.data_ptr(), d.data_ptr(), n_ff, in_f, sptr))
             for s_, d_ in pairs]
    ms = _time_calls(torch, stream, calls, len(calls))
    gbs = 2 * mat_bytes / (ms * 1e-3) / 1e9
    repack = {"m": n_ff, "k": in_f, "us": round(ms * 1e3, 3), "bytes": 2 * mat_bytes, "gbs": round(gbs, 1),
              "frac_hbm": round(gbs / hbm_gbs, 4)}
    del keep2, tables2
    return moe_v2, repack


def run_sub_benches(q, lib, h, torch, synth, stream, hbm_gbs):
    sptr = stream.cuda_stream
    out = {"gemv": [], "moe": None, "moe_v2": None, "repack_v2": None, "moe_down": None, "dequant": []}
    # GEMV: rotate over enough weight copies to exceed L2 several times
    for fmt in ("q4_k", "q8_0"):
        for m, k in ((4608, 1024), (1024, 4608)):
            rb = q.qmm_row_bytes(fmt, k)
            wbytes = m * rb
            w_np = synth.weights(fmt, m, k, wbytes)
            ncopy = max(2, math.ceil(400e6 / wbytes))
            ws = [torch.from_numpy(w_np).cuda() for _ in range(ncopy)]
            for n in (1, 2, 4, 8):
                x = torch.from_numpy(synth.activations(n, k)).cuda()
                d = torch.empty(n, m, dtype=torch.float32, device="cuda")
                calls = [(lambda wt=wt: lib.qmm_gemv(h, q.DTYPES[fmt], wt.data_ptr(), x.data_ptr(), d.data_ptr(),
                                                     m, k, n, sptr)) for wt in ws]
                ms = _time_calls(torch, stream, calls, 2 * ncopy)
                gbs = wbytes / (ms * 1e-3) / 1e9
                out["gemv"].append({"dtype": fmt, "m": m, "k": k, "n": n, "us": round(ms * 1e3, 3),
                                    "weight_gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm_gbs, 4)})
            del ws
    # MoE gate/up: 8 experts x {gate, up}, 4 rotated copies of the weight set
    in_f, n_ff, n_used = 4096, 2048, 8
    n_pairs = n_used
    rb = q.qmm_row_bytes("nvfp4", in_f)
    keep, tables = [], []
    for c in range(4):
        ptrs = []
        for p in range(2):
            for j in range(n_pairs):
                t = torch.from_numpy(synth.nvfp4_rows(synth.nvfp4_matrix_seed(c, j, p), n_ff, in_f)).cuda()
                keep.append(t)
                ptrs.append(t.data_ptr())
        tables.append(torch.tensor(ptrs + [0] * n_pairs, dtype=torch.int64, device="cuda"))
    scales = torch.tensor([0.5 + 0.01 * i for i in range(3 * n_pairs)], dtype=torch.float32, device="cuda")
    x = torch.from_numpy(synth.activations(1, in_f)).cuda()
    y = torch.empty(2, n_pairs, n_ff, dtype=torch.float32, device="cuda")
    calls = [(lambda tb=tb: lib.qmm_moe_gemv(h, q.NVFP4, tb.data_ptr(), scales.data_ptr(), x.data_ptr(),
                                             y.data_ptr(), in_f, n_ff, n_used, 1, sptr)) for tb in tables]
    ms = _time_calls(torch, stream, calls, 40)
    wbytes = 2 * n_pairs * n_ff * rb
    gbs = wbytes / (ms * 1e-3) / 1e9
    out["moe"] = {"us": round(ms * 1e3, 3), "weight_bytes": wbytes, "weight_gbs": round(gbs, 1),
                  "frac_hbm": round(gbs / hbm_gbs, 4)}
    # the same call on V2 rows (codes, then the scale stream) made by the
    # library's repack, and the repack itself (read + write of each matrix)
    try:
        out["moe_v2"], out["repack_v2"] = _moe_v2_sub(q, lib, h, torch, stream, keep, scales, x, y, in_f, n_ff,
                                                      n_used, n_pairs, wbytes, hbm_gbs)
    except Exception as exc:  # reported in the JSON line, never fatal to the headline measurement
        out["moe_v2"] = {"error": f"{type(exc).__name__}: {exc}"}
    del keep, tables
    # MoE down projection: 8 experts of [gin 4096][n_ff 2048], per-pair
    # activations, pairs summed into y; 6 rotated copies of the weight set
    gin, n_ff_d = 4096, 2048
    rb = q.qmm_row_bytes("nvfp4", n_ff_d)
    keep, tables = [], []
    for c in range(6):
        ptrs = []
        for j in range(n_pairs):
            t = torch.from_numpy(synth.nvfp4_rows(synth.nvfp4_matrix_seed(c, j, 2), gin, n_ff_d)).cuda()
            keep.append(t)
            ptrs.append(t.data_ptr())
        tables.append(torch.tensor(ptrs, dtype=torch.int64, device="cuda"))
    hact = torch.from_numpy(synth.activations(n_pairs, n_ff_d, seed=1234)).cuda()
    yd = torch.empty(1, gin, dtype=torch.float32, device="cuda")
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, 1)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    calls = [(lambda tb=tb: lib.qmm_moe_down(h, q.NVFP4, tb.data_ptr(), scales.data_ptr(), hact.data_ptr(),
                                             yd.data_ptr(), n_ff_d, gin, n_used, 1, ws.data_ptr(), wsb, sptr))
             for tb in tables]
    ms = _time_calls(torch, stream, calls, 48)
    wbytes = n_pairs * gin * rb
    gbs = wbytes / (ms * 1e-3) / 1e9
    out["moe_down"] = {"us": round(ms * 1e3, 3), "weight_bytes": wbytes, "weight_gbs": round(gbs, 1),
                       "frac_hbm": round(gbs / hbm_gbs, 4), "launches_per_call": 2}
    del keep, tables
    # dequant: read packed + write f32
    for fmt, m, k in (("q4_k", 4608, 1024), ("q6_k", 4608, 1024), ("nvfp4", 2048, 4096)):
        rb = q.qmm_row_bytes(fmt, k)
        w = torch.from_numpy(synth.weights(fmt, m, k, m * rb)).cuda()
        outs = [torch.empty(m, k, dtype=torch.float32, device="cuda") for _ in range(8)]
        calls = [(lambda o=o: lib.qmm_dequant(h, q.DTYPES[fmt], w.data_ptr(), o.data_ptr(), m, k,
                                              1.0, sptr)) for o in outs]
        ms = _time_calls(torch, stream, calls, 32)
        tot = m * rb + 4 * m * k
        gbs = tot / (ms * 1e-3) / 1e9
        out["dequant"].append({"dtype": fmt, "m": m, "k": k, "us": round(ms * 1e3, 3), "gbs": round(gbs, 1),
                               "frac_hbm": round(gbs / hbm_gbs, 4)})
        if fmt == "nvfp4":  # the same rows as V2 (codes, then the scale stream), made by the library's repack
            try:
                w2 = torch.empty_like(w)
                if lib.qmm_nvfp4_repack_v2(h, w.data_ptr(), w2.data_ptr(), m, k, sptr) != 0:
                    raise RuntimeError("qmm_nvfp4_repack_v2 refused the call")
                calls = [(lambda o=o: lib.qmm_dequant(h, q.NVFP4_V2, w2.data_ptr(), o.data_ptr(), m, k,
                                                      1.0, sptr)) for o in outs]
                ms = _time_calls(torch, stream, calls, 32)
                gbs = tot / (ms * 1e-3) / 1e9
                out["dequant"].append({"dtype": "nvfp4_v2", "m": m, "k": k, "us": round(ms * 1e3, 3),
                                       "gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm_gbs, 4)})
            except Exception as exc:
                out["dequant"].append({"dtype": "nvfp4_v2", "error": f"{type(exc).__name__}: {exc}"})
    st = q.qmm_sync_status(h)
    if st != 0:
        raise RuntimeError(f"device status {st} in the sub-benchmarks")
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sub", action="store_true", help="skip the GEMV / MoE / dequant sub-benchmarks")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--only", default=None,
                    help="comma-separated shape labels to keep (profiling runs; not a headline workload)")
    ap.add_argument("--copies", type=int, default=COPIES,
                    help="rotated input copies (profiling runs use 1 to keep the device footprint small)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
