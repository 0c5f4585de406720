#!/usr/bin/env python
"""Benchmark of the quantized-weight projection matmul on one GB300.

A step is one 512-token prefill pass over the LFM2.5-350M projection shapes
(ffn_gate 4608x1024, ffn_down 1024x4608, conv_in 3072x1024, attn_out
1024x1024) with W in f32, Q4_0 and Q8_0: twelve qmm_gemm calls through the C
ABI, on seeded synthetic inputs already resident in HBM.  The headline value is
the step's total algorithmic FLOPs (2*m*k*n per GEMM) over its device time.
Inputs rotate over three copies (about 3 x 115 MB, more than the 129 MB L2), so
every step reads its operands from HBM.

The same run also times the k-quant prefill GEMMs (the same four shapes with W
in Q4_K and Q6_K, a second step of eight calls), the small-batch GEMV (n = 1,
2, 4, 8 on 4608x1024 and 1024x4608, Q4_K and Q8_0), the NVFP4 MoE gate/up GEMV
(8 experts x 2 planes of 2048x4096, four rotated weight copies), the MoE down
projection and the standalone dequant, and reports their GB/s (weight bytes,
and all bytes moved) against the measured HBM bandwidth.  Every duration is
the median over at least seven rounds.

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
DTYPES = ["f32", "q4_0", "q8_0"]      # the headline step
KQ_DTYPES = ["q4_k", "q6_k"]           # the k-quant step, timed beside it
N_TOKENS = 512
ROUNDS = 7
COPIES = 3
WORKLOAD = ("LFM2.5-350M 512-token prefill projections: ffn_gate 4608x1024, ffn_down 1024x4608, "
            "conv_in 3072x1024, attn_out 1024x1024; W in f32, q4_0, q8_0; n=512")
# nominal dense tensor-core rates (PFLOP/s): f16/bf16 2.25, tf32 1.1
TF32_OVER_F16 = 1.1 / 2.25
# DRAM bytes (read + write) per launch of the tensor-core GEMM kernel, the
# mean over the step's 12 launches, from one ncu capture of this workload (the
# dram__bytes_read.sum + dram__bytes_write.sum counters of every launch of one
# step).  It describes the kernel sources it was taken on; if they change, the
# bench reports null.
GEMM_TRAFFIC_SOURCES = ("gemv_dequant_gemm_gb300/csrc/gemm_tc.cu", "gemv_dequant_gemm_gb300/csrc/decode.cuh",
                        "gemv_dequant_gemm_gb300/csrc/common.cuh")
GEMM_TRAFFIC_SHA16 = "173e19dc9c087f66"
GEMM_TRAFFIC_BYTES = 9.075e6


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


def _oracle_sample(ins, entries_per_gemm, seed=0, threads=0, keep=None):
    """Time the oracle on `entries_per_gemm` output entries of each GEMM
    (threads = 0: the OpenMP default, all host cores); with a list `keep`,
    append (label, fmt, n indices, m indices, values, sum|W*X|) per GEMM."""
    import oracle
    rng = np.random.default_rng(seed)
    flops, t = 0.0, 0.0
    for label, fmt, m, k, w, x in ins:
        ni = rng.integers(0, N_TOKENS, entries_per_gemm)
        mj = rng.integers(0, m, entries_per_gemm)
        t0 = time.perf_counter()
        ref, am = oracle.matmul_entries(fmt, w, x, m, k, N_TOKENS, ni, mj, threads=threads)
        t += time.perf_counter() - t0
        flops += 2.0 * k * entries_per_gemm
        if keep is not None:
            keep.append((label, fmt, ni, mj, ref, am))
    return flops, t


def _check_timed_outputs(gemms, kept):
    """The timed step's outputs (buffer copy 0, which every copy equals) at
    the oracle's sampled entries, against the tensor-core tolerance
    2e-3 * sum|W*X| + 1e-6."""
    by = {(g["label"], g["fmt"]): g for g in gemms}
    worst, bad, total = 0.0, 0, 0
    for label, fmt, ni, mj, ref, am in kept:
        got = by[(label, fmt)]["copies"][0]["dst"].cpu().numpy().astype(np.float64)[ni, mj]
        ratio = np.abs(got - ref) / (2e-3 * am + 1e-6)
        ratio[~np.isfinite(got)] = np.inf
        worst = max(worst, float(ratio.max()))
        bad += int((ratio > 1.0).sum())
        total += ni.size
    return {"entries": total, "outside_tolerance": bad, "worst_err_over_tol": round(worst, 4), "ok": bad == 0,
            "what": "the timed step's outputs at the sampled entries against the f64 oracle, "
                    "tolerance 2e-3*sum|W*X| + 1e-6"}


def _oracle_calibrate(ins, budget_s, threads=0):
    flops, t = _oracle_sample(ins, 64, seed=99, threads=threads)
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


def _alg_bytes(q, fmt, m, k, n):
    """Algorithmic bytes of one product: packed W, f32 X and f32 dst, each once."""
    return m * q.qmm_row_bytes(fmt, k) + 4 * n * k + 4 * n * m


def _med(xs):
    return float(statistics.median(xs))


def _build_gemms(q, torch, synth, dtypes, shapes, copies_n):
    """Per GEMM: host arrays and `copies_n` rotated device copies of (W, X, dst, workspace)."""
    gemms = []
    for label, m, k in shapes:
        x_np = synth.activations(N_TOKENS, k)
        for fmt in dtypes:
            w_np = synth.weights(fmt, m, k, m * q.qmm_row_bytes(fmt, k))
            wsb = q.qmm_gemm_workspace_bytes(fmt, m, k, N_TOKENS)
            copies = []
            for _ in range(copies_n):
                copies.append({
                    "w": torch.from_numpy(w_np).cuda(), "x": torch.from_numpy(x_np).cuda(),
                    "dst": torch.empty(N_TOKENS, m, dtype=torch.float32, device="cuda"),
                    "ws": torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda"),
                })
            gemms.append({"label": label, "fmt": fmt, "m": m, "k": k, "wsb": wsb, "w_np": w_np, "x_np": x_np,
                          "copies": copies, "flops": 2.0 * m * k * N_TOKENS,
                          "bytes": _alg_bytes(q, fmt, m, k, N_TOKENS)})
    return gemms


class _Runner:
    """Launches qmm_gemm for the GEMMs of a step through the C ABI."""

    def __init__(self, q, lib, h, torch, stream, gemms, copies_n):
        self.q, self.lib, self.h, self.torch, self.stream = q, lib, h, torch, stream
        self.sptr = stream.cuda_stream
        self.gemms, self.copies_n = gemms, copies_n

    def launch(self, g, c):
        b = g["copies"][c]
        st = self.lib.qmm_gemm(self.h, self.q.DTYPES[g["fmt"]], b["w"].data_ptr(), b["x"].data_ptr(),
                               b["dst"].data_ptr(), g["m"], g["k"], N_TOKENS,
                               b["ws"].data_ptr() if g["wsb"] else None, g["wsb"], self.sptr)
        if st:
            raise self.q.QmmError(st, "qmm_gemm")

    def step(self, c, evs=None):
        for i, g in enumerate(self.gemms):
            if evs is not None:
                evs[i][0].record(self.stream)
            self.launch(g, c)
            if evs is not None:
                evs[i][1].record(self.stream)

    def warm(self, n):
        for i in range(n):
            self.step(i % self.copies_n)

    def time_steps(self, steps):
        """Device time (ms) of each of `steps` steps, each its GEMMs back to back.
        A device-side sleep queued before each step keeps the GPU busy while
        the host enqueues it, so the events time kernels, not launch gaps."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for s in range(steps):
            torch.cuda._sleep(1_500_000)
            evs[s][0].record(self.stream)
            self.step(s % self.copies_n)
            evs[s][1].record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def time_calls(self, steps):
        """Per-call durations [steps][gemm] (ms): an event pair around every
        call, so these are single-call latencies (the events keep consecutive
        calls from overlapping)."""
        torch = self.torch
        evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in self.gemms]
               for _ in range(steps)]
        for s in range(steps):
            torch.cuda._sleep(1_500_000)
            self.step(s % self.copies_n, evs[s])
        torch.cuda.synchronize()
        return np.array([[a.elapsed_time(b) for a, b in row] for row in evs])


def _per_gemm(gemms, call_ms, f16_tflops, tf32_tflops, hbm_gbs):
    """Per GEMM: median single-call time, TFLOP/s, and the fraction of its
    roofline max(FLOPs at the tensor peak of its operand type, bytes at HBM)."""
    out = []
    for i, g in enumerate(gemms):
        us = _med(call_ms[:, i]) * 1e3
        peak = tf32_tflops if g["fmt"] == "f32" else f16_tflops
        t_tensor = g["flops"] / (peak * 1e12)
        t_hbm = g["bytes"] / (hbm_gbs * 1e9)
        ideal = max(t_tensor, t_hbm)
        out.append({"shape": g["label"], "dtype": g["fmt"], "us": round(us, 3),
                    "tflops": round(g["flops"] / (us * 1e-6) / 1e12, 2),
                    "bound": "tensor" if t_tensor >= t_hbm else "hbm",
                    "ideal_us": round(ideal * 1e6, 3), "frac": round(ideal / (us * 1e-6), 4)})
    return out


def _per_dtype(gemms, call_ms, dtypes):
    res = {}
    for f in dtypes:
        idx = [i for i, g in enumerate(gemms) if g["fmt"] == f]
        if not idx:
            continue
        fl = sum(gemms[i]["flops"] for i in idx)
        tt = sum(_med(call_ms[:, i]) for i in idx) * 1e-3
        res[f] = round(fl / tt / 1e12, 2)
    return res


def run_ours(args):
    import torch

    import gemv_dequant_gemm_gb300 as q
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

    # ---- prefill workload: COPIES sets of (W, X, dst, workspace) ----
    copies_n = max(1, args.copies)
    shapes = [s for s in SHAPES if not args.only or s[0] in args.only.split(",")]
    gemms = _build_gemms(q, torch, synth, DTYPES, shapes, copies_n)
    run = _Runner(q, lib, h, torch, stream, gemms, copies_n)
    flops_step = sum(g["flops"] for g in gemms)
    copy_mb = sum(b.numel() * b.element_size() for g in gemms for b in g["copies"][0].values()) / 1e6

    # launches of our kernels per step: x->f16 + tensor-core GEMM for packed W, one for f32 W
    # (all launched with programmatic dependent launch, so consecutive calls overlap)
    launches_per_step = sum(1 if g["fmt"] == "f32" else 2 for g in gemms)

    run.warm(args.warmup)
    torch.cuda.synchronize()
    if q.qmm_sync_status(h) != 0:
        raise RuntimeError("device status set during warm-up")

    # ---- timed region: K steps, each its 12 GEMMs back to back ----
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.25)
    wall0 = time.perf_counter()
    step_ms = run.time_steps(args.steps)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    status = q.qmm_sync_status(h)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    # per-GEMM durations: the same steps with an event pair around every call
    kb = max(ROUNDS, min(100, args.steps))
    call_ms = run.time_calls(kb)
    ms_per_step = slowest_rank_ms(_med(step_ms), world, "cuda")
    value = job_tflops(world, flops_step, ms_per_step)

    per_gemm = _per_gemm(gemms, call_ms, f16_tflops, tf32_tflops, hbm_gbs)
    per_dtype = _per_dtype(gemms, call_ms, DTYPES)
    # dominant kernel: the tensor-core GEMM (qmm_gemm, n=512), all its launches.
    # Its roofline is per GEMM max(FLOPs at the tensor peak of its operand
    # type, algorithmic bytes at HBM); `peak` is the step's FLOPs over the sum
    # of those ideal times, so frac = sum(ideal) / sum(measured).
    tot_t = sum(_med(call_ms[:, i]) for i in range(len(gemms))) * 1e-3
    ideal_t = sum(p["ideal_us"] for p in per_gemm) * 1e-6
    achieved = flops_step / tot_t / 1e12
    peak_eff = flops_step / ideal_t / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak_eff, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak_eff, 4), "traffic": _gemm_traffic(),
                "traffic_unit": "bytes per gemm_tc_kernel launch (DRAM read + write, ncu)",
                "kernel": "qmm_gemm tensor-core path (x_to_f16 + gemm_tc); per-call event-timed durations, "
                          f"median of {kb} steps",
                "peak_source": f"{peak_src}: bf16 dense {f16_tflops} TFLOP/s (f16 operands), tf32 = "
                               f"x{TF32_OVER_F16:.3f} nominal ratio, HBM {hbm_gbs} GB/s; per GEMM the slower of "
                               "FLOPs at its tensor peak and algorithmic bytes at HBM"}

    # ---- the same step replayed from a CUDA graph (one graph: a step on each
    # buffer copy); reported beside the stream-issued headline ----
    graph_step = None
    if not args.no_graph:
        try:
            gstream = torch.cuda.Stream()
            gstream.wait_stream(stream)
            grun = _Runner(q, lib, h, torch, gstream, gemms, copies_n)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gstream):
                for c in range(copies_n):
                    grun.step(c)
            torch.cuda.synchronize()
            reps = max(3, min(40, args.steps // copies_n))
            gevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            with torch.cuda.stream(gstream):
                graph.replay()  # warm
                for a, b in gevs:
                    torch.cuda._sleep(1_500_000)
                    a.record(gstream)
                    graph.replay()
                    b.record(gstream)
            torch.cuda.synchronize()
            if q.qmm_sync_status(h) != 0:
                raise RuntimeError("device status set during the graph replays")
            gms = _med([a.elapsed_time(b) / copies_n for a, b in gevs])
            graph_step = {"ms_per_step": round(gms, 5), "tflops": round(flops_step / (gms * 1e-3) / 1e12, 2),
                          "replays": reps, "steps_per_replay": copies_n,
                          "what": "the 12 GEMMs of a step on each of the rotated buffer copies captured once, "
                                  "replayed; median per step"}
            del graph
        except Exception as exc:  # reported, never fatal to the headline
            graph_step = {"error": f"{type(exc).__name__}: {exc}"}

    # ---- the k-quant step (config 2): the same shapes with W in Q4_K / Q6_K ----
    kquant = None
    if not args.no_kquant:
        try:
            kq = _build_gemms(q, torch, synth, KQ_DTYPES, shapes, copies_n)
            krun = _Runner(q, lib, h, torch, stream, kq, copies_n)
            krun.warm(max(3, args.warmup // 4))
            ksteps = max(ROUNDS, min(200, args.steps))
            kstep_ms = krun.time_steps(ksteps)
            kcall_ms = krun.time_calls(max(ROUNDS, min(100, args.steps)))
            if q.qmm_sync_status(h) != 0:
                raise RuntimeError("device status set in the k-quant step")
            kflops = sum(g["flops"] for g in kq)
            kpg = _per_gemm(kq, kcall_ms, f16_tflops, tf32_tflops, hbm_gbs)
            per_gemm += kpg
            per_dtype.update(_per_dtype(kq, kcall_ms, KQ_DTYPES))
            kquant = {"gemms": len(kq), "steps": ksteps, "ms_per_step": round(_med(kstep_ms), 5),
                      "tflops": round(kflops / (_med(kstep_ms) * 1e-3) / 1e12, 2),
                      "frac": round(sum(p["ideal_us"] for p in kpg) / (sum(p["us"] for p in kpg)), 4)}
            del kq, krun
        except Exception as exc:  # reported in the JSON line, never fatal to the headline measurement
            kquant = {"error": f"{type(exc).__name__}: {exc}"}

    # ---- e2e: host buffers through the public API ----
    e2e = None
    if not args.no_e2e:
        # every input of a step (W and X of the 12 GEMMs) in one pinned host
        # buffer, every result in another, each piece 256-byte aligned: one
        # copy up and one copy down per step; the copies overlap the kernels
        # of the neighbouring steps (inputs up on one stream, results down on
        # another, kernels waiting for their step's inputs), and a device
        # buffer set is refilled only after its last results are home
        def _al(v):
            return (v + 255) // 256 * 256
        offs, pos = [], 0
        for g in gemms:
            ow = pos
            pos = _al(pos + g["w_np"].nbytes)
            ox = pos
            pos = _al(pos + g["x_np"].nbytes)
            offs.append((ow, ox))
        in_bytes = pos
        douts, pos = [], 0
        for g in gemms:
            douts.append(pos)
            pos = _al(pos + N_TOKENS * g["m"] * 4)
        out_bytes = pos
        hin = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        hout = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
        for g, (ow, ox) in zip(gemms, offs):
            hin[ow:ow + g["w_np"].nbytes].copy_(torch.from_numpy(g["w_np"].view(np.uint8).reshape(-1)))
            hin[ox:ox + g["x_np"].nbytes].copy_(torch.from_numpy(g["x_np"].view(np.uint8).reshape(-1)))
        din = [torch.empty(in_bytes, dtype=torch.uint8, device="cuda") for _ in range(copies_n)]
        dout = [torch.empty(out_bytes, dtype=torch.uint8, device="cuda") for _ in range(copies_n)]
        h2d = sum(g["w_np"].nbytes + g["x_np"].nbytes for g in gemms)
        d2h = sum(N_TOKENS * g["m"] * 4 for g in gemms)
        e2e_steps = max(3, min(20, args.steps))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        for rep in range(2):  # one untimed pass, then the timed one
            torch.cuda.synchronize()
            ev0.record(stream)
            s_in.wait_event(ev0)
            s_out.wait_event(ev0)
            home = {}
            for s in range(e2e_steps):
                c = s % copies_n
                if c in home:
                    s_in.wait_event(home[c])
                with torch.cuda.stream(s_in):
                    din[c].copy_(hin, non_blocking=True)
                up = torch.cuda.Event()
                up.record(s_in)
                stream.wait_event(up)
                base_in, base_out = din[c].data_ptr(), dout[c].data_ptr()
                for gi, g in enumerate(gemms):
                    ow, ox = offs[gi]
                    ws = g["copies"][c]["ws"]
                    st = lib.qmm_gemm(h, q.DTYPES[g["fmt"]], base_in + ow, base_in + ox, base_out + douts[gi],
                                      g["m"], g["k"], N_TOKENS, ws.data_ptr() if g["wsb"] else None, g["wsb"],
                                      stream.cuda_stream)
                    if st:
                        raise q.QmmError(st, "qmm_gemm")
                done = torch.cuda.Event()
                done.record(stream)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    hout.copy_(dout[c], non_blocking=True)
                home[c] = torch.cuda.Event()
                home[c].record(s_out)
            for ev in home.values():
                stream.wait_event(ev)
            ev1.record(stream)
            torch.cuda.synchronize()
        e2e_ms = slowest_rank_ms(ev0.elapsed_time(ev1) / e2e_steps, world, "cuda")
        e2e = {"value": round(job_tflops(world, flops_step, e2e_ms), 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
               "overlap": "each step's inputs packed in one pinned buffer and copied up in one copy on one "
                          "stream, its results down in one copy on another, kernels on the compute stream; "
                          "every copy of every step inside the timed region"}

    # ---- a6-a8, f1-f3: GEMV, MoE, dequant (GB/s vs HBM) ----
    sub = None if args.no_sub else run_sub_benches(q, lib, h, torch, synth, stream, hbm_gbs)

    # ---- CPU baseline: the oracle on a bounded sample, all cores and one core ----
    cpu = None
    if rank == 0 and not args.no_cpu:
        ins = _oracle_inputs()
        cores = _cores()  # before any one-thread run changes the OpenMP default
        entries = _oracle_calibrate(ins, 12.0, threads=cores)
        kept = []
        f, t = _oracle_sample(ins, entries, seed=7, threads=cores, keep=kept)
        entries1 = _oracle_calibrate(ins, 6.0, threads=1)
        f1, t1 = _oracle_sample(ins, entries1, seed=8, threads=1)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{entries} random output entries of each of the 12 GEMMs (f64 oracle, OpenMP, {t:.1f} s)",
               "single_thread": {"value": f1 / t1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                                 "sample": f"{entries1} random output entries of each of the 12 GEMMs "
                                           f"(f64 oracle, one thread, {t1:.1f} s)"},
               "cpu": _cpu_model(), "check": _check_timed_outputs(gemms, kept)}

    q.qmm_destroy(h)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16/tf32 operands, f32 accumulate",
            "data": "synthetic (seeded LCG / xorshift64 streams)",
            "config": {"workload": WORKLOAD, "n": N_TOKENS, "dtypes": DTYPES,
                       "gemms_per_step": len(gemms), "flops_per_step": flops_step,
                       "timing": f"median of {args.steps} per-step event pairs; mean "
                                 f"{float(np.mean(step_ms)):.5f} ms",
                       "l2": f"inputs rotated over {copies_n} copies of {copy_mb:.0f} MB (L2 129 MB)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "per_dtype_tflops": per_dtype, "per_gemm": per_gemm, "kquant_step": kquant, "graph_step": graph_step, "roofline": roofline,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk, "timed_wall_s": round(wall, 3), "sub": sub,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def _time_calls(torch, stream, calls, reps, rounds=ROUNDS):
    """Device time (ms) per call of calls[i % len(calls)]() over `reps`
    back-to-back launches, one event pair around each round of `reps` calls
    (so the launches overlap as they do in a model's stream, programmatic
    dependent launch included, and no per-call event splits them); the
    median over `rounds` rounds, with the smallest and largest.  A
    device-side sleep queued before each round keeps the GPU busy while the
    host enqueues it."""
    for i in range(min(reps, 3)):
        calls[i % len(calls)]()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(rounds)]
    for r in range(rounds):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(max(2_000_000, 20_000 * reps))
        evs[r][0].record(stream)
        for i in range(reps):
            calls[(r * reps + i) % len(calls)]()
        evs[r][1].record(stream)
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) / reps for a, b in evs]
    return _med(per), min(per), max(per)


def _rate(label_bytes, ms, hbm_gbs):
    gbs = label_bytes / (ms * 1e-3) / 1e9
    return round(gbs, 1), round(gbs / hbm_gbs, 4)


def _moe_v2_sub(q, lib, h, torch, stream, keep, scales, x, y, in_f, n_ff, n_used, n_pairs, wbytes, tbytes, hbm_gbs):
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
    ms, lo, hi = _time_calls(torch, stream, calls, 40)
    wg, wf = _rate(wbytes, ms, hbm_gbs)
    tg, tf = _rate(tbytes, ms, hbm_gbs)
    moe_v2 = {"us": round(ms * 1e3, 3), "us_min": round(lo * 1e3, 3), "us_max": round(hi * 1e3, 3),
              "weight_bytes": wbytes, "weight_gbs": wg, "frac_hbm": wf, "total_bytes": tbytes, "total_gbs": tg,
              "frac_hbm_total": tf}
    pairs = list(zip(keep, keep2))
    calls = [(lambda s=s_, d=d_: lib.qmm_nvfp4_repack_v2(h, s.data_ptr(), d.data_ptr(), n_ff, in_f, sptr))
             for s_, d_ in pairs]
    ms, lo, hi = _time_calls(torch, stream, calls, len(calls))
    g, f = _rate(2 * mat_bytes, ms, hbm_gbs)
    repack = {"m": n_ff, "k": in_f, "us": round(ms * 1e3, 3), "bytes": 2 * mat_bytes, "gbs": g, "frac_hbm": f}
    del keep2, tables2
    return moe_v2, repack


def _moe_q8_sub(q, lib, h, torch, stream, tables, scales, x, in_f, n_ff, n_used, n_pairs, wbytes, hbm_gbs):
    sptr = stream.cuda_stream
    qd = torch.empty(1, in_f, dtype=torch.int8, device="cuda")
    dd = torch.empty(1, in_f // 32, dtype=torch.float32, device="cuda")
    y = torch.empty(2, n_pairs, n_ff, dtype=torch.float32, device="cuda")

    def quant():
        return lib.qmm_quantize_q8_1(h, x.data_ptr(), qd.data_ptr(), dd.data_ptr(), 1, in_f, sptr)

    def gemv(tb):
        return lib.qmm_moe_gemv_q8(h, q.NVFP4, tb.data_ptr(), scales.data_ptr(), qd.data_ptr(), dd.data_ptr(),
                                   y.data_ptr(), in_f, n_ff, n_used, 1, sptr)
    def fused(tb):
        return lib.qmm_moe_gemv_q8_fused(h, q.NVFP4, tb.data_ptr(), scales.data_ptr(), x.data_ptr(), y.data_ptr(),
                                         in_f, n_ff, n_used, 1, sptr)
    if quant() != 0 or gemv(tables[0]) != 0 or fused(tables[0]) != 0:
        raise RuntimeError("qmm_quantize_q8_1 / qmm_moe_gemv_q8 / qmm_moe_gemv_q8_fused refused the call")
    res = {}
    for label, calls, launches in (
            ("with_quantize", [(lambda tb=tb: quant() or gemv(tb)) for tb in tables], 2),
            ("fused", [(lambda tb=tb: fused(tb)) for tb in tables], 1),
            ("kernel_only", [(lambda tb=tb: gemv(tb)) for tb in tables], 1)):
        ms, lo, hi = _time_calls(torch, stream, calls, 40)
        wg, wf = _rate(wbytes, ms, hbm_gbs)
        res[label] = {"us": round(ms * 1e3, 3), "us_min": round(lo * 1e3, 3), "us_max": round(hi * 1e3, 3),
                      "weight_gbs": wg, "frac_hbm": wf, "launches_per_call": launches}
    res["weight_bytes"] = wbytes
    return res


def run_sub_benches(q, lib, h, torch, synth, stream, hbm_gbs):
    sptr = stream.cuda_stream
    out = {"timing": f"median over {ROUNDS} rounds of back-to-back calls (weights rotated through more "
                     "than 2x the L2 size); us_l2_warm: the same calls on one weight buffer, L2-resident",
           "gemv": [], "moe": None, "moe_q8": None, "moe_v2": None, "repack_v2": None, "moe_down": None,
           "moe_down_q8": None, "dequant": [], "fp4": None}
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
                ms, lo, hi = _time_calls(torch, stream, calls, ncopy)
                ms_warm, _, _ = _time_calls(torch, stream, calls[:1], ncopy)  # one weight buffer, L2-resident
                tbytes = _alg_bytes(q, fmt, m, k, n)
                wg, wf = _rate(wbytes, ms, hbm_gbs)
                tg, tf = _rate(tbytes, ms, hbm_gbs)
                out["gemv"].append({"dtype": fmt, "m": m, "k": k, "n": n, "us": round(ms * 1e3, 3),
                                    "us_min": round(lo * 1e3, 3), "us_max": round(hi * 1e3, 3),
                                    "weight_gbs": wg, "frac_hbm": wf, "total_gbs": tg, "frac_hbm_total": tf,
                                    "us_l2_warm": round(ms_warm * 1e3, 3)})
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
    ms, lo, hi = _time_calls(torch, stream, calls, 40)
    wbytes = 2 * n_pairs * n_ff * rb
    tbytes = wbytes + 4 * in_f + 2 * n_pairs * n_ff * 4 + 2 * n_pairs * (8 + 4)
    wg, wf = _rate(wbytes, ms, hbm_gbs)
    tg, tf = _rate(tbytes, ms, hbm_gbs)
    ms_warm, _, _ = _time_calls(torch, stream, calls[:1], 40)  # one weight set (75.5 MB), L2-resident
    out["moe"] = {"us": round(ms * 1e3, 3), "us_min": round(lo * 1e3, 3), "us_max": round(hi * 1e3, 3),
                  "weight_bytes": wbytes, "weight_gbs": wg, "frac_hbm": wf, "total_bytes": tbytes,
                  "total_gbs": tg, "frac_hbm_total": tf, "us_l2_warm": round(ms_warm * 1e3, 3)}
    # the same products on int8 (Q8_1) activations: the quantizer and the
    # dp4a kernel, two launches per call, and the kernel alone
    try:
        out["moe_q8"] = _moe_q8_sub(q, lib, h, torch, stream, tables, scales, x, in_f, n_ff, n_used, n_pairs,
                                    wbytes, hbm_gbs)
    except Exception as exc:  # reported in the JSON line, never fatal to the headline measurement
        out["moe_q8"] = {"error": f"{type(exc).__name__}: {exc}"}
    # the same call on V2 rows (codes, then the scale stream) made by the
    # library's repack, and the repack itself (read + write of each matrix)
    try:
        out["moe_v2"], out["repack_v2"] = _moe_v2_sub(q, lib, h, torch, stream, keep, scales, x, y, in_f, n_ff,
                                                      n_used, n_pairs, wbytes, tbytes, hbm_gbs)
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
    ms, lo, hi = _time_calls(torch, stream, calls, 48)
    wbytes = n_pairs * gin * rb
    # + activations and y: at this shape (n_ff 2048, 8 pairs) one grouped
    # kernel sums each token's pairs itself, with no products in the workspace
    tbytes = wbytes + 4 * n_pairs * n_ff_d + 4 * gin
    wg, wf = _rate(wbytes, ms, hbm_gbs)
    tg, tf = _rate(tbytes, ms, hbm_gbs)
    out["moe_down"] = {"us": round(ms * 1e3, 3), "us_min": round(lo * 1e3, 3), "us_max": round(hi * 1e3, 3),
                       "weight_bytes": wbytes, "weight_gbs": wg, "frac_hbm": wf, "total_bytes": tbytes,
                       "total_gbs": tg, "frac_hbm_total": tf, "launches_per_call": 1}
    try:  # on int8 (Q8_1) activations: quantizer, dp4a kernel, combine
        qd = torch.empty(n_pairs, n_ff_d, dtype=torch.int8, device="cuda")
        dd = torch.empty(n_pairs, n_ff_d // 32, dtype=torch.float32, device="cuda")

        def down_q8(tb):
            st = lib.qmm_quantize_q8_1(h, hact.data_ptr(), qd.data_ptr(), dd.data_ptr(), n_pairs, n_ff_d, sptr)
            return st or lib.qmm_moe_down_q8(h, q.NVFP4, tb.data_ptr(), scales.data_ptr(), qd.data_ptr(),
                                             dd.data_ptr(), yd.data_ptr(), n_ff_d, gin, n_used, 1, ws.data_ptr(),
                                             wsb, sptr)
        def down_q8_fused(tb):
            return lib.qmm_moe_down_q8_fused(h, q.NVFP4, tb.data_ptr(), scales.data_ptr(), hact.data_ptr(),
                                             yd.data_ptr(), n_ff_d, gin, n_used, 1, ws.data_ptr(), wsb, sptr)
        calls = [(lambda tb=tb: down_q8(tb)) for tb in tables]
        if calls[0]() != 0 or down_q8_fused(tables[0]) != 0:
            raise RuntimeError("qmm_moe_down_q8 / qmm_moe_down_q8_fused refused the call")
        ms, lo, hi = _time_calls(torch, stream, calls, 48)
        wg, wf = _rate(wbytes, ms, hbm_gbs)
        out["moe_down_q8"] = {"us": round(ms * 1e3, 3), "us_min": round(lo * 1e3, 3), "us_max": round(hi * 1e3, 3),
                              "weight_bytes": wbytes, "weight_gbs": wg, "frac_hbm": wf, "launches_per_call": 3}
        ms, lo, hi = _time_calls(torch, stream, [(lambda tb=tb: down_q8_fused(tb)) for tb in tables], 48)
        wg, wf = _rate(wbytes, ms, hbm_gbs)
        out["moe_down_q8"]["fused"] = {"us": round(ms * 1e3, 3), "us_min": round(lo * 1e3, 3),
                                       "us_max": round(hi * 1e3, 3), "weight_gbs": wg, "frac_hbm": wf,
                                       "launches_per_call": 2}
    except Exception as exc:
        out["moe_down_q8"] = {"error": f"{type(exc).__name__}: {exc}"}
    del keep, tables
    # dequant: read packed + write f32
    for fmt, m, k in (("q4_0", 4608, 1024), ("q8_0", 4608, 1024), ("q4_k", 4608, 1024), ("q6_k", 4608, 1024),
                      ("nvfp4", 2048, 4096)):
        rb = q.qmm_row_bytes(fmt, k)
        w = torch.from_numpy(synth.weights(fmt, m, k, m * rb)).cuda()
        outs = [torch.empty(m, k, dtype=torch.float32, device="cuda") for _ in range(8)]
        calls = [(lambda o=o: lib.qmm_dequant(h, q.DTYPES[fmt], w.data_ptr(), o.data_ptr(), m, k,
                                              1.0, sptr)) for o in outs]
        ms, lo, hi = _time_calls(torch, stream, calls, 32)
        tot = m * rb + 4 * m * k
        g, f = _rate(tot, ms, hbm_gbs)
        out["dequant"].append({"dtype": fmt, "m": m, "k": k, "us": round(ms * 1e3, 3), "gbs": g, "frac_hbm": f})
        if fmt == "nvfp4":  # the same rows as V2 (codes, then the scale stream), made by the library's repack
            try:
                w2 = torch.empty_like(w)
                if lib.qmm_nvfp4_repack_v2(h, w.data_ptr(), w2.data_ptr(), m, k, sptr) != 0:
                    raise RuntimeError("qmm_nvfp4_repack_v2 refused the call")
                calls = [(lambda o=o: lib.qmm_dequant(h, q.NVFP4_V2, w2.data_ptr(), o.data_ptr(), m, k,
                                                      1.0, sptr)) for o in outs]
                ms, lo, hi = _time_calls(torch, stream, calls, 32)
                g, f = _rate(tot, ms, hbm_gbs)
                out["dequant"].append({"dtype": "nvfp4_v2", "m": m, "k": k, "us": round(ms * 1e3, 3), "gbs": g,
                                       "frac_hbm": f})
            except Exception as exc:
                out["dequant"].append({"dtype": "nvfp4_v2", "error": f"{type(exc).__name__}: {exc}"})
    try:
        out["fp4"] = _fp4_sub(q, lib, h, torch, synth, stream, hbm_gbs)
    except Exception as exc:  # reported in the JSON line, never fatal to the headline measurement
        out["fp4"] = {"error": f"{type(exc).__name__}: {exc}"}
    st = q.qmm_sync_status(h)
    if st != 0:
        raise RuntimeError(f"device status {st} in the sub-benchmarks")
    return out


# nominal dense FP4 (NVFP4 block-scaled) over bf16 tensor rate: 13.5 / 2.25
FP4_OVER_BF16 = 13.5 / 2.25


def _fp4_sub(q, lib, h, torch, synth, stream, hbm_gbs):
    """The block-scaled FP4 prefill on the four 512-token shapes: weights from
    the NVFP4 stream repacked to V2 rows by the library, each call quantizing
    its f32 activation (qmm_quantize_nvfp4) and running qmm_gemm_fp4."""
    sptr = stream.cuda_stream
    _, f16_tflops, _ = _peaks()
    fp4_tflops = f16_tflops * FP4_OVER_BF16
    copies = 4
    items = []
    for label, m, k in SHAPES:
        rb = q.qmm_row_bytes("nvfp4_v2", k)
        v1 = torch.from_numpy(synth.nvfp4_rows(0x4F00 + m, m, k)).cuda()
        sets = []
        for _ in range(copies):
            w2 = torch.empty(m * rb, dtype=torch.uint8, device="cuda")
            if lib.qmm_nvfp4_repack_v2(h, v1.data_ptr(), w2.data_ptr(), m, k, sptr) != 0:
                raise RuntimeError("qmm_nvfp4_repack_v2 refused the call")
            sets.append({"w": w2, "x": torch.from_numpy(synth.activations(N_TOKENS, k)).cuda(),
                         "xq": torch.empty(N_TOKENS * rb, dtype=torch.uint8, device="cuda"),
                         "d": torch.empty(N_TOKENS, m, dtype=torch.float32, device="cuda")})
        flops = 2.0 * m * k * N_TOKENS
        byts = m * rb + 4 * N_TOKENS * k + 2 * N_TOKENS * rb + 4 * N_TOKENS * m
        items.append({"label": label, "m": m, "k": k, "sets": sets, "flops": flops, "bytes": byts})

    def call(it, c):
        s = it["sets"][c]
        st = lib.qmm_quantize_nvfp4(h, s["x"].data_ptr(), s["xq"].data_ptr(), N_TOKENS, it["k"], sptr)
        st = st or lib.qmm_gemm_fp4(h, s["w"].data_ptr(), s["xq"].data_ptr(), s["d"].data_ptr(), it["m"], it["k"],
                                   N_TOKENS, sptr)
        if st:
            raise RuntimeError(f"fp4 call status {st}")

    for c in range(copies):
        for it in items:
            call(it, c)
    torch.cuda.synchronize()
    # per call (quantize + GEMM) with an event pair around each; then the
    # four calls back to back as a step
    steps = 50
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in items]
           for _ in range(steps)]
    for s_ in range(steps):
        torch.cuda._sleep(1_000_000)
        for i, it in enumerate(items):
            evs[s_][i][0].record(stream)
            call(it, s_ % copies)
            evs[s_][i][1].record(stream)
    torch.cuda.synchronize()
    per = []
    tot_us, tot_ideal = 0.0, 0.0
    for i, it in enumerate(items):
        us = _med([evs[s_][i][0].elapsed_time(evs[s_][i][1]) for s_ in range(steps)]) * 1e3
        t_t = it["flops"] / (fp4_tflops * 1e12)
        t_h = it["bytes"] / (hbm_gbs * 1e9)
        ideal = max(t_t, t_h) * 1e6
        tot_us += us
        tot_ideal += ideal
        per.append({"shape": it["label"], "us": round(us, 3), "tflops": round(it["flops"] / (us * 1e-6) / 1e12, 1),
                    "bound": "tensor" if t_t >= t_h else "hbm", "ideal_us": round(ideal, 3),
                    "frac": round(ideal / us, 4)})
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ms = []
    for s_ in range(steps):
        torch.cuda._sleep(1_000_000)
        ev0.record(stream)
        for it in items:
            call(it, s_ % copies)
        ev1.record(stream)
        torch.cuda.synchronize()
        step_ms.append(ev0.elapsed_time(ev1))
    fl = sum(it["flops"] for it in items)
    ms = _med(step_ms)
    return {"workload": "the four 512-token shapes, W NVFP4 V2 rows, X quantized to NVFP4 per call",
            "launches_per_call": 2, "per_gemm": per, "step_us": round(ms * 1e3, 3),
            "step_tflops": round(fl / (ms * 1e-3) / 1e12, 1),
            "frac": round(tot_ideal / tot_us, 4),
            "peak": f"FP4 {fp4_tflops:.0f} TFLOP/s = measured bf16 x {FP4_OVER_BF16:.0f} (nominal ratio); "
                    f"HBM {hbm_gbs} GB/s; per GEMM the slower of the two"}


def run_profile_gemv(args):
    """One GEMV shape called back to back (a profiling run: not a bench line)."""
    import torch

    import gemv_dequant_gemm_gb300 as q
    import synth
    fmt, m, k, n = args.profile_gemv.split(",")
    m, k, n = int(m), int(k), int(n)
    torch.cuda.set_device(0)
    h = q.qmm_create(0)
    w = torch.from_numpy(synth.weights(fmt, m, k, m * q.qmm_row_bytes(fmt, k))).cuda()
    x = torch.from_numpy(synth.activations(n, k)).cuda()
    d = torch.empty(n, m, dtype=torch.float32, device="cuda")
    for _ in range(args.steps + args.warmup):
        q.qmm_gemv(h, fmt, w, x, d, m, k, n)
    torch.cuda.synchronize()
    st = q.qmm_sync_status(h)
    q.qmm_destroy(h)
    print(json.dumps({"profile_gemv": args.profile_gemv, "calls": args.steps + args.warmup, "status": st}))
    return 0 if st == 0 else 1


def run_profile_moe(args):
    """The NVFP4 MoE gate/up call (f32 or Q8_1 activations) on one weight set,
    called back to back (a profiling run: not a bench line)."""
    import torch

    import gemv_dequant_gemm_gb300 as q
    import synth
    mode = args.profile_moe
    in_f, n_ff, n_used = 4096, 2048, 8
    torch.cuda.set_device(0)
    h = q.qmm_create(0)
    mats = [torch.from_numpy(synth.nvfp4_rows(synth.nvfp4_matrix_seed(0, j, p), n_ff, in_f)).cuda()
            for p in range(2) for j in range(n_used)]
    table = torch.tensor([m.data_ptr() for m in mats], dtype=torch.int64, device="cuda")
    scales = torch.tensor([0.5 + 0.01 * i for i in range(2 * n_used)], dtype=torch.float32, device="cuda")
    x = torch.from_numpy(synth.activations(1, in_f)).cuda()
    y = torch.empty(2, n_used, n_ff, dtype=torch.float32, device="cuda")
    qd = torch.empty(1, in_f, dtype=torch.int8, device="cuda")
    dd = torch.empty(1, in_f // 32, dtype=torch.float32, device="cuda")
    for _ in range(args.steps + args.warmup):
        if mode == "q8":
            q.qmm_quantize_q8_1(h, x, qd, dd, 1, in_f)
            q.qmm_moe_gemv_q8(h, "nvfp4", table, scales, qd, dd, y, in_f, n_ff, n_used, 1)
        else:
            q.qmm_moe_gemv(h, "nvfp4", table, scales, x, y, in_f, n_ff, n_used, 1)
    torch.cuda.synchronize()
    st = q.qmm_sync_status(h)
    q.qmm_destroy(h)
    print(json.dumps({"profile_moe": mode, "calls": args.steps + args.warmup, "status": st}))
    return 0 if st == 0 else 1


def run_profile_dequant(args):
    """One dequant call repeated (a profiling run: not a bench line)."""
    import torch

    import gemv_dequant_gemm_gb300 as q
    import synth
    fmt, m, k = args.profile_dequant.split(",")
    m, k = int(m), int(k)
    torch.cuda.set_device(0)
    h = q.qmm_create(0)
    w = torch.from_numpy(synth.weights(fmt, m, k, m * q.qmm_row_bytes(fmt, k))).cuda()
    out = torch.empty(m, k, dtype=torch.float32, device="cuda")
    for _ in range(args.steps + args.warmup):
        q.qmm_dequant(h, fmt, w, out, m, k)
    torch.cuda.synchronize()
    st = q.qmm_sync_status(h)
    q.qmm_destroy(h)
    print(json.dumps({"profile_dequant": args.profile_dequant, "status": st}))
    return 0 if st == 0 else 1


def run_profile_fp4(args):
    """The FP4 prefill (quantize + GEMM) of one 512-token shape repeated (a
    profiling run: not a bench line)."""
    import torch

    import gemv_dequant_gemm_gb300 as q
    import synth
    label = args.profile_fp4
    _, m, k = [s for s in SHAPES if s[0] == label][0]
    torch.cuda.set_device(0)
    h = q.qmm_create(0)
    rb = q.qmm_row_bytes("nvfp4_v2", k)
    v1 = torch.from_numpy(synth.nvfp4_rows(0x4F00 + m, m, k)).cuda()
    w2 = torch.empty(m * rb, dtype=torch.uint8, device="cuda")
    q.qmm_nvfp4_repack_v2(h, v1, w2, m, k)
    x = torch.from_numpy(synth.activations(N_TOKENS, k)).cuda()
    xq = torch.empty(N_TOKENS * rb, dtype=torch.uint8, device="cuda")
    d = torch.empty(N_TOKENS, m, dtype=torch.float32, device="cuda")
    for _ in range(args.steps + args.warmup):
        q.qmm_quantize_nvfp4(h, x, xq, N_TOKENS, k)
        q.qmm_gemm_fp4(h, w2, xq, d, m, k, N_TOKENS)
    torch.cuda.synchronize()
    st = q.qmm_sync_status(h)
    q.qmm_destroy(h)
    print(json.dumps({"profile_fp4": label, "status": st}))
    return 0 if st == 0 else 1


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sub", action="store_true", help="skip the GEMV / MoE / dequant sub-benchmarks")
    ap.add_argument("--no-kquant", action="store_true", help="skip the Q4_K / Q6_K prefill step")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay of the step")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--only", default=None,
                    help="comma-separated shape labels to keep (profiling runs; not a headline workload)")
    ap.add_argument("--copies", type=int, default=COPIES,
                    help="rotated input copies (profiling runs use 1 to keep the device footprint small)")
    ap.add_argument("--profile-gemv", default=None, metavar="FMT,M,K,N",
                    help="call one GEMV shape warmup+steps times and exit (profiling runs)")
    ap.add_argument("--profile-moe", default=None, choices=["f32", "q8"],
                    help="call the NVFP4 MoE gate/up (f32 or Q8_1 activations) warmup+steps times and exit")
    ap.add_argument("--profile-dequant", default=None, metavar="FMT,M,K",
                    help="call one dequant shape warmup+steps times and exit (profiling runs)")
    ap.add_argument("--profile-fp4", default=None, choices=[s[0] for s in SHAPES],
                    help="call the FP4 prefill of one 512-token shape warmup+steps times and exit")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.profile_gemv:
        return run_profile_gemv(args)
    if args.profile_moe:
        return run_profile_moe(args)
    if args.profile_dequant:
        return run_profile_dequant(args)
    if args.profile_fp4:
        return run_profile_fp4(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
