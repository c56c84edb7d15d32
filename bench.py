#!/usr/bin/env python
"""Benchmark of the quantized-GEMM hot path on GB300.

Headline workload: the dense W4A8 (MXFP4 x MXFP8, group-32 E8M0) GEMM at
(M, N, K) = (4096, 3072, 4096) and (4096, 14336, 4096); one step = both GEMMs through
qgemm_dense, inputs resident in HBM.  Metric: TFLOP/s (2 M N K per GEMM).  Other
workloads (W4A16 M=8 GEMV, M=1 decode sweep, MoE) are reported under "extra".

Timing: exactly K steps run back to back between one pair of CUDA events on the launching
stream (barrier + synchronize on both sides).  No step finds its inputs in L2: consecutive
steps read different copies of the inputs, with at least three times the L2 capacity in
rotation (a step's copies were last touched several hundred MB of traffic earlier).
Workloads made of short kernels are captured once as a CUDA graph of whole steps and the
graph is replayed, so that host launch overhead does not pose as device time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (float64 numpy) on a bounded sample of the same
workload on this host's cores.  Under torchrun every rank runs an independent replica
(the path has no exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import functools
import csv
import io
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

import synth  # noqa: E402

SHAPES = [(4096, 3072, 4096), (4096, 14336, 4096)]
METRIC = "W4A8/W4A16 GEMM TFLOPS and M=1 weight GB/s, % of GB300 roofline"
WORKLOAD = "dense W4A8 MXFP4xMXFP8 g32 (4096,3072,4096)+(4096,14336,4096)"


def flops_of(shapes):
    return sum(2.0 * m * n * k for m, n, k in shapes)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.out or "")) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- distributed
def dist_setup():
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
    """The slowest rank's value (NCCL on the GPUs; gloo on host tensors)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_rank_step, world, ms_per_step):
    """Every rank runs the same step on its own replica (weak scaling): the job's throughput
    is all ranks' FLOP over the slowest rank's step time."""
    return flop_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


# ----------------------------------------------------------------------------- our arm
class W4A8Problem:
    """One dense W4A8 GEMM with `replicas` copies of its inputs (weights, scales,
    activations); run(i) reads copy i mod replicas."""

    def __init__(self, M, N, K, cfg_id=1, replicas=1):
        import moe_qw_repack_gb300.qw as Q
        self.Q = Q
        p = synth.w4a8_problem(M, N, K, cfg_id=cfg_id)
        self.M, self.N, self.K = M, N, K
        self.desc = Q.qw_repack_query(Q.QW_W_MXFP4_G32, 1, N, K)
        wp, sp = Q.empty_packed(self.desc)
        err = Q.new_error_flag()
        Q.qw_repack(self.desc, torch.from_numpy(p["w_canon"]).cuda(),
                    torch.from_numpy(p["s_canon"]).cuda(), wp, sp, err)
        assert Q.qw_read_error(err) == 0
        self.A_host = torch.from_numpy(p["A"]).pin_memory()
        self.Asf_host = torch.from_numpy(p["A_sf"]).pin_memory()
        A, Asf = self.A_host.cuda(), self.Asf_host.cuda()
        self.copies = [(wp, sp, A, Asf)] + [(wp.clone(), sp.clone(), A.clone(), Asf.clone())
                                            for _ in range(replicas - 1)]
        self.C = torch.empty((M, N), dtype=torch.int16, device="cuda")
        self.C_host = torch.empty((M, N), dtype=torch.int16).pin_memory()
        self.err = Q.new_error_flag()
        # the workspace the call asks for (none for a dense call today; passed as a caller
        # should)
        self.wsn = Q.qgemm_workspace_size(self.desc, Q.QW_A_MXFP8_G32, M)
        self.ws = torch.empty(max(self.wsn, 16), dtype=torch.uint8, device="cuda")

    def run(self, i=0):
        Q = self.Q
        wp, sp, A, Asf = self.copies[i % len(self.copies)]
        Q.qgemm_dense(self.desc, wp, sp, Q.QW_A_MXFP8_G32, A, Asf, None, self.C, self.M, self.ws,
                      self.wsn, self.err)

    # end to end, two slots: slot k holds one step's activations and results on the device
    def _slot(self, k):
        if not hasattr(self, "_slots"):
            self._slots = []
            for j in range(2):
                A, Asf = self.copies[j % len(self.copies)][2:]
                if j >= len(self.copies):
                    A, Asf = A.clone(), Asf.clone()
                C = self.C if j == 0 else torch.empty_like(self.C)
                Ch = self.C_host if j == 0 else torch.empty_like(self.C_host).pin_memory()
                self._slots.append((A, Asf, C, Ch))
        return self._slots[k]

    def load_slot(self, k):
        """Pinned host activations and scales -> slot k (on the current stream)."""
        A, Asf, _, _ = self._slot(k)
        A.copy_(self.A_host, non_blocking=True)
        Asf.copy_(self.Asf_host, non_blocking=True)

    def run_slot(self, k, i):
        """The GEMM on slot k's activations with weight copy i (public call)."""
        Q = self.Q
        A, Asf, C, _ = self._slot(k)
        wp, sp = self.copies[i % len(self.copies)][:2]
        Q.qgemm_dense(self.desc, wp, sp, Q.QW_A_MXFP8_G32, A, Asf, None, C, self.M, self.ws,
                      self.wsn, self.err)

    def store_slot(self, k):
        """Slot k's BF16 result -> pinned host memory (on the current stream)."""
        _, _, C, Ch = self._slot(k)
        Ch.copy_(C, non_blocking=True)


def time_e2e_pipelined(probs, steps, warmup, world):
    """End-to-end time per step through the public call: every step copies its activations
    in from pinned host memory and its results out to pinned host memory.  Copies in run on
    one stream, the GEMMs on the current stream and copies out on a third, over two device
    slots, so a step's copies overlap the GEMMs of its neighbours (events order each slot's
    reuse).  Returns (ms per step, steps timed)."""
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    gemm_done = [torch.cuda.Event(), torch.cuda.Event()]
    out_done = [torch.cuda.Event(), torch.cuda.Event()]

    def step(i):
        k = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(gemm_done[k])  # the GEMMs two steps back are done with slot k
            for pr in probs:
                pr.load_slot(k)
            in_ready[k].record(s_in)
        comp.wait_event(in_ready[k])
        comp.wait_event(out_done[k])  # slot k's previous results have left the device
        for pr in probs:
            pr.run_slot(k, i)
        gemm_done[k].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(gemm_done[k])
            for pr in probs:
                pr.store_slot(k)
            out_done[k].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for i in range(steps):
        step(warmup + i)
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    b.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return max_over_ranks(a.elapsed_time(b) / steps, world), steps


def time_copies_only(probs, steps, world):
    """The same per-step host copies as time_e2e_pipelined with no GEMM: copies in on one
    stream, copies out on another, both directions at once.  Returns ms per step: the time
    the node's host link alone needs for a step's bytes."""
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def step(i):
        with torch.cuda.stream(s_in):
            for pr in probs:
                pr.load_slot(i % 2)
        with torch.cuda.stream(s_out):
            for pr in probs:
                pr.store_slot((i + 1) % 2)
    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for i in range(steps):
        step(i)
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    b.record(comp)
    torch.cuda.synchronize()
    return max_over_ranks(a.elapsed_time(b) / steps, world)


def l2_bytes():
    return int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0) or (126 << 20))


def replicas_for(step_bytes, cap=256):
    """Copies of a step's inputs so that at least 3 x L2 of them are in rotation."""
    need = -(-3 * l2_bytes() // max(1, int(step_bytes)))
    return int(max(1, min(cap, need)))


def time_region(fns, steps, warmup, world, graph_steps=0):
    """Warm up, then time exactly `steps` steps back to back between one pair of CUDA events
    on the current stream; step i runs f(i) for f in fns (i selects the input copy).  With
    graph_steps > 0 that many steps are captured once as a CUDA graph and replayed (the
    step count is rounded up to a whole number of replays).  Returns (ms per step, steps
    timed, graph used)."""
    for i in range(warmup):
        for f in fns:
            f(i)
    torch.cuda.synchronize()
    graph = None
    if graph_steps > 0:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="thread_local"):
                for i in range(graph_steps):
                    for f in fns:
                        f(i)
            graph.replay()
            torch.cuda.synchronize()
        except RuntimeError:
            graph = None
            torch.cuda.synchronize()
    reps = -(-steps // graph_steps) if graph is not None else steps
    n = reps * graph_steps if graph is not None else steps
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    if graph is not None:
        for _ in range(reps):
            graph.replay()
    else:
        for i in range(n):
            for f in fns:
                f(i)
    b.record()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return max_over_ranks(a.elapsed_time(b) / n, world), n, graph is not None


def extra_w4a16(steps, warmup, world, only=None):
    """Config 1 (M=8, N=K=2048 INT4) and the M=1 decode sweep: device time per GEMM (CUDA
    graph of back-to-back launches over weight copies that do not fit L2), weight GB/s."""
    import moe_qw_repack_gb300.qw as Q
    out = {}
    peaks, _ = measured_peaks()
    cases = [("cfg1_w4a16_m8_2048x2048_int4", 8, 2048, 2048, 4)]
    for bits in (4, 3):
        for (N, K) in [(14336, 4096), (4096, 14336), (4096, 4096)]:
            cases.append((f"cfg3_m1_{N}x{K}_int{bits}", 1, N, K, bits))
    # WnA16 formats with no workload of their own, on the first decode shape
    cases.append(("m1_14336x4096_int2", 1, 14336, 4096, 2))
    cases.append(("m1_14336x4096_int1", 1, 14336, 4096, 1))
    cases.append(("m1_14336x4096_fp4", 1, 14336, 4096, "fp4"))
    # few 16-row blocks and long K: the decode GEMV splits K across the CTAs of a cluster
    cases.append(("m1_1024x32768_int4_splitk", 1, 1024, 32768, 4))
    cases.append(("m1_512x16384_int4_splitk", 1, 512, 16384, 4))
    for name, M, N, K, bits in cases:
        if only and only not in name:
            continue
        if bits == "fp4":
            p = synth.fp4w_problem(M, N, K, cfg_id=2)
            wfmt, wbits = Q.QW_W_FP4E2M1_G128_BF16, 4
        else:
            p = synth.w4a16_problem(M, N, K, bits=bits, cfg_id=0 if M == 8 else 2)
            wfmt = {4: Q.QW_W_INT4_G128_BF16, 3: Q.QW_W_INT3_G128_BF16,
                    2: Q.QW_W_INT2_G128_BF16, 1: Q.QW_W_INT1_G128_BF16}[bits]
            wbits = bits
        d = Q.qw_repack_query(wfmt, 1, N, K)
        wp, sp = Q.empty_packed(d)
        Q.qw_repack(d, torch.from_numpy(p["w_canon"]).cuda(), torch.from_numpy(p["s_canon"]).cuda(), wp, sp)
        wbytes = N * K * wbits / 8 + N * (K // 128) * 2  # packed weights + BF16 scales
        R = replicas_for(wp.numel() + sp.numel())
        copies = [(wp, sp)] + [(wp.clone(), sp.clone()) for _ in range(R - 1)]
        A = torch.from_numpy(p["A"].view(np.int16)).cuda()
        C = torch.empty((M, N), dtype=torch.int16, device="cuda")
        wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, M)
        ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")

        def fn(i, copies=copies, d=d, A=A, C=C, M=M, ws=ws, wsn=wsn):
            w, s = copies[i % len(copies)]
            Q.qgemm_dense(d, w, s, Q.QW_A_BF16, A, None, None, C, M, ws, wsn)
        ms, n, graph = time_region([fn], max(steps, R), warmup, world, graph_steps=R)
        gbs = wbytes / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 2), "weight_GBps": round(gbs, 1),
                     "hbm_frac": round(gbs / peaks["hbm_gbs"], 3),
                     "tflops": round(2 * M * N * K / (ms * 1e-3) / 1e12, 3),
                     "launches": n, "weight_copies": R, "graph": graph}
        out[name].update(stream_read_reference(copies, steps, warmup, world, wbytes, peaks))
        del copies
        torch.cuda.empty_cache()
    return out


def stream_read_reference(copies, steps, warmup, world, nbytes, peaks):
    """A plain streaming read of the same packed weights (qw_stream_read), timed like the
    GEMV: a CUDA graph of back-to-back launches over the same copies.  'plain' launches in
    stream order; 'chained' as programmatic dependents with every load before the wait (the
    overlap a kernel that needs nothing from its predecessor can have; a GEMV must wait for
    its activations)."""
    import moe_qw_repack_gb300.qw as Q
    sink = torch.zeros(Q.QW_STREAM_READ_SINK_WORDS, dtype=torch.int32, device="cuda")
    res = {}
    for chained in (False, True):
        def rd(i, chained=chained):
            w, _ = copies[i % len(copies)]
            Q.qw_stream_read(w, w.numel(), sink, chained)
        ms, _, _ = time_region([rd], max(steps, len(copies)), warmup, world,
                               graph_steps=len(copies))
        wb = copies[0][0].numel()
        key = "stream_read_chained_frac" if chained else "stream_read_frac"
        res[key] = round(wb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)
    return res


def extra_fp8w(steps, warmup, world, only=None):
    """FP8-weight WnA16 (E4M3 codes, BF16 group-128 scales, BF16 activations): the M=1 decode
    shapes (weight GB/s of codes + scales) and one large-M dense GEMM on the tcgen05 path
    (TFLOP/s against the measured BF16 burst: the MMAs are BF16)."""
    import moe_qw_repack_gb300.qw as Q
    out = {}
    peaks, _ = measured_peaks()
    for name, M, N, K in [("fp8w_m1_14336x4096", 1, 14336, 4096),
                          ("fp8w_m1_4096x14336", 1, 4096, 14336),
                          ("fp8w_4096x14336x4096", 4096, 14336, 4096)]:
        if only and only not in name:
            continue
        p = synth.fp8w_problem(M, N, K, cfg_id=970)
        d = Q.qw_repack_query(Q.QW_W_FP8E4M3_G128_BF16, 1, N, K)
        wp, sp = Q.empty_packed(d)
        Q.qw_repack(d, torch.from_numpy(p["w_canon"]).cuda(), torch.from_numpy(p["s_canon"]).cuda(),
                    wp, sp)
        A = torch.from_numpy(p["A"].view(np.int16)).cuda()
        step_in = d.w_bytes + d.s_bytes + (A.numel() * 2 if M > 1 else 0)
        R = replicas_for(step_in)
        copies = [(wp, sp, A)] + [(wp.clone(), sp.clone(), A.clone() if M > 1 else A)
                                  for _ in range(R - 1)]
        C = torch.empty((M, N), dtype=torch.int16, device="cuda")
        wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, M)
        ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")

        def fn(i, copies=copies, d=d, C=C, M=M, ws=ws, wsn=wsn):
            w, s_, a = copies[i % len(copies)]
            Q.qgemm_dense(d, w, s_, Q.QW_A_BF16, a, None, None, C, M, ws, wsn)
        if M == 1:
            ms, n, graph = time_region([fn], max(steps, R), warmup, world, graph_steps=R)
            wbytes = N * K + N * (K // 128) * 2
            gbs = wbytes / (ms * 1e-3) / 1e9
            out[name] = {"us": round(ms * 1e3, 2), "weight_GBps": round(gbs, 1),
                         "hbm_frac": round(gbs / peaks["hbm_gbs"], 3), "launches": n,
                         "weight_copies": R, "graph": graph}
        else:
            ms, n, _ = time_region([fn], max(5, min(steps, 50)), warmup, world)
            tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
            out[name] = {"us": round(ms * 1e3, 1), "tflops": round(tf, 1),
                         "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 3),
                         "input_copies": R, "steps": n}
        del copies
        torch.cuda.empty_cache()
    return out


def extra_w4a8_decode(steps, warmup, world):
    """W4A8 (MXFP4 weights x MXFP8 activations) decode on the M=1 decode shapes, and an
    8-row batch on the first: device time per GEMM (CUDA graph of back-to-back launches over
    weight copies that do not fit L2), weight GB/s (E2M1 codes + E8M0 scales)."""
    import moe_qw_repack_gb300.qw as Q
    out = {}
    peaks, _ = measured_peaks()
    for (M, N, K) in [(1, 14336, 4096), (1, 4096, 14336), (1, 4096, 4096), (8, 14336, 4096)]:
        p = synth.w4a8_problem(M, N, K, cfg_id=260)
        d = Q.qw_repack_query(Q.QW_W_MXFP4_G32, 1, N, K)
        wp, sp = Q.empty_packed(d)
        Q.qw_repack(d, torch.from_numpy(p["w_canon"]).cuda(), torch.from_numpy(p["s_canon"]).cuda(),
                    wp, sp)
        wbytes = N * K // 2 + N * K // 32
        R = replicas_for(wp.numel() + sp.numel())
        copies = [(wp, sp)] + [(wp.clone(), sp.clone()) for _ in range(R - 1)]
        A, Asf = torch.from_numpy(p["A"]).cuda(), torch.from_numpy(p["A_sf"]).cuda()
        C = torch.empty((M, N), dtype=torch.int16, device="cuda")

        def fn(i, copies=copies, d=d, A=A, Asf=Asf, C=C, M=M):
            w, s = copies[i % len(copies)]
            Q.qgemm_dense(d, w, s, Q.QW_A_MXFP8_G32, A, Asf, None, C, M, None, 0)
        ms, n, graph = time_region([fn], max(steps, R), warmup, world, graph_steps=R)
        gbs = wbytes / (ms * 1e-3) / 1e9
        name = f"w4a8_m{M}_{N}x{K}"
        out[name] = {"us": round(ms * 1e3, 2), "weight_GBps": round(gbs, 1),
                     "hbm_frac": round(gbs / peaks["hbm_gbs"], 3),
                     "launches": n, "weight_copies": R, "graph": graph}
        out[name].update(stream_read_reference(copies, steps, warmup, world, wbytes, peaks))
        del copies
        torch.cuda.empty_cache()
    return out


def extra_w4a4(steps, warmup, world):
    """W4A4 (NVFP4 x NVFP4, tcgen05 kind::mxf4nvf4) on the headline's larger shape.  The
    FP4 dense denominator is 6 x the measured BF16 burst (nominal 13.5 / 2.25 PF/s)."""
    import moe_qw_repack_gb300.qw as Q
    peaks, _ = measured_peaks()
    M, N, K = 4096, 14336, 4096
    p = synth.w4a4_problem(M, N, K, cfg_id=760)
    d = Q.qw_repack_query(Q.QW_W_NVFP4_G16, 1, N, K)
    wp, sp = Q.empty_packed(d)
    Q.qw_repack(d, torch.from_numpy(p["w_canon"]).cuda(), torch.from_numpy(p["s_canon"]).cuda(),
                wp, sp)
    A, Asf = torch.from_numpy(p["A"]).cuda(), torch.from_numpy(p["A_sf"]).cuda()
    step_in = d.w_bytes + d.s_bytes + A.numel() + Asf.numel()
    R = replicas_for(step_in)
    copies = [(wp, sp, A, Asf)] + [(wp.clone(), sp.clone(), A.clone(), Asf.clone())
                                   for _ in range(R - 1)]
    C = torch.empty((M, N), dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_NVFP4_G16, M)
    ws = torch.empty(max(wsn, 16), dtype=torch.uint8, device="cuda")

    def fn(i):
        w, s, a, asf = copies[i % R]
        Q.qgemm_dense(d, w, s, Q.QW_A_NVFP4_G16, a, asf, None, C, M, ws, wsn)
    ms, n, _ = time_region([fn], steps, warmup, world)
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    return {"w4a4_nvfp4_4096x14336x4096": {"us": round(ms * 1e3, 1), "tflops": round(tf, 1),
                                           "frac_fp4_peak": round(tf / (6 * peaks["bf16_tflops"]), 3),
                                           "input_copies": R, "steps": n}}


def extra_w8a8(steps, warmup, world):
    """W8A8 MX kind (MXFP8 weights x MXFP8 activations) on the headline's larger shape."""
    import moe_qw_repack_gb300.qw as Q
    peaks, _ = measured_peaks()
    M, N, K = 4096, 14336, 4096
    p = synth.w8a8_problem(M, N, K, cfg_id=7)
    d = Q.qw_repack_query(Q.QW_W_MXFP8_G32, 1, N, K)
    wp, sp = Q.empty_packed(d)
    Q.qw_repack(d, torch.from_numpy(p["w_canon"]).cuda(), torch.from_numpy(p["s_canon"]).cuda(),
                wp, sp)
    A, Asf = torch.from_numpy(p["A"]).cuda(), torch.from_numpy(p["A_sf"]).cuda()
    step_in = d.w_bytes + d.s_bytes + A.numel() + Asf.numel()
    R = replicas_for(step_in)
    copies = [(wp, sp, A, Asf)] + [(wp.clone(), sp.clone(), A.clone(), Asf.clone())
                                   for _ in range(R - 1)]
    C = torch.empty((M, N), dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_MXFP8_G32, M)
    ws = torch.empty(max(wsn, 16), dtype=torch.uint8, device="cuda")

    def fn(i):
        w, s, a, asf = copies[i % R]
        Q.qgemm_dense(d, w, s, Q.QW_A_MXFP8_G32, a, asf, None, C, M, ws, wsn)
    ms, n, _ = time_region([fn], steps, warmup, world)
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    return {"w8a8_mxfp8_4096x14336x4096": {"us": round(ms * 1e3, 1), "tflops": round(tf, 1),
                                           "frac_fp8_peak": round(tf / (2 * peaks["bf16_tflops"]), 3),
                                           "input_copies": R, "steps": n}}


MMA_PROBES = (  # (name, mode, N, FLOP per MMA): the instruction forms the GEMMs issue
    ("f16_tmem_a_n128", 0, 128, 2 * 128 * 128 * 16),   # W4A16 tcgen05 GEMM
    ("f16_smem_n256", 1, 256, 2 * 128 * 256 * 16),
    ("mxf8f6f4_n256", 2, 256, 2 * 128 * 256 * 32),     # W4A8 GEMM, MMAs only
    ("mxf8f6f4_cp_n256", 3, 256, 2 * 128 * 256 * 32),  # ... with its scale copies
    ("mxf8f6f4_cp_ahead_n256", 4, 256, 2 * 128 * 256 * 32),  # copies a stage ahead
    ("mxf8f6f4_cp_wide_n256", 5, 256, 2 * 128 * 256 * 32),   # two 128-lane copies a stage
    ("mxf4nvf4_n256", 6, 256, 2 * 128 * 256 * 64),           # W4A4 GEMM, MMAs only
    ("mxf4nvf4_cp_n256", 7, 256, 2 * 128 * 256 * 64),        # ... with its scale copies
)


def extra_mma_rate(iters=4096):
    """The tcgen05 MMA issue rate (qw_mma_rate_probe): per instruction form, the median over
    SMs of cycles and ns per MMA, and the TF/s ceiling that rate gives on all SMs."""
    import moe_qw_repack_gb300.qw as Q
    out = {}
    for name, mode, n, flop in MMA_PROBES:
        cyc, ns = Q.mma_rate(mode, n, iters)
        c, t = float(np.median(cyc)), float(np.median(ns))
        out[name] = {"cycles_per_mma": round(c, 1), "ns_per_mma": round(t, 2),
                     "sm_ghz": round(c / t, 3), "sms": int(cyc.size),
                     "ceiling_tflops": round(flop * cyc.size / t / 1e3, 1)}
    return {"mma_rate": out}


def extra_moe(steps, warmup, world, only=None, scale=1):
    """Grouped MoE workloads: W4A8 (E=256, top-8, T=4096, 7168 -> 4096) and the W4A16
    intermediate-640 token sweep (E=128, top-8, up 4096 -> 1280 plus down 640 -> 4096).
    One step = route + permute + grouped GEMM(s) (+ for W4A16 the SiLU*mul between the
    projections and the top-k combine after them); inputs drawn on the device.  Steps are
    replayed from a CUDA graph; each part is also timed alone the same way."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import moe_qw_repack_gb300.qw as Q
    import synth.device as sd
    from qwtest import moe_pipeline
    peaks, _ = measured_peaks()
    out = {}

    def parts(fns, n_steps, graph_steps):
        tot, n, graph = time_region(fns, n_steps, warmup, world, graph_steps=graph_steps)
        each = [time_region([f], n_steps, 1, world, graph_steps=graph_steps)[0] for f in fns]
        return tot, each, n, graph
    # -- W4A8, E=256 (the active experts' weights alone are ~2.4 GB per step); `scale`
    # divides E and T (a smaller case of the same kernels for profiler captures)
    E, T, K, N, k = 256 // scale, 4096 // scale, 7168, 4096, 8
    name4 = f"cfg4_moe_w4a8_E{E}_T{T}"
    if only and only not in name4:
        return _extra_moe_w4a16(steps, warmup, world, only, parts, out, peaks)
    r = moe_pipeline(Q.QW_A_MXFP8_G32, Q.QW_W_MXFP4_G32, E, T, K, N, k, cfg_id=3)
    tot, each, n, graph = parts([r["route"], r["permute"], r["gemm"]], steps, 4)
    assert Q.qw_read_error(r["err"]) == 0
    # the Indexed path: route + one GEMM that gathers the rows by pair id (no permute)
    tot_ix, _, _ = time_region([r["route"], r["gemm_indexed"]], steps, warmup, world,
                               graph_steps=4)
    gemm_ix = time_region([r["gemm_indexed"]], steps, 1, world, graph_steps=4)[0]
    assert Q.qw_read_error(r["err"]) == 0
    cnt = np.diff(r["offsets"].cpu().numpy())
    active = int((cnt > 0).sum())
    P = T * k
    flop = 2.0 * P * N * K
    gemm_ms = each[2]
    wbytes = active * (N * K // 2 + N * K // 32)
    out[name4] = {
        "us_total": round(tot * 1e3, 1), "us_route": round(each[0] * 1e3, 1),
        "us_permute": round(each[1] * 1e3, 1), "us_gemm": round(gemm_ms * 1e3, 1),
        "gemm_tflops": round(flop / (gemm_ms * 1e-3) / 1e12, 1),
        "gemm_frac_fp8_peak": round(flop / (gemm_ms * 1e-3) / 1e12 / (2 * peaks["bf16_tflops"]), 3),
        "us_total_indexed": round(tot_ix * 1e3, 1), "us_gemm_indexed": round(gemm_ix * 1e3, 1),
        "active_experts": active, "active_weight_GB": round(wbytes / 1e9, 3),
        "weight_stream_frac_hbm": round(wbytes / (gemm_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
        "steps": n, "graph": graph}
    # BF16 -> MXFP8 activation quantizer for the same tokens (T x hidden 7168)
    xa = sd.bf16_activations(T, K, cfg_id=3)
    qa = torch.empty((T, K), dtype=torch.uint8, device="cuda")
    qsf = torch.empty((T, K // 32), dtype=torch.uint8, device="cuda")
    qerr = Q.new_error_flag()
    q_ms = time_region([lambda i: Q.qw_quantize_mxfp8(xa, T, K, qa, qsf, qerr)], steps, warmup,
                       world, graph_steps=4)[0]
    assert Q.qw_read_error(qerr) == 0
    qbytes = T * K * 2 + T * K + T * K // 32
    out[name4].update({
        "us_quantize_bf16_to_mxfp8": round(q_ms * 1e3, 1),
        "quantize_frac_hbm": round(qbytes / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)})
    del r, xa, qa, qsf
    torch.cuda.empty_cache()
    return _extra_moe_w4a16(steps, warmup, world, only, parts, out, peaks)


def _extra_moe_w4a16(steps, warmup, world, only, parts, out, peaks):
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import moe_qw_repack_gb300.qw as Q
    import synth.device as sd
    from qwtest import moe_pipeline
    # -- W4A16, E=128, intermediate 640
    E, k = 128, 8
    names = {T: f"cfg5_moe_w4a16_E128_T{T}" for T in (1, 16, 256, 2048, 8192)}
    if only and not any(only in n for n in names.values()):
        return out
    up_w = sd.int_weights(E, 1280, 4096, bits=4, cfg_id=4)
    dn_w = sd.int_weights(E, 4096, 640, bits=4, cfg_id=4)
    for T in (1, 16, 256, 2048, 8192):
        if only and only not in names[T]:
            continue
        P = T * k
        up = moe_pipeline(Q.QW_A_BF16, Q.QW_W_INT4_G128_BF16, E, T, 4096, 1280, k, cfg_id=4,
                          weights=up_w)
        x = sd.bf16_activations(P, 640, cfg_id=40 + T)
        dn = moe_pipeline(Q.QW_A_BF16, Q.QW_W_INT4_G128_BF16, E, T, 640, 4096, k, cfg_id=4,
                          weights=dn_w, x_sorted=x, route_from=up)
        up["route"]()  # the routing is the same every step: size the weight copies for it
        n_active = int((np.diff(up["offsets"].cpu().numpy()) > 0).sum())
        R = min(32, replicas_for(n_active * (1280 * 4096 // 2 + 4096 * 640 // 2)))
        up["set_replicas"](R)
        dn["set_replicas"](R)
        # the layer's remaining steps: silu(gate) * up -> the down projection's input x, and
        # the top-k weighted combine of the down projection's rows back to the T tokens
        lg = up["logits_dev"]
        y = torch.empty((T, 4096), dtype=torch.int16, device="cuda")
        cws_n = Q.qgemm_moe_combine_workspace_size(T, k)
        cws = torch.empty(cws_n, dtype=torch.uint8, device="cuda")
        cerr = Q.new_error_flag()

        def silu(i, up=up, x=x, P=P):
            Q.qw_silu_mul(up["C"], P, 640, x)

        def combine(i, dn=dn, up=up, lg=lg, y=y, T=T, cws=cws, cws_n=cws_n, cerr=cerr):
            Q.qgemm_moe_combine(dn["C"], up["sorted_pairs"], up["topk_ids"], lg, T, E, k, 4096,
                                y, cws, cws_n, cerr)
        n_steps = max(steps, R) if T <= 256 else max(5, steps // 4)
        tot, each, n, graph = parts([up["route"], up["permute"], up["gemm"], silu, dn["gemm"],
                                     combine], n_steps, max(R, 4))
        assert Q.qw_read_error(cerr) == 0
        assert Q.qw_read_error(up["err"]) == 0 and Q.qw_read_error(dn["err"]) == 0
        cnt = np.diff(up["offsets"].cpu().numpy())
        active = int((cnt > 0).sum())
        up_ms, dn_ms = each[2], each[4]
        wbytes_up = active * (1280 * 4096 // 2 + 1280 * 32 * 2)
        wbytes_dn = active * (4096 * 640 // 2 + 4096 * 5 * 2)
        flop = 2.0 * P * (1280 * 4096 + 4096 * 640)
        out[names[T]] = {
            "us_total": round(tot * 1e3, 1), "us_route": round(each[0] * 1e3, 1),
            "us_permute": round(each[1] * 1e3, 1),
            "us_up": round(up_ms * 1e3, 1), "us_silu_mul": round(each[3] * 1e3, 1),
            "us_down": round(dn_ms * 1e3, 1), "us_combine": round(each[5] * 1e3, 1),
            "gemm_tflops": round(flop / ((up_ms + dn_ms) * 1e-3) / 1e12, 2),
            "active_experts": active,
            "weight_GBps": round((wbytes_up + wbytes_dn) / ((up_ms + dn_ms) * 1e-3) / 1e9, 1),
            "weight_frac_hbm": round((wbytes_up + wbytes_dn) / ((up_ms + dn_ms) * 1e-3) / 1e9
                                     / peaks["hbm_gbs"], 3),
            "steps": n, "weight_copies": R, "graph": graph}
        del up, dn, x
        torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank):
    import moe_qw_repack_gb300.qw as Q
    peaks, peak_src = measured_peaks()
    step_in = 0
    for m, n, k in SHAPES:
        d = Q.qw_repack_query(Q.QW_W_MXFP4_G32, 1, n, k)
        step_in += d.w_bytes + d.s_bytes + m * k + m * k // 32
    R = replicas_for(step_in)
    probs = [W4A8Problem(m, n, k, replicas=R) for m, n, k in SHAPES]
    fns = [pr.run for pr in probs]
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        t0 = time.perf_counter()
        ms, n, _ = time_region(fns, args.steps, args.warmup, world)
        wall = time.perf_counter() - t0
    for pr in probs:
        code = Q.qw_read_error(pr.err)
        if code != 0:
            raise RuntimeError(f"device error flag {code}")
    per_gemm = [time_region([f], args.steps, args.warmup, world)[0] for f in fns]
    F = flops_of(SHAPES)
    value = whole_job_tflops(F, world, ms)
    # roofline of the dominant kernel: every launch in the timed region is the W4A8 GEMM,
    # so its average launch time is the region time over the launches
    achieved = F / (ms * 1e-3) / 1e12
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # FP8 dense = 2 x BF16 dense (nominal ratio 4.5 / 2.25)
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "gemm_w4a8_traffic.json")
    if os.path.exists(tpath):
        try:
            tj = json.load(open(tpath))
            src = open(os.path.join(ROOT, "moe_qw_repack_gb300", "csrc", "gemm_w4a8_tc.cu"), "rb").read()
            import hashlib
            if tj.get("source_sha256") == hashlib.sha256(src).hexdigest():
                traffic = tj.get("dram_bytes_per_step")
        except (OSError, ValueError):
            traffic = None

    # end to end: pinned host activations -> device, both GEMMs, results -> pinned host
    e_ms, e_n = time_e2e_pipelined(probs, max(3, args.steps), 2, world)
    h2d = sum(pr.A_host.numel() + pr.Asf_host.numel() for pr in probs)
    d2h = sum(pr.C.numel() * 2 for pr in probs)
    link_ms = time_copies_only(probs, max(3, min(args.steps, 100)), world)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3xe2m1",
        "data": "synthetic (splitmix64 seed 20261202; E2M1 uniform over 16 codes, E4M3 of N(0,1), "
                "E8M0 uniform 118..126)",
        "config": {"workload": WORKLOAD,
                   "l2": f"inputs larger than L2: steps rotate over {R} copies of the inputs "
                         f"({step_in / 2**20:.0f} MiB per copy, {R * step_in / 2**20:.0f} MiB in "
                         f"rotation; each step also writes {d2h / 2**20:.0f} MiB); no flush",
                   "timing": "K steps back to back between one CUDA event pair",
                   "per_gemm_ms": [round(t, 4) for t in per_gemm],
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(whole_job_tflops(F, world, e_ms), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "how": "qgemm_dense per step with its activations copied in from pinned host "
                       "memory and its BF16 results copied out to pinned host memory; copies in, "
                       "GEMMs and copies out on three streams over two device slots",
                "steps": e_n,
                # the same copies with no GEMM: what the host link alone allows
                "copies_only_ms_per_step": round(link_ms, 4),
                "host_link_GBps": round((h2d + d2h) / (link_ms * 1e-3) / 1e9, 1),
                "frac_of_copies_only": round(link_ms / e_ms, 3)},
        "gpu_launches": len(fns) * n,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp8_peak, 4), "traffic": traffic,
                     "traffic_note": "DRAM read + write bytes per step from one ncu capture; "
                                     "writes of C still dirty in L2 when a launch ends are not "
                                     "in it, so it reads below the algorithmic bytes",
                     "peak_source": f"{peak_src} bf16 burst x 2 (FP8 / BF16 nominal)"},
        "clocks": clk.summary(),
        "wall_s_timed_loop": round(wall, 3),
    }
    del probs
    torch.cuda.empty_cache()
    if not args.no_extra:
        line["extra"] = extra_w4a16(max(5, min(args.steps, 200)), 3, world)
        line["extra"].update(extra_w8a8(max(5, min(args.steps, 100)), 3, world))
        line["extra"].update(extra_w4a4(max(5, min(args.steps, 100)), 3, world))
        line["extra"].update(extra_w4a8_decode(max(5, min(args.steps, 200)), 3, world))
        line["extra"].update(extra_fp8w(max(5, min(args.steps, 200)), 3, world))
        line["extra"].update(extra_moe(max(5, min(args.steps, 40)), 3, world))
        line["extra"].update(extra_mma_rate())
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    line["summary"] = summarize(line)  # last key: every configured workload's fraction
    return line


def summarize(line):
    """One compact entry per configured workload (fraction of its roofline), in the order
    of the workload list, so that the end of the printed line carries all of them."""
    ex = line.get("extra", {})
    sm = {"cfg2_w4a8_frac_fp8": line["roofline"]["frac"],
          "e2e_over_device": round(line["e2e"]["value"] / line["value"], 3),
          "e2e_frac_of_host_link": line["e2e"].get("frac_of_copies_only")}

    def get(name, key):
        v = ex.get(name, {}).get(key)
        return v if v is not None else None
    sm["cfg1_m8_frac_hbm"] = get("cfg1_w4a16_m8_2048x2048_int4", "hbm_frac")
    sm["cfg1_stream_read_frac"] = [get("cfg1_w4a16_m8_2048x2048_int4", "stream_read_frac"),
                                   get("cfg1_w4a16_m8_2048x2048_int4", "stream_read_chained_frac")]
    sm["w4a8_m1_frac_hbm"] = [get(f"w4a8_m1_{n}x{k}", "hbm_frac")
                              for n, k in ((14336, 4096), (4096, 14336), (4096, 4096))]
    for bits in (4, 3):
        sm[f"cfg3_int{bits}_frac_hbm"] = [get(f"cfg3_m1_{n}x{k}_int{bits}", "hbm_frac")
                                          for n, k in ((14336, 4096), (4096, 14336), (4096, 4096))]
    sm["cfg3_stream_read_frac"] = [get(f"cfg3_m1_{n}x{k}_int4", "stream_read_frac")
                                   for n, k in ((14336, 4096), (4096, 14336), (4096, 4096))]
    sm["cfg3_stream_read_chained_frac"] = [get(f"cfg3_m1_{n}x{k}_int4", "stream_read_chained_frac")
                                           for n, k in ((14336, 4096), (4096, 14336), (4096, 4096))]
    sm["m1_splitk_frac_hbm"] = [get("m1_1024x32768_int4_splitk", "hbm_frac"),
                                get("m1_512x16384_int4_splitk", "hbm_frac")]
    sm["cfg4_gemm_frac_fp8"] = get("cfg4_moe_w4a8_E256_T4096", "gemm_frac_fp8_peak")
    sm["cfg5_weight_frac_hbm"] = {t: get(f"cfg5_moe_w4a16_E128_T{t}", "weight_frac_hbm")
                                  for t in (1, 16, 256)}
    sm["cfg5_tflops"] = {t: get(f"cfg5_moe_w4a16_E128_T{t}", "gemm_tflops") for t in (2048, 8192)}
    sm["cfg5_us_step"] = {t: get(f"cfg5_moe_w4a16_E128_T{t}", "us_total")
                          for t in (1, 16, 256, 2048, 8192)}
    # the tensor-core GEMMs against the issue rate of the MMA form they use (measured above,
    # scaled from the probe's SM clock to the one sampled during the timed region)
    mr = ex.get("mma_rate", {})

    def ceiling(name):
        r = mr.get(name, {})
        c, ghz = r.get("ceiling_tflops"), r.get("sm_ghz")
        mhz = line.get("clocks", {}).get("sm_mhz")
        return c * (mhz / 1e3) / ghz if (c and ghz and mhz) else c
    ceil_mx = ceiling("mxf8f6f4_cp_n256")
    ceil_f16 = ceiling("f16_tmem_a_n128")
    t8192 = sm["cfg5_tflops"].get(8192)
    sm["frac_of_mma_issue_ceiling"] = {
        "cfg2_w4a8": round(line["value"] / ceil_mx, 3) if ceil_mx else None,
        "cfg5_T8192_w4a16": round(t8192 / ceil_f16, 3) if (ceil_f16 and t8192) else None}
    return sm


# ----------------------------------------------------------------------------- oracle arm
@functools.lru_cache(maxsize=2)
def _oracle_inputs(M, N, K):
    return synth.w4a8_problem(M, N, K, cfg_id=1)


CPU_SAMPLE_ROWS_B = 4096  # rows of (4096,14336,4096) in the oracle's timed sample


def cpu_baseline(rows_b=CPU_SAMPLE_ROWS_B, min_seconds=10.0, rows_a=None):
    """Time the float64 oracle on a bounded sample: the first `rows_a` rows (default all) of
    (4096,3072,4096) plus the first `rows_b` rows of (4096,14336,4096) (rows_b = 0: none),
    repeated until at least `min_seconds` of CPU work."""
    from oracle import qgemm as OQ
    sample = [(4096, 3072, 4096, None if rows_a is None else np.arange(rows_a))]
    if rows_b:
        sample.append((4096, 14336, 4096, np.arange(rows_b)))
    probs = [_oracle_inputs(M, N, K) for M, N, K, _ in sample]  # drawn once, not timed
    flops = 0.0
    t = 0.0
    reps = 0
    while reps == 0 or (t < min_seconds and reps < 8):  # at least one repetition
        for (M, N, K, rows), p in zip(sample, probs):
            t0 = time.perf_counter()
            OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K,
                                   rows=rows)
            t += time.perf_counter() - t0
            flops += 2.0 * (M if rows is None else len(rows)) * N * K
        reps += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    what = "all rows" if rows_a is None else f"first {rows_a} rows"
    what += f" + (4096,14336,4096) first {rows_b} rows" if rows_b else ""
    return {"value": round(flops / t / 1e12, 5), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"(4096,3072,4096) {what}, x{reps}: {flops / 1e9:.1f} GFLOP in {t:.2f} s "
                      f"(weight decode + float64 matmul per call)"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    vals = []
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state; warm-up steps are skipped deliberately
    cb = None
    # each step is a bounded sample sized so that the whole run stays within a few minutes:
    # a few steps take a large sample, many steps a row subset of the smaller shape (each
    # call decodes that shape's weights, ~0.3 s on these hosts)
    # One step is one repetition of the cpu_baseline leg's sample (the same shapes and rows,
    # so the two report the same rate), about 3 s on these hosts; past 40 steps the
    # sample keeps its shapes with proportionally fewer rows so the run stays short.
    if args.oracle_rows:  # a short sample: that many rows of the (4096, 3072, 4096) GEMM
        kw = dict(rows_b=0, min_seconds=0.0, rows_a=args.oracle_rows)
    elif args.steps <= 40:
        kw = dict(rows_b=CPU_SAMPLE_ROWS_B, min_seconds=0.0)
    else:
        f = 40.0 / args.steps
        kw = dict(rows_b=max(64, int(CPU_SAMPLE_ROWS_B * f)), min_seconds=0.0,
                  rows_a=max(64, int(4096 * f)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cb = cpu_baseline(**kw)
        vals.append(cb["value"])
    wall = time.perf_counter() - t0
    v = statistics.median(vals)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall / args.steps * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": cb["sample"]},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-w4a16", action="store_true",
                    help="time only the W4A16 GEMV workloads (a profiling aid)")
    ap.add_argument("--only-moe", action="store_true",
                    help="time only the grouped MoE workloads (a profiling aid)")
    ap.add_argument("--only-w4a8-decode", action="store_true",
                    help="only the single-token W4A8 (MXFP4 x MXFP8) decode rows")
    ap.add_argument("--only-mx-dense", action="store_true",
                    help="only the dense W8A8 and W4A4 GEMM rows (--case w8a8 / w4a4: one)")
    ap.add_argument("--only-fp8w", action="store_true",
                    help="time only the FP8-weight WnA16 workloads (a profiling aid)")
    ap.add_argument("--moe-scale", type=int, default=1,
                    help="with --only-moe: divide the E=256 W4A8 workload's experts and tokens "
                         "by this (a smaller case for profiler captures)")
    ap.add_argument("--case", default=None,
                    help="with --only-w4a16 / --only-moe / --only-fp8w: run only the cases "
                         "whose name contains this string")
    ap.add_argument("--oracle-rows", type=int, default=0,
                    help="with --impl reference: a short step sample of that many rows of the "
                         "(4096, 3072, 4096) GEMM (default: the cpu_baseline leg's sample)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup) if args.impl == "ours" else args.warmup
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        line = run_reference(args, world, rank)
    elif args.only_w4a16:
        world, rank, _ = dist_setup()
        line = {"extra": extra_w4a16(args.steps, args.warmup, world, args.case)}
    elif args.only_moe:
        world, rank, _ = dist_setup()
        line = {"extra": extra_moe(args.steps, args.warmup, world, args.case, args.moe_scale)}
    elif args.only_mx_dense:
        world, rank, _ = dist_setup()
        line = {"extra": {}}
        if not args.case or args.case in "w8a8_mxfp8":
            line["extra"].update(extra_w8a8(args.steps, args.warmup, world))
        if not args.case or args.case in "w4a4_nvfp4":
            line["extra"].update(extra_w4a4(args.steps, args.warmup, world))
    elif args.only_w4a8_decode:
        world, rank, _ = dist_setup()
        line = {"extra": extra_w4a8_decode(args.steps, args.warmup, world)}
    elif args.only_fp8w:
        world, rank, _ = dist_setup()
        line = {"extra": extra_fp8w(args.steps, args.warmup, world, args.case)}
    else:
        world, rank, _ = dist_setup()
        line = run_ours(args, world, rank)
    if line is not None and int(os.environ.get("RANK", "0")) == 0:
        print(json.dumps(line), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
