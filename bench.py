#!/usr/bin/env python3
"""Benchmark: OUT_PROD / MUL_MAT_ID_BACK on one GB300 (or N replicas).

One step is one pass of the hot path over one batch of synthetic input.  The
headline workload is the largest dense training OUT_PROD through a frozen
quantised weight: a = q8_0 of a N(0, 0.02) [5120, 17408] matrix, b = an f32
gradient [1024, 17408] ~ N(0,1)*1e3 with 0.2% outliers of magnitude
U(6.6e4, 1.5e5); `value` is its algorithmic TFLOP/s (2*M*N*K per call).  The
same line carries `parts`: the other rows of the path measured in the same run
(rank-r LoRA gradient GB/s, grouped-head broadcast, the other dense shapes,
MUL_MAT_ID_BACK), each with its own roofline.

Timing: W warm-up steps, then K timed steps, each bracketed by CUDA events on
the launching stream, each preceded by a ~100 us device-side wait so that the
host has enqueued the step before the GPU reaches it.  No L2 flush is written: the headline's inputs (166 MB)
are larger than L2 (129 MB), and every smaller workload rotates through
ceil(2 * L2 / bytes) + 1 copies of its inputs and outputs, so each call reads
data that the previous calls have evicted.  With torchrun each rank runs an
independent replica (no data-path collective); rank 0 prints the max over
ranks.

Roofline of the dense kernels: tensor-pipe utilisation, i.e. the TF32 tensor
work of the 3xTF32 scheme (three TF32 products per multiply-add, 3 * 2MNK
flops) per second over the dense TF32 peak measured in the same run (cuBLAS
TF32 GEMM 8192^3, best of 10); the algorithmic 2MNK/t is printed beside it.
Skinny rank-r kernels: algorithmic bytes per second over the measured HBM
copy bandwidth.  MUL_MAT_ID_BACK: the larger of its HBM and tensor-pipe times
over the measured time.

`--impl reference` times the CPU oracle on a bounded sample of the same
workload on the host's cores (there is no other implementation to run).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "OUT_PROD TFLOP/s (dense) and GB/s (rank-r) on 1 GB300, % of roofline"
DENSE_M, DENSE_K, DENSE_N = 5120, 17408, 1024
WORKLOAD = (f"dense OUT_PROD q8_0 x f32 m{DENSE_M} k{DENSE_K} n{DENSE_N} "
            "(frozen quantised weight, gradient with 0.2% outliers to 1.5e5)")
L2_BYTES = 129 << 20
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25          # nominal dense ratio (context only)
# DRAM bytes (read + write) of one launch of the tensor-core tile kernel on the
# headline workload, from the ncu capture summarised in
# profiles/tc_out_prod_q8_m5120_k17408_n1024.md, and the digest of the kernel
# sources it was taken on: the figure is reported only while the sources in
# this tree still hash to that digest (null once the kernel has changed).
TC_TRAFFIC = {"bytes": 419260160, "sources_sha256": "220a162cface34a3fa6e6ba2b30504ca352dae2b034e929c8e7726ddedd56c44"}
TC_SOURCES = ("ggml_out_prod_gb300/csrc/dense_tc.cu", "ggml_out_prod_gb300/csrc/tc_ptx.cuh")


def _sources_digest():
    h = hashlib.sha256()
    for rel in TC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic():
    if TC_TRAFFIC["bytes"] is None or TC_TRAFFIC["sources_sha256"] != _sources_digest():
        return None
    return TC_TRAFFIC["bytes"]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def rotation_sets(bytes_per_set):
    """Copies of a workload's inputs and outputs to cycle through so that
    every call reads HBM, not L2: ceil(2 * L2 / bytes) + 1 (1 once one set is
    larger than twice L2)."""
    if bytes_per_set >= 2 * L2_BYTES:
        return 1
    return int(math.ceil(2 * L2_BYTES / bytes_per_set)) + 1


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
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
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

# A device-side wait of ~100 us enqueued before each timed call: while the
# GPU runs it the host enqueues the call and its closing event, so the events
# bracket device time only, not the host's launch overhead (a 10 us kernel
# costs more than that to launch from Python).  It touches no memory.
HOST_LEAD_CYCLES = 200_000


def host_lead(torch):
    torch.cuda._sleep(HOST_LEAD_CYCLES)


def time_rotating(torch, calls, steps, warmup):
    """Per-call CUDA-event times (ms) on the current stream, cycling through
    `calls` (one per rotation set), after `warmup` untimed calls."""
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        calls[i % len(calls)]()
    torch.cuda.synchronize()
    evs = []
    for i in range(steps):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        host_lead(torch)
        s.record(stream)
        calls[(warmup + i) % len(calls)]()
        e.record(stream)
        evs.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier_max(torch, value, ws):
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(ws, flops_per_rank, ms_step_max):
    """TFLOP/s of the whole job: every rank's work over the slowest rank's
    step time (replicas: each rank runs the full workload)."""
    return ws * flops_per_rank / (ms_step_max * 1e-3) / 1e12


def _cublas_tf32(torch, device):
    """Dense TF32 peak: cuBLAS TF32 GEMM 8192^3, best of 10 (TFLOP/s)."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        n = 8192
        x = torch.randn(n, n, device=device)
        y = torch.randn(n, n, device=device)
        for _ in range(3):
            x @ y
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record()
            x @ y
            e.record()
            torch.cuda.synchronize()
            best = min(best, s.elapsed_time(e))
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def dense_roofline(flops, us, tf32_peak, products=3):
    """Tensor-pipe utilisation of a 3xTF32 (or 2xTF32) product."""
    pipe = products * flops / (us * 1e-6) / 1e12
    return {"bound": "tensor", "achieved": round(pipe, 2), "peak": round(tf32_peak, 1),
            "unit": "TFLOP/s", "frac": round(pipe / tf32_peak, 4),
            "algorithmic_TFLOP/s": round(flops / (us * 1e-6) / 1e12, 2)}


def hbm_roofline(byts, us, hbm):
    gbs = byts / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(gbs / hbm, 4)}


def bench_config(ws):
    """The `config` of both arms' lines (the same workload and layout)."""
    return {"workload": WORKLOAD, "parallelism": f"replicas x{ws}",
            "l2": "inputs larger than L2 (166 MB), no flush; smaller parts rotate "
                  "ceil(2*L2/bytes)+1 input sets"}


def gpu_arm(args):
    import torch

    import ggml_out_prod_gb300 as op

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    op.build()
    op.lib()
    peaks, peak_kind = _peaks()
    hbm = peaks["hbm_gbs"]
    tf32_peak = _cublas_tf32(torch, device)
    clocks = ClockSampler(device.index if device.index is not None else 0)

    # ---- headline: dense q8_0 OUT_PROD, the largest shape ----------------
    a_np, b_np = synth.dense_quant(synth.TYPE_Q8_0, DENSE_M, DENSE_K, DENSE_N)
    a = torch.from_numpy(a_np).to(device)
    b = torch.from_numpy(b_np).to(device)
    ne_a, ne_b = (DENSE_M, DENSE_K, 1, 1), (DENSE_N, DENSE_K, 1, 1)
    out = torch.empty((1, 1, DENSE_N, DENSE_M), dtype=torch.float32, device=device)
    nws = op.oop_out_prod_workspace_size(op.TYPE_Q8_0, ne_a, ne_b)
    ws_buf = torch.empty(max(nws, 1), dtype=torch.uint8, device=device)
    flops = 2.0 * DENSE_M * DENSE_N * DENSE_K
    in_bytes = a_np.nbytes + b_np.nbytes
    assert in_bytes > L2_BYTES, "the headline's inputs must be larger than L2"

    def dense_call():
        op.out_prod(a, b, a_type=op.TYPE_Q8_0, ne_a=ne_a, out=out, workspace=ws_buf,
                    path=op.PATH_TCGEN05)

    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for _ in range(args.warmup):
        dense_call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = []
    launches = 0
    t_region0 = time.perf_counter()
    for _ in range(args.steps):
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        k0 = torch.cuda.Event(enable_timing=True)
        k1 = torch.cuda.Event(enable_timing=True)
        for e in (k0, k1):          # create the events before handing them over
            e.record(stream)
        op.profile_main_kernel(k0, k1)
        host_lead(torch)
        s0.record(stream)
        dense_call()
        launches += op.last_launch_count()
        s1.record(stream)
        evs.append((s0, s1, k0, k1))
    torch.cuda.synchronize()
    region_s = time.perf_counter() - t_region0
    step_ms = [s0.elapsed_time(s1) for s0, s1, _, _ in evs]
    main_ms = [k0.elapsed_time(k1) for _, _, k0, k1 in evs]
    ms_step = statistics.mean(step_ms)
    ms_main = statistics.mean(main_ms)
    ms_step_max = _barrier_max(torch, ms_step, ws)
    value = whole_job_value(ws, flops, ms_step_max)

    # ---- e2e: host buffers through the C ABI's host entry ------------------
    # (oop_out_prod_host: copies in, product, copy of dst out, one call; the
    # timed region ends when dst is back in host memory)
    a_host = torch.from_numpy(a_np).pin_memory()
    b_host = torch.from_numpy(b_np).pin_memory()
    dst_host = torch.empty((1, 1, DENSE_N, DENSE_M), dtype=torch.float32, pin_memory=True)
    nbuf = op.oop_out_prod_host_buffer_size(op.TYPE_Q8_0, ne_a, ne_b)
    dev_buf = torch.empty(nbuf, dtype=torch.uint8, device=device)

    def e2e_call():
        op.out_prod_host(a_host, b_host, a_type=op.TYPE_Q8_0, ne_a=ne_a, out=dst_host,
                         device_buffer=dev_buf)

    for _ in range(max(1, args.warmup)):
        e2e_call()
    torch.cuda.synchronize()
    e2e_t = []
    for _ in range(args.steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_call()
        e2e_t.append(time.perf_counter() - t0)
    e2e_s = _barrier_max(torch, statistics.mean(e2e_t), ws)
    del dev_buf, a_host, b_host, dst_host

    # ---- the other rows of the path (same run) ----------------------------
    parts = {}
    psteps = max(args.steps, 20)

    def skinny_part(r):
        an, bn = synth.lora_rank(r)
        byts = 4.0 * (2560 * 512 + r * 512 + 2560 * r)
        sets = rotation_sets(byts)
        ta = [torch.from_numpy(an).to(device) for _ in range(sets)]
        tb = [torch.from_numpy(bn).to(device) for _ in range(sets)]
        o = [torch.empty((1, 1, r, 2560), dtype=torch.float32, device=device) for _ in range(sets)]
        calls = [(lambda i=i: op.out_prod(ta[i], tb[i], out=o[i], path=op.PATH_SKINNY))
                 for i in range(sets)]
        us = statistics.mean(time_rotating(torch, calls, psteps, 3)) * 1e3
        return {"workload": f"LoRA rank-{r} gradient: a [2560, 512] f32, b [{r}, 512]",
                "us": round(us, 3), "bytes": byts, "rotation_sets": sets,
                "roofline": hbm_roofline(byts, us, hbm)}

    for r in synth.LORA_RANKS:
        parts[f"lora_r{r}"] = skinny_part(r)

    # rank-r gradients for many slices in one launch (steady-state streaming;
    # src0 is 335 MB, larger than twice L2, so one set suffices)
    nsl = 64
    an = synth.make_a(synth.TYPE_F32, (2560, 512, nsl, 1), 70)
    ta = torch.from_numpy(an).to(device)
    del an
    for r in synth.LORA_RANKS:
        bn = synth.make_b((r, 512, nsl, 1), 71, std=100.0, outliers=True)
        tb = torch.from_numpy(bn).to(device)
        o = torch.empty((1, nsl, r, 2560), dtype=torch.float32, device=device)
        byts = 4.0 * nsl * (2560 * 512 + r * 512 + 2560 * r)
        call = (lambda tb=tb, o=o: op.out_prod(ta, tb, out=o, path=op.PATH_SKINNY))
        us = statistics.mean(time_rotating(torch, [call], max(args.steps, 10), 3)) * 1e3
        parts[f"lora_r{r}_x64_slices"] = {
            "workload": f"64 rank-{r} gradients in one launch: a [2560, 512, 64] f32, b [{r}, 512, 64]",
            "us": round(us, 3), "bytes": byts, "rotation_sets": rotation_sets(byts),
            "roofline": hbm_roofline(byts, us, hbm)}
        del tb, o
    del ta

    for n_seq in (1, 2):
        an, bn = synth.grouped_heads(n_seq)
        byts = an.nbytes + bn.nbytes + 4 * 128 * 128 * 16 * n_seq
        sets = rotation_sets(byts)
        ta = [torch.from_numpy(an).to(device) for _ in range(sets)]
        tb = [torch.from_numpy(bn).to(device) for _ in range(sets)]
        o = [torch.empty((n_seq, 16, 128, 128), dtype=torch.float32, device=device)
             for _ in range(sets)]
        calls = [(lambda i=i: op.out_prod(ta[i], tb[i], out=o[i])) for i in range(sets)]
        us = statistics.mean(time_rotating(torch, calls, psteps, 3)) * 1e3
        fl = 2.0 * 128 * 128 * 512 * 16 * n_seq

        # the same slices as one launch per slice (the per-slice loop)
        def per_slice(i):
            for i3 in range(n_seq):
                for i2 in range(16):
                    op.out_prod(ta[i][i3, i2 // 4], tb[i][i3, i2], out=o[i][i3, i2],
                                ne_a=(128, 512, 1, 1))

        loops = [(lambda i=i: per_slice(i)) for i in range(sets)]
        t2 = time_rotating(torch, loops, max(args.steps // 2, 5), 2)
        parts[f"grouped_heads_x{n_seq}"] = {
            "workload": f"a [128, 512, 4, {n_seq}], b [128, 512, 16, {n_seq}], dps2 = 4",
            "us_one_launch": round(us, 3), "rotation_sets": sets,
            "us_per_slice_loop": round(statistics.mean(t2) * 1e3, 3),
            "launches_per_slice_loop": 16 * n_seq,
            "roofline": dense_roofline(fl, us, tf32_peak)}
        del ta, tb, o

    # the rank-r LoRA gradients of one 4B layer in one launch: dA and dB of the
    # seven adapted projections (14 narrow OUT_PRODs over 512 tokens), against
    # one launch per gradient
    T, r = 512, 8
    lay = [(K_in, N_out) for K_in, N_out in synth.LAYER_4B_PROJ]
    ms = [k for k, _ in lay] + [n for _, n in lay]
    byts = sum(4.0 * (m * T + r * T + m * r) for m in ms)
    sets = rotation_sets(byts)
    lists = []
    for si in range(sets):
        probs = []
        for j, m in enumerate(ms):
            ta = torch.from_numpy(synth.make_a(synth.TYPE_F32, (m, T, 1, 1), 400 + j)[0, 0]).to(device)
            tb = torch.from_numpy(synth.make_b((r, T, 1, 1), 430 + j, std=100.0,
                                               outliers=True)[0, 0]).to(device)
            probs.append((ta, tb, torch.empty((r, m), device=device)))
        lists.append(probs)
    us_b = statistics.mean(time_rotating(
        torch, [(lambda pr=pr: op.out_prod_batch(pr)) for pr in lists], psteps, 3)) * 1e3
    us_l = statistics.mean(time_rotating(
        torch, [(lambda pr=pr: [op.out_prod(a_, b_, out=d_, path=op.PATH_SKINNY)
                                for a_, b_, d_ in pr]) for pr in lists], psteps, 3)) * 1e3
    parts["lora_layer_r8_batched"] = {
        "workload": "dA and dB of the 4B's 7 adapted projections at rank 8 over 512 tokens "
                    "(14 narrow OUT_PRODs, a [M, 512] f32, M from 1024 to 9728)",
        "us_one_launch": round(us_b, 3), "us_one_launch_per_gradient": round(us_l, 3),
        "bytes": byts, "rotation_sets": sets, "roofline": hbm_roofline(byts, us_b, hbm)}
    del lists

    # both adapter gradients of one projection (the 4B's q: 2560 -> 4096) in one launch
    K_in, N_out = 2560, 4096
    byts = 4.0 * ((K_in + N_out) * T + 2 * r * T + (K_in + N_out) * r)
    sets = rotation_sets(byts)
    ins = []
    for si in range(sets):
        ins.append(tuple(torch.from_numpy(v).to(device) for v in (
            synth.make_a(synth.TYPE_F32, (K_in, T, 1, 1), 460)[0, 0],
            synth.make_b((r, T, 1, 1), 461)[0, 0],
            synth.make_b((N_out, T, 1, 1), 462, std=100.0, outliers=True)[0, 0],
            synth.make_b((r, T, 1, 1), 463, std=100.0, outliers=True)[0, 0])))
    us = statistics.mean(time_rotating(
        torch, [(lambda v=v: op.lora_backward(*v)) for v in ins], psteps, 3)) * 1e3
    parts["lora_backward_q_proj_r8"] = {
        "workload": "dA {2560, 8} and dB {8, 4096} of one projection over 512 tokens, one launch",
        "us": round(us, 3), "bytes": byts, "rotation_sets": sets,
        "roofline": hbm_roofline(byts, us, hbm)}
    del ins

    # dx of a MUL_MAT backward through the transposed gradient view (no copy
    # of dy^T): W q8_0 [5120, 5120], dy [5120, 1024]
    Kw, R, T2 = 5120, 5120, 1024
    Wq = torch.from_numpy(synth.make_a(synth.TYPE_Q8_0, (Kw, R, 1, 1), 470, std=0.02)).to(device)
    dyv = torch.from_numpy(synth.make_b((R, T2, 1, 1), 471, std=1e3, outliers=True)).to(device)
    dyT = dyv.transpose(2, 3)
    o = torch.empty((1, 1, T2, Kw), dtype=torch.float32, device=device)
    wsz = op.oop_out_prod_strided_workspace_size(op.TYPE_Q8_0, (Kw, R, 1, 1), (T2, R, 1, 1),
                                                 op.nb_of(dyT))
    wsb = torch.empty(max(wsz, 1), dtype=torch.uint8, device=device)
    us = statistics.mean(time_rotating(torch, [lambda: op.out_prod(
        Wq, dyT, a_type=op.TYPE_Q8_0, ne_a=(Kw, R, 1, 1), out=o, workspace=wsb)],
        max(args.steps, 10), 3)) * 1e3
    fl = 2.0 * Kw * R * T2
    parts["dx_transposed_view_q8_0_m5120_k5120_n1024"] = {
        "workload": "dx = OUT_PROD(W, dy^T) with dy^T read in place: W q8_0 [5120, 5120], "
                    "dy [5120, 1024]", "us_call": round(us, 2),
        "TFLOP/s_call": round(fl / (us * 1e-6) / 1e12, 2), "rotation_sets": 1,
        "inputs": "W 27.9 MB + dy 21 MB; each call also writes and reads its 42 MB split"}
    del Wq, dyv, dyT, o, wsb

    # every dense shape, q8_0 and q4_0 (and q4_K, the pages' perf weight):
    # whole call and tile kernel alone
    for m, k in synth.DENSE_MK:
        x = synth.normal(synth.tensor_seed(30), m * k, std=0.02).reshape(1, 1, k, m)
        bn = synth.make_b((DENSE_N, k, 1, 1), 31, std=1e3, outliers=True)
        fl = 2.0 * m * DENSE_N * k
        wsz = op.oop_out_prod_workspace_size(op.TYPE_Q8_0, (m, k, 1, 1), (DENSE_N, k, 1, 1))
        wsb = torch.empty(max(wsz, 1), dtype=torch.uint8, device=device)
        for tid, tname, quant in ((synth.TYPE_Q8_0, "q8_0", synth.quantize_q8_0),
                                  (synth.TYPE_Q4_0, "q4_0", synth.quantize_q4_0),
                                  (synth.TYPE_Q4_K, "q4_K", synth.quantize_q4_k)):
            an = quant(x)
            byts = an.nbytes + bn.nbytes + 4 * m * DENSE_N
            sets = rotation_sets(byts)
            ta = [torch.from_numpy(an).to(device) for _ in range(sets)]
            tb = [torch.from_numpy(bn).to(device) for _ in range(sets)]
            o = [torch.empty((1, 1, DENSE_N, m), dtype=torch.float32, device=device)
                 for _ in range(sets)]

            def call(i):
                op.out_prod(ta[i], tb[i], a_type=tid, ne_a=(m, k, 1, 1), out=o[i], workspace=wsb,
                            path=op.PATH_TCGEN05)

            for i in range(3):
                call(i % sets)
            torch.cuda.synchronize()
            rec = []
            for i in range(max(3, args.steps // 4)):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                ev[2].record(stream)
                ev[3].record(stream)
                op.profile_main_kernel(ev[2], ev[3])
                host_lead(torch)
                ev[0].record(stream)
                call((3 + i) % sets)
                ev[1].record(stream)
                rec.append(ev)
            torch.cuda.synchronize()
            us_call = statistics.mean(e[0].elapsed_time(e[1]) for e in rec) * 1e3
            us_kern = statistics.mean(e[2].elapsed_time(e[3]) for e in rec) * 1e3
            parts[f"dense_{tname}_m{m}_k{k}_n{DENSE_N}"] = {
                "us_call": round(us_call, 2), "us_tile_kernel": round(us_kern, 2),
                "TFLOP/s_call": round(fl / (us_call * 1e-6) / 1e12, 2),
                "rotation_sets": sets,
                "roofline": dense_roofline(fl, us_kern, tf32_peak)}
            del ta, tb, o
        del wsb, x, bn

    for wt, nm in ((synth.TYPE_F32, "f32"), (synth.TYPE_BF16, "bf16")):
        W, ids, g = synth.moe_back(wt)
        Wt = W.view(np.int16) if wt == synth.TYPE_BF16 else W
        fl = 2.0 * 2048 * 768 * 8 * 512
        byts = W.nbytes + g.nbytes + 4.0 * 2048 * 8 * 512 + ids.nbytes
        sets = rotation_sets(byts)
        tW = [torch.from_numpy(Wt).to(device) for _ in range(sets)]
        tids = [torch.from_numpy(ids).to(device) for _ in range(sets)]
        tg = [torch.from_numpy(g).to(device) for _ in range(sets)]
        o = [torch.empty((512, 8, 2048), dtype=torch.float32, device=device) for _ in range(sets)]
        wsz = op.oop_mul_mat_id_back_workspace_size(wt, (2048, 768, 32), (8, 512))
        wsb = torch.empty(max(wsz, 1), dtype=torch.uint8, device=device)
        # roof: the larger of the HBM time and the tensor-pipe time (three
        # TF32 products per multiply-add for f32 W, two for bf16 W)
        products = 3 if wt == synth.TYPE_F32 else 2
        roof_us = max(byts / (hbm * 1e9), products * fl / (tf32_peak * 1e12)) * 1e6
        entry = {"workload": f"E=32 W {nm} [2048, 768], 8 of 32 experts per token, 512 tokens",
                 "bytes": byts, "rotation_sets": sets, "roof_us": round(roof_us, 2)}
        for path, pname in ((op.PATH_TCGEN05, "grouped_tcgen05"), (op.PATH_SIMT, "per_slot")):
            calls = [(lambda i=i, path=path: op.mul_mat_id_back(
                tW[i], tids[i], tg[i], w_type=wt, out=o[i], workspace=wsb, path=path))
                for i in range(sets)]
            n = psteps if path == op.PATH_TCGEN05 else max(3, args.steps // 4)
            us = statistics.mean(time_rotating(torch, calls, n, 2)) * 1e3
            entry[pname] = {"us": round(us, 3), "TFLOP/s": round(fl / (us * 1e-6) / 1e12, 3),
                            "GB/s": round(byts / (us * 1e-6) / 1e9, 1),
                            "roofline_frac": round(roof_us / us, 4)}
        parts[f"mul_mat_id_back_{nm}"] = entry
        del tW, tids, tg, o, wsb

    # MUL_MAT_ID's expert-weight gradient at the same shapes: 32 experts
    # [2048, 768], x one row per slot, 8 of 32 experts per token, 512 tokens
    W, ids, g = synth.moe_back(synth.TYPE_F32)
    x = synth.normal(synth.tensor_seed(480), 512 * 8 * 2048).reshape(512, 8, 2048)
    fl = 2.0 * 2048 * 768 * 8 * 512
    byts = x.nbytes + g.nbytes + ids.nbytes + 4.0 * 2048 * 768 * 32
    sets = rotation_sets(byts)
    tx = [torch.from_numpy(x).to(device) for _ in range(sets)]
    tids = [torch.from_numpy(ids).to(device) for _ in range(sets)]
    tg = [torch.from_numpy(g).to(device) for _ in range(sets)]
    o = [torch.empty((32, 768, 2048), dtype=torch.float32, device=device) for _ in range(sets)]
    wsz = op.oop_mul_mat_id_weight_grad_workspace_size((2048, 8, 512), (768, 8, 512), 32)
    wsb = torch.empty(max(wsz, 1), dtype=torch.uint8, device=device)
    us = statistics.mean(time_rotating(torch, [(lambda i=i: op.mul_mat_id_weight_grad(
        tx[i], tids[i], tg[i], 32, out=o[i], workspace=wsb)) for i in range(sets)],
        psteps, 2)) * 1e3
    roof_us = max(byts / (hbm * 1e9), 3 * fl / (tf32_peak * 1e12)) * 1e6
    parts["mul_mat_id_expert_weight_grad_f32"] = {
        "workload": "dW [2048, 768, 32] from x [2048, 8, 512], dy [768, 8, 512], 8 of 32 "
                    "experts per token", "us": round(us, 3),
        "TFLOP/s": round(fl / (us * 1e-6) / 1e12, 3), "bytes": byts, "rotation_sets": sets,
        "roof_us": round(roof_us, 2), "roofline_frac": round(roof_us / us, 4)}
    del tx, tids, tg, o, wsb, x, W, g

    clk = clocks.stop()
    assert op.device_status() == 0, "device status word set"

    # ---- roofline of the dominant kernel (the tensor-core tile kernel) ----
    roof = dense_roofline(flops, ms_main * 1e3, tf32_peak)
    roof.update({
        "peak_note": f"dense TF32 peak measured in this run: cuBLAS TF32 GEMM 8192^3, best of "
                     f"10 (of measured); for context, {peak_kind} bf16 burst "
                     f"{peaks['bf16_tflops']} x nominal 1.1/2.25 = "
                     f"{peaks['bf16_tflops'] * NOMINAL_TF32_OVER_BF16:.1f}",
        "kernel": "tc_out_prod_kernel (tcgen05 3xTF32): achieved = 3 * 2*M*N*K TF32 flops per "
                  "launch / its mean CUDA-event time",
        "kernel_ms": round(ms_main, 4), "split_prepass_ms": round(ms_step - ms_main, 4),
        "traffic": _traffic()})

    cpu = cpu_baseline(args.cpu_seconds) if rank == 0 and ws == 1 else None
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded splitmix64 normals, q8_0-quantised weight, 0.2% outliers)",
        "config": bench_config(ws),
        "e2e": {"value": round(ws * flops / e2e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(a_np.nbytes + b_np.nbytes),
                "d2h_bytes_per_step": int(4 * DENSE_M * DENSE_N)},
        "gpu_launches": launches,
        "clocks": clk,
        "roofline": roof,
        "cpu_baseline": cpu,
        "parts": parts,
        "region_s": round(region_s, 3),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the CPU oracle as a baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------

def _oracle_sample(seconds_target: float):
    import oracle
    oracle.build()
    a, b = synth.dense_quant(synth.TYPE_Q8_0, DENSE_M, DENSE_K, DENSE_N)
    ne_a, ne_b = (DENSE_M, DENSE_K, 1, 1), (DENSE_N, DENSE_K, 1, 1)
    rng = np.random.default_rng(0)
    cores = len(os.sched_getaffinity(0))
    # calibrate on a small sample, then size the timed one
    n = 512
    while True:
        coords = np.stack([rng.integers(0, DENSE_M, n), rng.integers(0, DENSE_N, n),
                           np.zeros(n, np.int64), np.zeros(n, np.int64)], 1)
        t0 = time.perf_counter()
        oracle.out_prod_at(a, synth.TYPE_Q8_0, b, ne_a, ne_b, coords, nthreads=cores)
        dt = time.perf_counter() - t0
        if dt > 0.5 or n >= 1 << 22:
            break
        n *= 4
    n_final = int(max(n, min(1 << 24, n * seconds_target / max(dt, 1e-3))))
    return a, b, ne_a, ne_b, n_final, cores


def cpu_baseline(seconds_target: float):
    import oracle
    a, b, ne_a, ne_b, n, cores = _oracle_sample(seconds_target)
    rng = np.random.default_rng(1)
    coords = np.stack([rng.integers(0, DENSE_M, n), rng.integers(0, DENSE_N, n),
                       np.zeros(n, np.int64), np.zeros(n, np.int64)], 1)
    t0 = time.perf_counter()
    oracle.out_prod_at(a, synth.TYPE_Q8_0, b, ne_a, ne_b, coords, nthreads=cores)
    dt = time.perf_counter() - t0
    flops = 2.0 * DENSE_K * n
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} random dst elements of the headline workload (each a {DENSE_K}-term "
                      f"fp64 sum), {dt:.1f} s"}


def reference_arm(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    a, b, ne_a, ne_b, n, cores = _oracle_sample(max(1.0, args.cpu_seconds / max(args.steps, 1)))
    rng = np.random.default_rng(2)
    for _ in range(args.warmup):
        coords = np.stack([rng.integers(0, DENSE_M, 256), rng.integers(0, DENSE_N, 256),
                           np.zeros(256, np.int64), np.zeros(256, np.int64)], 1)
        oracle.out_prod_at(a, synth.TYPE_Q8_0, b, ne_a, ne_b, coords, nthreads=cores)
    times = []
    for _ in range(args.steps):
        coords = np.stack([rng.integers(0, DENSE_M, n), rng.integers(0, DENSE_N, n),
                           np.zeros(n, np.int64), np.zeros(n, np.int64)], 1)
        t0 = time.perf_counter()
        oracle.out_prod_at(a, synth.TYPE_Q8_0, b, ne_a, ne_b, coords, nthreads=cores)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = 2.0 * DENSE_K * n / dt / 1e12
    sample = (f"{n} random dst elements of the headline workload per step "
              f"(each a {DENSE_K}-term fp64 sum)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(ws),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
