#!/usr/bin/env python3
"""Benchmark: OUT_PROD / MUL_MAT_ID_BACK on one GB300 (or N replicas).

One step is one pass of the hot path over one batch of synthetic input.  The
headline workload is the dense training OUT_PROD through a frozen quantised
weight: a = q8_0 of a N(0, 0.02) [5120, 5120] matrix, b = an f32 gradient
[1024, 5120] ~ N(0,1)*1e3 with 0.2% outliers of magnitude U(6.6e4, 1.5e5);
`value` is its algorithmic TFLOP/s (2*M*N*K per call).  The same line carries
`parts`: the other rows of the path measured in the same run (rank-r LoRA
gradient GB/s, grouped-head broadcast, MUL_MAT_ID_BACK).

Timing: W warm-up steps, then K timed steps; before every timed step a 512 MB
buffer is written to flush L2 (129 MB); each step is bracketed by CUDA events
on the launching stream.  With torchrun each rank runs an independent replica
(no data-path collective); rank 0 prints the max over ranks.

`--impl reference` times the CPU oracle on a bounded sample of the same
workload on the host's cores (there is no other implementation to run).
"""

from __future__ import annotations

import argparse
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

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "OUT_PROD TFLOP/s (dense) and GB/s (rank-r) on 1 GB300, % of roofline"
DENSE_M, DENSE_K, DENSE_N = 5120, 5120, 1024
WORKLOAD = (f"dense OUT_PROD q8_0 x f32 m{DENSE_M} k{DENSE_K} n{DENSE_N} "
            "(frozen quantised weight, gradient with 0.2% outliers to 1.5e5)")
L2_FLUSH_BYTES = 512 << 20
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25          # nominal dense ratio
# DRAM bytes (read + write) of one launch of the tensor-core tile kernel on the
# headline workload, from the ncu capture summarised in
# profiles/tc_out_prod_q8_m5120_k5120_n1024.md; None while that capture does
# not match the kernel in this tree.
TC_TRAFFIC_BYTES = 83_122_688


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


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

class Timer:
    """Per-step CUDA events on the launching stream, with an L2 flush before
    each timed step."""

    def __init__(self, torch, device):
        self.torch = torch
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def flush(self):
        self.flush_buf.fill_(1.0)

    def run(self, fn, steps, warmup, flush=True):
        """flush=False only for inputs larger than L2, which evict themselves."""
        torch = self.torch
        for _ in range(warmup):
            if flush:
                self.flush()
            fn()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        evs = []
        for _ in range(steps):
            if flush:
                self.flush()
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
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
    """cuBLAS TF32 GEMM throughput (context for the TF32 roofline)."""
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
        for _ in range(5):
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
    timer = Timer(torch, device)
    clocks = ClockSampler(device.index if device.index is not None else 0)

    # ---- headline: dense q8_0 OUT_PROD -------------------------------------
    a_np, b_np = synth.dense_quant(synth.TYPE_Q8_0, DENSE_M, DENSE_K, DENSE_N)
    a = torch.from_numpy(a_np).to(device)
    b = torch.from_numpy(b_np).to(device)
    ne_a = (DENSE_M, DENSE_K, 1, 1)
    out = torch.empty((1, 1, DENSE_N, DENSE_M), dtype=torch.float32, device=device)
    nws = op.oop_out_prod_workspace_size(op.TYPE_Q8_0, ne_a, (DENSE_N, DENSE_K, 1, 1))
    ws_buf = torch.empty(max(nws, 1), dtype=torch.uint8, device=device)
    flops = 2.0 * DENSE_M * DENSE_N * DENSE_K

    def dense_call():
        op.out_prod(a, b, a_type=op.TYPE_Q8_0, ne_a=ne_a, out=out, workspace=ws_buf,
                    path=op.PATH_TCGEN05)

    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for _ in range(args.warmup):
        timer.flush()
        dense_call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = []
    launches = 0
    t_region0 = time.perf_counter()
    for _ in range(args.steps):
        timer.flush()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        k0 = torch.cuda.Event(enable_timing=True)
        k1 = torch.cuda.Event(enable_timing=True)
        for e in (k0, k1):          # create the events before handing them over
            e.record(stream)
        op.profile_main_kernel(k0, k1)
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
    nbuf = op.oop_out_prod_host_buffer_size(op.TYPE_Q8_0, ne_a, (DENSE_N, DENSE_K, 1, 1))
    dev_buf = torch.empty(nbuf, dtype=torch.uint8, device=device)

    def e2e_call():
        op.out_prod_host(a_host, b_host, a_type=op.TYPE_Q8_0, ne_a=ne_a, out=dst_host,
                         device_buffer=dev_buf)

    for _ in range(max(1, args.warmup)):
        e2e_call()
    torch.cuda.synchronize()
    e2e_t = []
    for _ in range(args.steps):
        timer.flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_call()
        e2e_t.append(time.perf_counter() - t0)
    e2e_s = _barrier_max(torch, statistics.mean(e2e_t), ws)

    # ---- the other rows of the path (same run) ----------------------------
    parts = {}
    hbm = peaks["hbm_gbs"]

    def skinny_part(r, steps):
        an, bn = synth.lora_rank(r)
        ta, tb = torch.from_numpy(an).to(device), torch.from_numpy(bn).to(device)
        o = torch.empty((1, 1, r, 2560), dtype=torch.float32, device=device)
        t = timer.run(lambda: op.out_prod(ta, tb, out=o, path=op.PATH_SKINNY), steps, 3)
        byts = 4.0 * (2560 * 512 + r * 512 + 2560 * r)
        us = statistics.mean(t) * 1e3
        return {"workload": f"LoRA rank-{r} gradient: a [2560, 512] f32, b [{r}, 512]",
                "us": round(us, 3), "GB/s": round(byts / (us * 1e-6) / 1e9, 1),
                "frac_of_measured_hbm": round(byts / (us * 1e-6) / 1e9 / hbm, 4),
                "frac_of_8TBs": round(byts / (us * 1e-6) / 8e12, 4), "bytes": byts}

    for r in synth.LORA_RANKS:
        parts[f"lora_r{r}"] = skinny_part(r, max(args.steps, 20))

    # rank-r gradients for many slices in one launch (steady-state streaming).
    # src0 is 335 MB, larger than L2, so these steps need no flush; the
    # figure after a flush is reported beside it (the flush leaves up to 129 MB
    # of dirty lines that are written back during the call).
    nsl = 64
    an = synth.make_a(synth.TYPE_F32, (2560, 512, nsl, 1), 70)
    ta = torch.from_numpy(an).to(device)
    del an
    for r in synth.LORA_RANKS:
        bn = synth.make_b((r, 512, nsl, 1), 71, std=100.0, outliers=True)
        tb = torch.from_numpy(bn).to(device)
        o = torch.empty((1, nsl, r, 2560), dtype=torch.float32, device=device)
        call = (lambda tb=tb, o=o: op.out_prod(ta, tb, out=o, path=op.PATH_SKINNY))
        t = timer.run(call, max(args.steps, 10), 3, flush=False)
        tf = timer.run(call, max(args.steps, 10), 3)
        byts = 4.0 * nsl * (2560 * 512 + r * 512 + 2560 * r)
        us, usf = statistics.mean(t) * 1e3, statistics.mean(tf) * 1e3
        parts[f"lora_r{r}_x64_slices"] = {
            "workload": f"64 rank-{r} gradients in one launch: a [2560, 512, 64] f32, b [{r}, 512, 64]",
            "us": round(us, 3), "GB/s": round(byts / (us * 1e-6) / 1e9, 1),
            "frac_of_measured_hbm": round(byts / (us * 1e-6) / 1e9 / hbm, 4),
            "l2": "inputs larger than L2, no flush",
            "us_after_l2_flush": round(usf, 3),
            "frac_of_measured_hbm_after_flush": round(byts / (usf * 1e-6) / 1e9 / hbm, 4)}
        del tb, o
    del ta

    for n_seq in (1, 2):
        an, bn = synth.grouped_heads(n_seq)
        ta, tb = torch.from_numpy(an).to(device), torch.from_numpy(bn).to(device)
        o = torch.empty((n_seq, 16, 128, 128), dtype=torch.float32, device=device)
        t = timer.run(lambda: op.out_prod(ta, tb, out=o), max(args.steps, 20), 3)
        us = statistics.mean(t) * 1e3
        fl = 2.0 * 128 * 128 * 512 * 16 * n_seq
        # the same slices as one launch per slice (the per-slice loop)
        o2 = torch.empty_like(o)

        def per_slice():
            for i3 in range(n_seq):
                for i2 in range(16):
                    op.out_prod(ta[i3, i2 // 4], tb[i3, i2], out=o2[i3, i2], ne_a=(128, 512, 1, 1))

        t2 = timer.run(per_slice, max(args.steps // 2, 5), 2)
        parts[f"grouped_heads_x{n_seq}"] = {
            "workload": f"a [128, 512, 4, {n_seq}], b [128, 512, 16, {n_seq}], dps2 = 4",
            "us_one_launch": round(us, 3), "TFLOP/s": round(fl / (us * 1e-6) / 1e12, 3),
            "us_per_slice_loop": round(statistics.mean(t2) * 1e3, 3),
            "launches_per_slice_loop": 16 * n_seq}
        del ta, tb, o, o2

    # every dense shape, q8_0 and q4_0: whole call and tile kernel alone
    for m, k in synth.DENSE_MK:
        x = synth.normal(synth.tensor_seed(30), m * k, std=0.02).reshape(1, 1, k, m)
        bn = synth.make_b((DENSE_N, k, 1, 1), 31, std=1e3, outliers=True)
        tb = torch.from_numpy(bn).to(device)
        o = torch.empty((1, 1, DENSE_N, m), dtype=torch.float32, device=device)
        wsz = op.oop_out_prod_workspace_size(op.TYPE_Q8_0, (m, k, 1, 1), (DENSE_N, k, 1, 1))
        wsb = torch.empty(max(wsz, 1), dtype=torch.uint8, device=device)
        fl = 2.0 * m * DENSE_N * k
        for tid, tname, quant in ((synth.TYPE_Q8_0, "q8_0", synth.quantize_q8_0),
                                  (synth.TYPE_Q4_0, "q4_0", synth.quantize_q4_0)):
            ta = torch.from_numpy(quant(x)).to(device)

            def call():
                op.out_prod(ta, tb, a_type=tid, ne_a=(m, k, 1, 1), out=o, workspace=wsb,
                            path=op.PATH_TCGEN05)

            for _ in range(3):
                timer.flush()
                call()
            torch.cuda.synchronize()
            rec = []
            for _ in range(max(3, args.steps // 4)):
                timer.flush()
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                ev[2].record(stream)
                ev[3].record(stream)
                op.profile_main_kernel(ev[2], ev[3])
                ev[0].record(stream)
                call()
                ev[1].record(stream)
                rec.append(ev)
            torch.cuda.synchronize()
            us_call = statistics.mean(e[0].elapsed_time(e[1]) for e in rec) * 1e3
            us_kern = statistics.mean(e[2].elapsed_time(e[3]) for e in rec) * 1e3
            peak_tf32 = peaks["bf16_tflops"] * NOMINAL_TF32_OVER_BF16
            parts[f"dense_{tname}_m{m}_k{k}_n{DENSE_N}"] = {
                "us_call": round(us_call, 2), "us_tile_kernel": round(us_kern, 2),
                "TFLOP/s_call": round(fl / (us_call * 1e-6) / 1e12, 2),
                "TFLOP/s_tile_kernel": round(fl / (us_kern * 1e-6) / 1e12, 2),
                "pipe_frac_3xtf32": round(3 * fl / (us_kern * 1e-6) / 1e12 / peak_tf32, 4)}
            del ta
        del tb, o, wsb, x

    for wt, nm in ((synth.TYPE_F32, "f32"), (synth.TYPE_BF16, "bf16")):
        W, ids, g = synth.moe_back(wt)
        tW = torch.from_numpy(W.view(np.int16) if wt == synth.TYPE_BF16 else W).to(device)
        tids, tg = torch.from_numpy(ids).to(device), torch.from_numpy(g).to(device)
        o = torch.empty((512, 8, 2048), dtype=torch.float32, device=device)
        wsz = op.oop_mul_mat_id_back_workspace_size(wt, (2048, 768, 32), (8, 512))
        wsb = torch.empty(max(wsz, 1), dtype=torch.uint8, device=device)
        fl = 2.0 * 2048 * 768 * 8 * 512
        byts = W.nbytes + g.nbytes + 4.0 * 2048 * 8 * 512 + ids.nbytes
        entry = {"workload": f"E=32 W {nm} [2048, 768], 8 of 32 experts per token, 512 tokens"}
        for path, pname in ((op.PATH_TCGEN05, "grouped_tcgen05"), (op.PATH_SIMT, "per_slot")):
            t = timer.run(lambda: op.mul_mat_id_back(tW, tids, tg, w_type=wt, out=o, workspace=wsb,
                                                     path=path), max(3, args.steps // 4), 2)
            us = statistics.mean(t) * 1e3
            entry[pname] = {"us": round(us, 3), "TFLOP/s": round(fl / (us * 1e-6) / 1e12, 3),
                            "GB/s": round(byts / (us * 1e-6) / 1e9, 1)}
        parts[f"mul_mat_id_back_{nm}"] = entry
        del tW, tids, tg, o, wsb

    clk = clocks.stop()
    assert op.device_status() == 0, "device status word set"
    tf32_cublas = _cublas_tf32(torch, device)

    # ---- roofline of the dominant kernel (the tensor-core tile kernel) ----
    achieved = flops / (ms_main * 1e-3) / 1e12
    peak = peaks["bf16_tflops"] * NOMINAL_TF32_OVER_BF16
    roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "pipe_frac_3xtf32": round(3 * achieved / peak, 4),
            "peak_note": f"TF32 = {peak_kind} bf16 burst {peaks['bf16_tflops']} x nominal "
                         f"1.1/2.25 (of {peak_kind}); cuBLAS TF32 8192^3 in this run: "
                         f"{tf32_cublas:.0f} TFLOP/s",
            "kernel": "tc_out_prod_kernel (tcgen05 3xTF32), algorithmic 2*M*N*K per launch",
            "kernel_ms": round(ms_main, 4), "split_prepass_ms": round(ms_step - ms_main, 4),
            "traffic": TC_TRAFFIC_BYTES}

    cpu = cpu_baseline(args.cpu_seconds) if rank == 0 and ws == 1 else None
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded splitmix64 normals, q8_0-quantised weight, 0.2% outliers)",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{ws}",
                   "l2": "512 MB buffer written before every timed step",
                   "precision": "3xTF32 split on tensor cores, fp32 accumulation with Kahan fold"},
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
            "config": {"workload": WORKLOAD, "parallelism": "host cores"},
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
