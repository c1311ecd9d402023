#!/usr/bin/env python
"""Benchmark of the NF4 quantize -> double quant -> dequantize -> GEMV path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One STEP is one pass of the whole decode-side path over the Llama-7B decode
workload: for each of the three weights [4096x4096], [11008x4096] and
[4096x11008] (bf16 N(0, 0.02) with 0.1 % outliers, seeds 10-12; x ~ N(0, 1)
bf16, M = 1): nf4q_quantize_dq (absmax + codes + packing, then the double
quantization of the scales; one call, two kernels), nf4q_dequantize (bf16
out) and nf4q_gemv.  Inputs are resident in HBM when
the timed region starts; L2 is flushed (256 MiB write) before every step,
outside the step's events.  `value` is the step's algorithmic bytes divided
by its device time (CUDA events), summed over ranks.

The same run also times, on their own workloads, the prefill GEMM (14336x4096
weight, M = 64..2048, TFLOP/s), the GEMV alone with L2 flushed before each
launch (all three decode weights, and the 28672x8192 weight at M = 1..16 with
NF4 and FP4 codes; back-to-back launches over copies of the packed weight
that together exceed L2), and the 32-layer Llama-3-8B-shaped stack (whole-stack
quantize + double quant, and one decode token through its 224 GEMVs).

Multi-GPU: one process per GPU under torchrun; every rank runs the same
workload on its own GPU (replicas: the path has no exchange step), time is
the max over ranks, value the sum.  `--impl reference` times the CPU oracle
on a bounded sample of the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NF4 GEMV effective weight GB/s and % of HBM peak; NF4 GEMM TFLOP/s"
WORKLOAD = ("Llama-7B decode shapes [4096x4096], [11008x4096], [4096x11008], bf16 "
            "N(0,0.02) + 0.1% outliers, x bf16 N(0,1) M=1; step = quantize + double "
            "quant + dequantize + GEMV per weight")
NS_HBM_GBS = 8000.0   # the "~8 TB/s" HBM figure the target is stated against


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sust=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    except Exception:
        return dict(hbm=6400.0, bf16=1800.0, bf16_sust=1400.0, src="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (100 ms) while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.path is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ byte counts
def nbytes_state(n_elem):
    nb = n_elem // 64
    nd = (nb + 255) // 256
    return n_elem // 2 + nb + 4 * nd + 4     # packed + absmax_q + scale2 + offset


def kernel_bytes(N, K, M=1):
    n = N * K
    nb = n // 64
    nd = (nb + 255) // 256
    b = {
        "quantize": 2 * n + n // 2 + 4 * nb,
        "double_quant": 4 * nb + nb + 4 * nd + 4,
        "dequantize": nbytes_state(n) + 2 * n,
        "gemv": nbytes_state(n) + 2 * M * K + 2 * M * N,
    }
    b["quantize_dq"] = b["quantize"] + b["double_quant"]
    return b


# DRAM bytes (read + write) per call of each phase of the step, averaged over
# the three weights, from one ncu capture of this script (the launch list in
# profiles/ncu_launches_llama7b_decode_step.md).  They hold only for the
# kernel sources they were measured on: `traffic` is reported as null as soon
# as the digest of those sources (STEP_SOURCES) differs.
MEASURED_TRAFFIC = {"csrc_digest": "31ec09fb8be0ae02",
                    "quantize_dq": 75457172, "dequantize": 36857290, "gemv": 18425694}


# The sources of the step's kernels and of their launch code.
STEP_SOURCES = ("common.cuh", "tables.h", "lut.cuh", "tma.cuh", "quantize.cuh",
                "double_quant.cuh", "dequantize.cuh", "gemv_mma.cuh", "nf4q.cu")


def csrc_digest() -> str:
    import hashlib
    d = os.path.join(ROOT, "dequant_matmul_quantize_b300", "csrc")
    h = hashlib.sha256()
    for f in STEP_SOURCES:
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ ranks
def rank_env():
    """(rank, world size, local rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(v: float, world: int, dist=None, device=None) -> float:
    """The largest v over all ranks (an all-reduce MAX); v itself on one rank."""
    if world == 1:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank (one replica per GPU, weak scaling) moves
    bytes_per_rank_step per step, and the job's step time is the slowest
    rank's."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ------------------------------------------------------------------ our path
def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = rank_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import dequant_matmul_quantize_b300 as nq
    import synth
    from dequant_matmul_quantize_b300 import build
    build.build()
    L = nq.lib()
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    R = ctypes.byref

    def barrier():
        if world > 1:
            dist.barrier()

    def slowest(v):
        return max_over_ranks(v, world, dist, dev)

    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what} failed with status {st}")

    # ---- the decode workload
    mats = []
    for i in range(3):
        w, x = synth.llama7b_decode(i, device=dev)
        N, K = w.shape
        qw = nq.QuantizedWeight.empty(N, K, device=dev)
        ws = nq.dq_workspace(N * K // 64, dev)
        out = torch.empty(N, K, dtype=torch.bfloat16, device=dev)
        y = torch.empty(1, N, dtype=torch.bfloat16, device=dev)
        mats.append(dict(w=w, x=x, N=N, K=K, qw=qw, s=qw.struct(), ws=ws, out=out, y=y,
                         bytes=kernel_bytes(N, K)))
    names = ["quantize_dq", "dequantize", "gemv"]
    nphase = len(names)
    # per weight: quantize (with the first double-quant pass) + per-256 pass,
    # dequantize, gemv
    launches_per_step = 3 * (2 + 1 + 1)

    def launch(m, k, st=None):
        s = m["s"]
        sp_ = (st or stream).cuda_stream
        if k == 0:
            check(L.nf4q_quantize_dq(m["w"].data_ptr(), nq.IN_BF16, R(s), m["ws"].data_ptr(),
                                     m["ws"].numel(), sp_), "quantize_dq")
        elif k == 1:
            check(L.nf4q_dequantize(R(s), m["out"].data_ptr(), sp_), "dequantize")
        else:
            check(L.nf4q_gemv(R(s), m["x"].data_ptr(), 1, m["y"].data_ptr(), sp_), "gemv")

    # The timed step.  The three weights are independent problems: each gets
    # its own pair of streams.  On the first, quantize + double quant, then
    # dequantize; on the second, the GEMV as soon as the weight's quantized
    # state is ready.  Every stream first waits for the step's start and the
    # main stream waits for all of them at its end, so the step's events
    # bracket all of its work.
    s_a = [torch.cuda.Stream(dev) for _ in mats]
    s_b = [torch.cuda.Stream(dev) for _ in mats]
    Ent = lambda: torch.cuda.Event()
    ev_go = Ent()
    ev_q = [Ent() for _ in mats]
    ev_end = [Ent() for _ in range(2 * len(mats))]

    def fork(main):
        ev_go.record(main)
        for sa, sb in zip(s_a, s_b):
            sa.wait_event(ev_go)
            sb.wait_event(ev_go)

    def join(main):
        for i, (sa, sb) in enumerate(zip(s_a, s_b)):
            ev_end[2 * i].record(sa)
            ev_end[2 * i + 1].record(sb)
        for e in ev_end:
            main.wait_event(e)

    def step(main=None):
        main = main or stream
        fork(main)
        for i, m in enumerate(mats):
            launch(m, 0, s_a[i])
            ev_q[i].record(s_a[i])
            s_b[i].wait_event(ev_q[i])
            launch(m, 2, s_b[i])
            launch(m, 1, s_a[i])
        join(main)

    def step_serial(evs):
        j = 0
        for m in mats:
            for k in range(nphase):
                evs[j].record(stream)
                launch(m, k)
                j += 1
        evs[j].record(stream)

    # The step as one CUDA graph (its streams become branches), so that the
    # host's launch cost does not pace the device.
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    torch.cuda.synchronize()

    step_bytes = sum(m["bytes"][n] for m in mats for n in names)
    E = lambda: torch.cuda.Event(enable_timing=True)

    # per-phase breakdown: the same work one kernel at a time on one stream
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    n_serial = max(3, min(args.steps, 200))
    ser = [[E() for _ in range(3 * nphase + 1)] for _ in range(n_serial)]
    for i in range(n_serial):
        flush()
        step_serial(ser[i])
    torch.cuda.synchronize()
    kern_ms = {n: 0.0 for n in names}
    for evs in ser:
        for j in range(3 * nphase):
            kern_ms[names[j % nphase]] += evs[j].elapsed_time(evs[j + 1])
    serial_ms = sum(kern_ms.values())

    for _ in range(max(3, args.warmup)):
        flush()
        graph.replay()
    torch.cuda.synchronize()
    per_step = [(E(), E()) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush()
            per_step[i][0].record(stream)
            graph.replay()
            per_step[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        wall = time.perf_counter() - t0
    clocks = clk.summary()
    step_times = sorted(a.elapsed_time(b) for a, b in per_step)
    dev_ms = sum(step_times)

    def pct(q):
        return round(step_times[min(len(step_times) - 1, int(q * len(step_times)))], 4)
    dom = max(kern_ms, key=kern_ms.get)            # the largest share of the serial step
    dom_ms = kern_ms[dom] / n_serial * args.steps  # its launches, timed one by one
    dev_ms_max = slowest(dev_ms)
    ms_per_step = dev_ms_max / args.steps
    value = job_throughput(world, step_bytes, ms_per_step)

    # roofline of the kernel with the largest share of the step, timed with
    # events around each of its launches on its stream (the serial pass: the
    # graph's nodes carry no events)
    dom_bytes = sum(m["bytes"][dom] for m in mats)      # per step, 3 launches
    launches_dom = 3 * args.steps
    achieved = (dom_bytes * args.steps / launches_dom) / (dom_ms / launches_dom * 1e-3) / 1e9
    traffic_ok = csrc_digest() == MEASURED_TRAFFIC["csrc_digest"]
    roofline = {"kernel": "nf4q_" + dom, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm"], "unit": "GB/s", "frac": round(achieved / peaks["hbm"], 4),
                "peak_source": peaks["src"] + " HBM copy bandwidth",
                "bytes_per_launch": dom_bytes // 3,
                "traffic": MEASURED_TRAFFIC.get(dom) if traffic_ok else None,
                "traffic_note": "DRAM read+write per call from the ncu launch list; writes "
                                "still in L2 when the kernel ends are not counted",
                "share_of_serial_step": round(kern_ms[dom] / serial_ms, 3)}
    breakdown = {n: {"ms_per_step": round(kern_ms[n] / n_serial, 4),
                     "GB/s": round(sum(m["bytes"][n] for m in mats)
                                   / (kern_ms[n] / n_serial * 1e-3) / 1e9, 1),
                     "share": round(kern_ms[n] / serial_ms, 3),
                     "bytes_per_call": sum(m["bytes"][n] for m in mats) // 3,
                     "traffic_per_call": MEASURED_TRAFFIC.get(n) if traffic_ok else None}
                 for n in names}
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "ms_per_step_p10_p50_p90": [pct(0.1), pct(0.5), pct(0.9)],
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "bytes_per_step": step_bytes,
                   "l2": "flushed before every step (256 MiB write, outside the events)",
                   "streams": "one CUDA graph per step; each weight on its own two "
                              "branches: quantize + double quant then dequantize, and the "
                              "GEMV once the quantized state is ready",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "breakdown": {"note": f"the same step one kernel at a time on one stream "
                              f"({n_serial} steps, L2 flushed), "
                              f"{round(serial_ms / n_serial, 4)} ms per step", **breakdown},
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": round(wall, 4),
        "clocks": clocks,
    }

    # ---- e2e: host buffers, copies inside the timed region
    host_w = [m["w"].cpu().pin_memory() for m in mats]
    host_x = [m["x"].cpu().pin_memory() for m in mats]
    host_y = [torch.empty(1, m["N"], dtype=torch.bfloat16).pin_memory() for m in mats]
    h2d = sum(t.numel() * 2 for t in host_w) + sum(t.numel() * 2 for t in host_x)
    d2h = sum(t.numel() * 2 for t in host_y)

    def e2e_step():
        # the same streams as the timed step: each weight's inputs are copied
        # in on its first stream, its y copied out after its GEMV
        fork(stream)
        for i, (m, hw, hx, hy) in enumerate(zip(mats, host_w, host_x, host_y)):
            with torch.cuda.stream(s_a[i]):
                m["w"].copy_(hw, non_blocking=True)
                m["x"].copy_(hx, non_blocking=True)
            launch(m, 0, s_a[i])
            ev_q[i].record(s_a[i])
            s_b[i].wait_event(ev_q[i])
            launch(m, 2, s_b[i])
            with torch.cuda.stream(s_b[i]):
                hy.copy_(m["y"], non_blocking=True)
            launch(m, 1, s_a[i])
        join(stream)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = E(), E()
    barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = slowest(e0.elapsed_time(e1)) / e2e_steps
    result["e2e"] = {"value": round(job_throughput(world, step_bytes, e2e_ms), 1),
                     "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                     "api": "C ABI via the ctypes binding, pinned host buffers"}

    if not args.no_extras:
        result.update(run_extras(args, nq, L, synth, torch, dev, peaks, flush, E, stream))

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_sample()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_extras(args, nq, L, synth, torch, dev, peaks, flush, E, stream):
    """GEMV alone (L2 flushed before each launch), prefill GEMM, and the
    Llama-3-8B stack.  Each timed with CUDA events per launch."""
    out = {}
    sp = stream.cuda_stream
    R = ctypes.byref
    reps = 10

    def timed(fn, n=reps, do_flush=True):
        ts = []
        for _ in range(2):
            fn()
        for _ in range(n):
            if do_flush:
                flush()
            a, b = E(), E()
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what} failed with status {st}")

    def gemv_timed(qw, x, M, y, n_launch=None):
        """Average GEMV time over back-to-back launches that rotate through
        copies of the packed weight and its int8 scales (together > 400 MB,
        so every launch reads its weight from HBM); one event pair around
        all of them, best of three rounds."""
        ncopy = max(4, -(-400_000_000 // (qw.rows * qw.cols // 2)))
        cps = [nq.QuantizedWeight(qw.packed.clone(), qw.absmax, qw.absmax_q.clone(), qw.scale2,
                                  qw.offset, qw.rows, qw.cols, qw.code, qw.double_quant)
               for _ in range(ncopy)]
        structs = [c.struct() for c in cps]
        for st in structs:
            check(L.nf4q_gemv(R(st), x.data_ptr(), M, y.data_ptr(), sp), "gemv")
        n = n_launch or 4 * ncopy
        best = None
        for _ in range(3):
            a, b = E(), E()
            a.record(stream)
            for i in range(n):
                L.nf4q_gemv(R(structs[i % ncopy]), x.data_ptr(), M, y.data_ptr(), sp)
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b) / n
            best = ms if best is None else min(best, ms)
        del cps
        return best

    # GEMV alone on the three decode weights
    gem = []
    tot_b, tot_ms = 0, 0.0
    for i in range(3):
        w, x = synth.llama7b_decode(i, device=dev)
        qw = nq.quantize(w)
        y = torch.empty(1, w.shape[0], dtype=torch.bfloat16, device=dev)
        ms = gemv_timed(qw, x, 1, y)
        b = kernel_bytes(*w.shape)["gemv"]
        gem.append({"shape": list(w.shape), "us": round(ms * 1e3, 2),
                    "GB/s": round(b / (ms * 1e-3) / 1e9, 1)})
        tot_b += b
        tot_ms += ms
        del w, qw
    gbs = tot_b / (tot_ms * 1e-3) / 1e9
    out["gemv"] = {"workload": "Llama-7B decode weights, M=1, each launch reads its weight "
                               "from HBM (rotating copies > L2)",
                   "GB/s": round(gbs, 1), "frac_measured_hbm": round(gbs / peaks["hbm"], 4),
                   "frac_8TBps": round(gbs / NS_HBM_GBS, 4), "per_weight": gem}

    # 70B-MLP weight, M sweep, NF4 and FP4
    w = synth.mlp70b_weight(device=dev)
    sweep = []
    for code in ("nf4", "fp4"):
        qw = nq.quantize(w, code)
        for M in (1, 4, 8, 16):
            x = synth.mlp70b_x(M, device=dev)
            y = torch.empty(M, w.shape[0], dtype=torch.bfloat16, device=dev)
            ms = gemv_timed(qw, x, M, y)
            b = kernel_bytes(*w.shape, M=M)["gemv"]
            sweep.append({"code": code, "M": M, "us": round(ms * 1e3, 2),
                          "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                          "frac_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peaks["hbm"], 4)})
        del qw
    # fp16 compute dtype (NF4 codes, fp16 x and y)
    qw = nq.quantize(w, "nf4", compute_dtype="f16")
    for M in (1, 16):
        x = synth.mlp70b_x(M, device=dev).to(torch.float16)
        y = torch.empty(M, w.shape[0], dtype=torch.float16, device=dev)
        ms = gemv_timed(qw, x, M, y)
        b = kernel_bytes(*w.shape, M=M)["gemv"]
        sweep.append({"code": "nf4", "compute_dtype": "f16", "M": M, "us": round(ms * 1e3, 2),
                      "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                      "frac_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peaks["hbm"], 4)})
    del qw
    del w
    out["gemv_70b_mlp"] = {"workload": "28672x8192 bf16 N(0,0.015), rotating copies > L2",
                           "points": sweep}

    # prefill GEMM
    w = synth.prefill_weight(device=dev)
    qw = nq.quantize(w)
    s = qw.struct()
    pts = []
    for M in (16, 32, 64, 256, 512, 2048):
        x = synth.prefill_x(M, device=dev)
        y = torch.empty(M, w.shape[0], dtype=torch.bfloat16, device=dev)
        fn = (lambda: L.nf4q_gemm(R(s), x.data_ptr(), M, y.data_ptr(), sp))
        ms = timed(fn)
        fl = 2.0 * M * w.shape[0] * w.shape[1]
        tf = fl / (ms * 1e-3) / 1e12
        ms_gemv = None
        if M <= 16:
            ms_gemv = timed(lambda: L.nf4q_gemv(R(s), x.data_ptr(), M, y.data_ptr(), sp))
        # the two-kernel alternative: dequantize, then cuBLAS bf16
        deq = torch.empty_like(w)
        def two():
            L.nf4q_dequantize(R(s), deq.data_ptr(), sp)
            torch.matmul(x, deq.T, out=y)
        ms_two = timed(two)
        pts.append({"M": M, "us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                    "frac_bf16_burst": round(tf / peaks["bf16"], 4),
                    "us_dequant_plus_cublas": round(ms_two * 1e3, 1),
                    **({"us_gemv": round(ms_gemv * 1e3, 1)} if ms_gemv else {})})
        del deq
    # fp16 compute dtype at M = 2048 (fp16 X and Y, f16 tcgen05 MMA); the
    # bf16 peak stands in for fp16's (same nominal dense rate)
    qh = nq.quantize(w, "nf4", compute_dtype="f16")
    sh = qh.struct()
    M = 2048
    xh = synth.prefill_x(M, device=dev).to(torch.float16)
    yh = torch.empty(M, w.shape[0], dtype=torch.float16, device=dev)
    ms = timed(lambda: L.nf4q_gemm(R(sh), xh.data_ptr(), M, yh.data_ptr(), sp))
    tf = 2.0 * M * w.shape[0] * w.shape[1] / (ms * 1e-3) / 1e12
    pts.append({"M": M, "compute_dtype": "f16", "us": round(ms * 1e3, 1),
                "TFLOP/s": round(tf, 1), "frac_bf16_burst": round(tf / peaks["bf16"], 4)})
    del qh, xh, yh
    out["gemm"] = {"workload": "prefill 14336x4096 NF4 weight, X bf16 [M x 4096] (and one "
                               "fp16 point)",
                   "points": pts, "peak_bf16_tflops": peaks["bf16"],
                   "peak_source": peaks["src"] + " cuBLAS bf16 burst"}

    # input gradient through the frozen weight: dX [M x 4096] = dY [M x 14336] . w_hat
    N, K = w.shape
    pts = []
    for M in (256, 512, 2048, 4096):
        dy = synth.activations(M, N, seed=M + N, device=dev)
        dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        ms = timed(lambda: L.nf4q_matmul_dx(R(s), dy.data_ptr(), N, M, dx.data_ptr(), sp))
        deq = torch.empty_like(w)

        def two():
            L.nf4q_dequantize(R(s), deq.data_ptr(), sp)
            torch.matmul(dy, deq, out=dx)
        ms_two = timed(two)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        pts.append({"M": M, "us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                    "frac_bf16_burst": round(tf / peaks["bf16"], 4),
                    "us_dequant_plus_cublas": round(ms_two * 1e3, 1)})
        del deq, dy, dx
    out["gemm_dx"] = {"workload": "QLoRA base-layer backward: dX = dY . w_hat, prefill "
                                  "14336x4096 NF4 weight, dY bf16 [M x 14336]",
                      "points": pts, "peak_bf16_tflops": peaks["bf16"],
                      "peak_source": peaks["src"] + " cuBLAS bf16 burst"}
    del w, qw

    # LLM.int8(): vector-wise int8 weight, decomposition matmul at decode sizes
    w = synth.int8_mlp70b_weight(device=dev)
    N, K = w.shape
    wq = nq.int8_quantize_weight(w)
    ms_q = timed(lambda: nq.int8_quantize_weight(w), n=3)
    cps = [nq.Int8Weight(wq.q.clone(), wq.scale, N, K) for _ in range(2)]
    pts = []
    for M in (1, 4, 8, 16):
        x = synth.int8_mlp70b_x(M, device=dev)
        ws = nq.int8_workspace(M, K, dev)
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        for c in cps:
            nq.int8_matmul(c, x, workspace=ws, out=y)
        best = None
        for _ in range(3):
            a, b = E(), E()
            a.record(stream)
            for i in range(10):
                nq.int8_matmul(cps[i % 2], x, workspace=ws, out=y)
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b) / 10
            best = ms if best is None else min(best, ms)
        by = N * K + 4 * N + 2 * M * K + 2 * M * N     # int8 weight + scales + x + y
        pts.append({"M": M, "us": round(best * 1e3, 1), "GB/s": round(by / (best * 1e-3) / 1e9, 1),
                    "frac_measured_hbm": round(by / (best * 1e-3) / 1e9 / peaks["hbm"], 4)})
    del cps, wq
    out["llm_int8"] = {"workload": "fp16 28672x8192 N(0,0.015) weight quantized to int8 per "
                                   "row; x fp16 N(0,1) with 0.5 % outlier feature columns x20; "
                                   "threshold 6.0; two weight copies alternate (> L2)",
                       "quantize_weight_us": round(ms_q * 1e3, 1),
                       "quantize_weight_GB/s": round(3 * N * K / (ms_q * 1e-3) / 1e9, 1),
                       "points": pts}
    del w

    # Llama-3-8B stack: whole-stack quantize + double quant, one decode token
    if not args.no_stack:
        stack = []
        tot_n = 0
        for layer in range(synth.LLAMA3_8B_LAYERS):
            for mid in range(7):
                w = synth.llama3_8b_matrix(layer, mid, device=dev)
                x = synth.llama3_8b_x(layer, mid, device=dev)
                qw = nq.QuantizedWeight.empty(*w.shape, device=dev)
                ws = nq.dq_workspace(w.numel() // 64, dev)
                y = torch.empty(1, w.shape[0], dtype=torch.bfloat16, device=dev)
                stack.append((w, x, qw, qw.struct(), ws, y))
                tot_n += w.numel()

        def quant_all():
            for w, x, qw, s, ws, y in stack:
                L.nf4q_quantize_dq(w.data_ptr(), nq.IN_BF16, R(s), ws.data_ptr(), ws.numel(), sp)

        def token():
            for w, x, qw, s, ws, y in stack:
                L.nf4q_gemv(R(s), x.data_ptr(), 1, y.data_ptr(), sp)

        qms = timed(quant_all, n=3)
        qbytes = sum(kernel_bytes(*t[0].shape)["quantize_dq"] for t in stack)
        tms = timed(token, n=5)
        tbytes = sum(kernel_bytes(*t[0].shape)["gemv"] for t in stack)
        # the same 224 launches captured once in a CUDA graph and replayed:
        # no host work between kernels
        gs = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            for w, x, qw, s, ws, y in stack:
                check(L.nf4q_gemv(R(s), x.data_ptr(), 1, y.data_ptr(), gs.cuda_stream), "gemv")
            gs.synchronize()
            with torch.cuda.graph(graph, stream=gs):
                for w, x, qw, s, ws, y in stack:
                    L.nf4q_gemv(R(s), x.data_ptr(), 1, y.data_ptr(), gs.cuda_stream)
        torch.cuda.synchronize()
        gms = timed(graph.replay, n=5)
        out["llama3_8b_stack"] = {
            "workload": "32 layers x {q,k,v,o,gate,up,down}, 6.98e9 weights, bf16 N(0,0.02)",
            "quantize_dq_ms": round(qms, 3), "quantize_dq_GB/s": round(qbytes / (qms * 1e-3) / 1e9, 1),
            "decode_token_ms": round(tms, 4), "decode_token_GB/s": round(tbytes / (tms * 1e-3) / 1e9, 1),
            "decode_token_graph_ms": round(gms, 4),
            "decode_token_graph_GB/s": round(tbytes / (gms * 1e-3) / 1e9, 1),
            "decode_gemv_launches": len(stack)}
        del graph
        del stack
    return out


# ------------------------------------------------------------------ oracle (CPU)
def _limit_threads():
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(1)
    except Exception:
        return None


_DECODE_CPU = None


def _decode_cpu():
    """The three decode weights and their x rows on the CPU (drawn once)."""
    global _DECODE_CPU
    if _DECODE_CPU is None:
        import synth
        _DECODE_CPU = [synth.llama7b_decode(i, device="cpu") for i in range(3)]
    return _DECODE_CPU


def oracle_sample(rows=None, weights=(0, 1, 2)):
    """The oracle's whole path - quantize, double quant, dequantize, fp64
    GEMV - on the first `rows` rows (all if None) of the given decode
    weights.  Returns (seconds, algorithmic bytes of the same work on the GPU
    path)."""
    import numpy as np
    import torch
    from oracle import nf4_oracle as o
    tot, by = 0.0, 0
    for i in weights:
        w, x = _decode_cpu()[i]
        wf = (w if rows is None else w[:rows]).float().numpy()
        xb = x.view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        r = o.quantize_full(wf)
        o.matmul_ref(xb, r["w_hat"].reshape(wf.shape))
        tot += time.perf_counter() - t0
        by += sum(kernel_bytes(*wf.shape).values())
    return tot, by


def cpu_baseline_sample():
    """One whole decode step of the oracle (all three weights, every row),
    single-threaded: about 10-20 s on a server core."""
    import os
    lim = _limit_threads()
    dt, b = oracle_sample()
    if lim is not None:
        lim.unregister() if hasattr(lim, "unregister") else None
    return {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 3),
            "host_cpus": os.cpu_count(), "affinity": len(os.sched_getaffinity(0)),
            "sample": "one whole step: the three decode weights, every row - quantize + "
                      "double quant + dequantize + fp64 GEMV (NumPy, one thread)"}


def run_reference(args):
    rank, world, _ = rank_env()
    if rank != 0:
        return
    lim = _limit_threads()
    rows = 128  # per step, so that a run of --steps 1000 ends in a couple of minutes
    for _ in range(max(3, args.warmup)):
        oracle_sample(rows, weights=(0,))
    tot, b = 0.0, 0
    for _ in range(args.steps):
        dt, bb = oracle_sample(rows, weights=(0,))
        tot += dt
        b += bb
    value = b / tot / 1e9
    sample = (f"rows 0..{rows - 1} of the 4096x4096 decode weight per step: quantize + "
              "double quant + dequantize + fp64 GEMV (NumPy, one thread)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="only the step and e2e")
    ap.add_argument("--no-stack", action="store_true", help="skip the 7B-weight stack")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
