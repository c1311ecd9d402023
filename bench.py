#!/usr/bin/env python
"""Benchmark of the NF4 decode GEMV, with the rest of the path as extras.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One STEP is one decode token through the 32-layer Llama-3-8B-shaped stack:
224 NF4 GEMVs (M = 1) over the weights q [4096x4096], k, v [1024x4096],
o [4096x4096], gate, up [14336x4096] and down [4096x14336] of every layer
(bf16 N(0, 0.02), seed 1000 * layer + matrix, quantized once to NF4 with
double quantization before timing; x ~ N(0, 1) bf16, one per layer input:
q, k and v share theirs, as do gate and up).  They run as 128 launches, as a
decoder issues them: per layer the groups (q, k, v), (o), (gate, up) and
(down), each one nf4q_gemv_multi_ex call with NF4Q_GEMV_WEIGHTS_STATIC (the
weights are quantized once before timing and never written again, so each
launch may load its first weight tiles while the one before it finishes;
x is read after it).  The packed weights and scales
(3.61 GB) are far larger than L2, so every step reads them from HBM.  The
launches are one CUDA graph; `value` is the token's algorithmic bytes
(packed codes + int8 scales + scale2 + offset + x + y of every GEMV) over
its device time, summed over ranks.

The same run also reports, each on its own workload: the whole path of the
Llama-7B decode shapes (quantize + double quant, dequantize and GEMV of
[4096x4096], [11008x4096], [4096x11008]), the GEMV alone on those weights
and on the 28672x8192 weight at M = 1..16 with NF4 and FP4 codes (the
block-scale-folded kernel and the exact one), the whole-stack quantization,
the prefill GEMM (14336x4096, M = 16..2048, TFLOP/s, against dequantize +
cuBLAS), the QLoRA input gradient and the LLM.int8() matmul.

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
WORKLOAD = ("Llama-3-8B-shaped stack, 32 layers x {q,k,v,o,gate,up,down}, bf16 N(0,0.02), "
            "NF4 blocksize 64 + double quant; step = one decode token: 224 NF4 GEMVs in 128 "
            "launches (q/k/v and gate/up share their x), M=1, x bf16 N(0,1)")
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


# DRAM bytes (read + write) per launch of the GEMV kernel on the decode
# token: the mean over layer 0's four launches (every layer has the same
# shapes), from one ncu capture of dram__bytes_read.sum and
# dram__bytes_write.sum (`python profile_cases.py layer`, the second pass's
# four gemv_lut_kernel launches).  They hold only for the kernel sources they
# were measured on: `traffic` is reported as null as soon as the digest of
# those sources' code (STEP_SOURCES, comments and blank space left out)
# differs.
MEASURED_TRAFFIC = {"csrc_digest": "ed3b68c4f60fdfb5", "gemv_per_launch": 28178560}


# The sources of the step's kernel and of its launch code.
STEP_SOURCES = ("common.cuh", "tables.h", "lut.cuh", "tma.cuh", "gemv_lut.cuh",
                "gemv_mma.cuh", "nf4q.cu")


def code_of(text: str) -> str:
    """C/C++ source without its comments and with blank space collapsed (the
    sources' string literals hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def csrc_digest() -> str:
    import hashlib
    d = os.path.join(ROOT, "dequant_matmul_quantize_b300", "csrc")
    h = hashlib.sha256()
    for f in STEP_SOURCES:
        h.update(f.encode())
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(code_of(fh.read()).encode())
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
# the launches of one layer: (name, matrix ids of LLAMA3_8B_LAYER sharing x)
GROUPS = (("qkv", (0, 1, 2)), ("o", (3,)), ("gate_up", (4, 5)), ("down", (6,)))


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
    E = lambda: torch.cuda.Event(enable_timing=True)

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

    # ---- the stack: bf16 weights drawn on the device, quantized once (the
    # whole-stack quantize + double quant is timed here as an extra)
    bf = []
    for layer in range(synth.LLAMA3_8B_LAYERS):
        for mid in range(7):
            bf.append(synth.llama3_8b_matrix(layer, mid, device=dev))
    mats = []
    for i, w in enumerate(bf):
        N, K = w.shape
        qw = nq.QuantizedWeight.empty(N, K, device=dev)
        mats.append(dict(qw=qw, s=qw.struct(), N=N, K=K, mid=i % 7, layer=i // 7,
                         ws=nq.dq_workspace(N * K // 64, dev),
                         y=torch.empty(1, N, dtype=torch.bfloat16, device=dev)))

    def quant_all():
        for w, m in zip(bf, mats):
            check(L.nf4q_quantize_dq(w.data_ptr(), nq.IN_BF16, R(m["s"]), m["ws"].data_ptr(),
                                     m["ws"].numel(), sp), "quantize_dq")

    quant_all()
    torch.cuda.synchronize()
    q_ms = []
    for _ in range(3):
        a, b = E(), E()
        a.record(stream)
        quant_all()
        b.record(stream)
        b.synchronize()
        q_ms.append(a.elapsed_time(b))
    q_bytes = sum(kernel_bytes(*w.shape)["quantize_dq"] for w in bf)
    stack_quant = {"workload": "the 224 stack weights, bf16 in, nf4q_quantize_dq each",
                   "ms": round(min(q_ms), 3),
                   "GB/s": round(q_bytes / (min(q_ms) * 1e-3) / 1e9, 1),
                   "frac_measured_hbm": round(q_bytes / (min(q_ms) * 1e-3) / 1e9 / peaks["hbm"], 4),
                   "bytes": q_bytes}
    del bf
    torch.cuda.empty_cache()

    # the token's launches: per layer q/k/v (one x), o, gate/up (one x) and
    # down, each group one nf4q_gemv_multi_ex call (weights static).  All x of a token live in one
    # buffer and all y in another (views per launch), so that a step's inputs
    # and outputs cross PCIe in one copy each.
    n_x = sum(mats[layer * 7 + mids[0]]["K"] for layer in range(synth.LLAMA3_8B_LAYERS)
              for _, mids in GROUPS)
    x_all = torch.empty(n_x, dtype=torch.bfloat16, device=dev)
    y_all = torch.empty(sum(m["N"] for m in mats), dtype=torch.bfloat16, device=dev)
    yo = 0
    for m in mats:
        m["y"] = y_all[yo:yo + m["N"]].view(1, m["N"])
        yo += m["N"]
    groups = []
    xo = 0
    for layer in range(synth.LLAMA3_8B_LAYERS):
        for name, mids in GROUPS:
            ms_ = [mats[layer * 7 + mid] for mid in mids]
            x = x_all[xo:xo + ms_[0]["K"]].view(1, ms_[0]["K"])
            x.copy_(synth.llama3_8b_x(layer, mids[0], device=dev))
            xo += ms_[0]["K"]
            grp = dict(name=name, mats=ms_, x=x, K=ms_[0]["K"],
                       bytes=sum(nbytes_state(m["N"] * m["K"]) + 2 * m["N"] for m in ms_)
                       + 2 * ms_[0]["K"])
            grp["wp"] = (ctypes.POINTER(nq.NF4QWeight) * len(ms_))(
                *[ctypes.pointer(m["s"]) for m in ms_])
            grp["yp"] = (ctypes.c_void_p * len(ms_))(*[m["y"].data_ptr() for m in ms_])
            groups.append(grp)
    token_bytes = sum(g_["bytes"] for g_ in groups)

    def launch_group(g_, st):
        check(L.nf4q_gemv_multi_ex(g_["wp"], len(g_["mats"]), g_["x"].data_ptr(), 1, g_["yp"],
                                   nq.GEMV_WEIGHTS_STATIC, st), "gemv_multi_ex")

    # ---- the token as one CUDA graph of its 128 launches
    gs = torch.cuda.Stream(dev)

    def capture(subset):
        with torch.cuda.stream(gs):
            for g_ in subset:
                launch_group(g_, gs.cuda_stream)
            gs.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gs):
                for g_ in subset:
                    launch_group(g_, gs.cuda_stream)
        torch.cuda.synchronize()
        return g

    graph = capture(groups)
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    per_step = [(E(), E()) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            per_step[i][0].record(stream)
            graph.replay()
            per_step[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        wall = time.perf_counter() - t0
    clocks = clk.summary()
    step_times = sorted(a.elapsed_time(b) for a, b in per_step)
    dev_ms = slowest(sum(step_times))
    ms_per_step = dev_ms / args.steps
    value = job_throughput(world, token_bytes, ms_per_step)

    def pct(q):
        return round(step_times[min(len(step_times) - 1, int(q * len(step_times)))], 4)

    # per group kind: the 32 launches of one kind as their own graph
    by_type = {}
    for name, mids in GROUPS:
        sub = [g_ for g_ in groups if g_["name"] == name]
        g = capture(sub)
        for _ in range(3):
            g.replay()
        a, b = E(), E()
        a.record(stream)
        for _ in range(10):
            g.replay()
        b.record(stream)
        b.synchronize()
        ms = a.elapsed_time(b) / 10 / len(sub)
        by = sub[0]["bytes"]
        by_type[name] = {"shapes": [[m["N"], m["K"]] for m in sub[0]["mats"]],
                         "us": round(ms * 1e3, 2), "GB/s": round(by / (ms * 1e-3) / 1e9, 1),
                         "frac_measured_hbm": round(by / (ms * 1e-3) / 1e9 / peaks["hbm"], 4)}
        del g

    # roofline of the step's one kernel: algorithmic bytes per launch over
    # the average launch time, both over the timed steps
    launches = len(groups)
    achieved = (token_bytes / launches) / (ms_per_step / launches * 1e-3) / 1e9
    traffic_ok = MEASURED_TRAFFIC["csrc_digest"] == csrc_digest()
    roofline = {"kernel": "nf4q_gemv (gemv_lut_kernel, block-scale folded)", "bound": "hbm",
                "achieved": round(achieved, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm"], 4),
                "peak_source": peaks["src"] + " HBM copy bandwidth",
                "frac_of_8TBps": round(achieved / NS_HBM_GBS, 4),
                "bytes_per_launch": token_bytes // launches,
                "traffic": MEASURED_TRAFFIC["gemv_per_launch"] if traffic_ok else None,
                "traffic_note": "DRAM read+write per launch, averaged over the token's "
                                "launches, from an ncu capture of the same kernel sources"}
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "ms_per_step_p10_p50_p90": [pct(0.1), pct(0.5), pct(0.9)],
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": token_config(world),
        "roofline": roofline,
        "gemv_by_group": by_type,
        "gpu_launches": launches * args.steps,
        "wall_s_timed_region": round(wall, 4),
        "clocks": clocks,
    }

    # ---- e2e: the token as a serving loop runs it: x copied in from pinned
    # host memory and each layer's y read back into pinned host memory, the
    # copies on their own streams so that they overlap the kernels (x in
    # copies of layers 0, 1, 2-3, 4-7, 8-15 and 16-31, each layer waiting for
    # the one that holds its x; a layer's y is read as soon as
    # its launches are done), the public C-ABI calls of the token as above -
    # all of it one CUDA graph per step - and the host waiting for the last y
    host_x = x_all.cpu().pin_memory()
    host_y = torch.empty(y_all.numel(), dtype=torch.bfloat16).pin_memory()
    h2d = host_x.numel() * 2
    d2h = host_y.numel() * 2
    per_layer = len(GROUPS)
    x_span, y_span = [], []  # element ranges of each layer's x and y
    for layer in range(synth.LLAMA3_8B_LAYERS):
        gl = groups[layer * per_layer:(layer + 1) * per_layer]
        x0 = gl[0]["x"].data_ptr() - x_all.data_ptr()
        x1 = gl[-1]["x"].data_ptr() - x_all.data_ptr() + 2 * gl[-1]["K"]
        x_span.append((x0 // 2, x1 // 2))
        ms_ = [m for g_ in gl for m in g_["mats"]]
        y0 = min(m["y"].data_ptr() for m in ms_) - y_all.data_ptr()
        y1 = max(m["y"].data_ptr() + 2 * m["N"] for m in ms_) - y_all.data_ptr()
        y_span.append((y0 // 2, y1 // 2))
    assert x_span[0][0] == 0 and x_span[-1][1] == x_all.numel()
    assert y_span[0][0] == 0 and y_span[-1][1] == y_all.numel()
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_body():
        fork = torch.cuda.Event()
        fork.record(gs)
        h2d_s.wait_event(fork)
        d2h_s.wait_event(fork)
        # x in copies that double in layers (0, 1, 2-3, 4-7, ...): each lands
        # long before its first layer runs, and only the first launch of
        # each waits for it
        x_ready = {}
        with torch.cuda.stream(h2d_s):
            lo = 0
            while lo < synth.LLAMA3_8B_LAYERS:
                hi = min(max(1, 2 * lo), synth.LLAMA3_8B_LAYERS)
                a, b = x_span[lo][0], x_span[hi - 1][1]
                x_all[a:b].copy_(host_x[a:b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(h2d_s)
                x_ready[lo] = ev
                lo = hi
        for layer in range(synth.LLAMA3_8B_LAYERS):
            if layer in x_ready:
                gs.wait_event(x_ready[layer])
            for g_ in groups[layer * per_layer:(layer + 1) * per_layer]:
                launch_group(g_, gs.cuda_stream)
            done = torch.cuda.Event()
            done.record(gs)
            d2h_s.wait_event(done)
            a, b = y_span[layer]
            with torch.cuda.stream(d2h_s):
                host_y[a:b].copy_(y_all[a:b], non_blocking=True)
        join = torch.cuda.Event()
        join.record(d2h_s)
        gs.wait_event(join)
        join2 = torch.cuda.Event()
        join2.record(h2d_s)
        gs.wait_event(join2)

    with torch.cuda.stream(gs):
        e2e_body()
    gs.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=gs):
        e2e_body()
    torch.cuda.synchronize()

    def e2e_step():
        e2e_graph.replay()
        gs.synchronize()

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = slowest((time.perf_counter() - t0) * 1e3) / e2e_steps
    # the y that crossed to the host is the step's y
    if not torch.equal(host_y, y_all.cpu()):
        raise SystemExit("e2e: the y read back differs from the device's")
    result["e2e"] = {"value": round(job_throughput(world, token_bytes, e2e_ms), 1),
                     "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                     "api": "the token's nf4q_gemv_multi_ex C-ABI calls (ctypes "
                            "binding); every step x copied in from pinned host memory (copies of "
                            "layers 0, 1, 2-3, 4-7, 8-15, 16-31, each layer waiting for its own) "
                            "and each layer's y read back to "
                            "pinned host memory as soon as its launches are done, on copy streams "
                            "that overlap the kernels, all of it captured once in a CUDA graph "
                            "and replayed per step; host synchronised per step, host wall clock "
                            "around the steps"}
    result["llama3_8b_stack_quantize"] = stack_quant
    del mats, groups, graph
    torch.cuda.empty_cache()

    if not args.no_extras:
        result.update(run_extras(args, nq, L, synth, torch, dev, peaks, flush, E, stream))

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result.update(cpu_baselines())
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_extras(args, nq, L, synth, torch, dev, peaks, flush, E, stream):
    """The whole path on the Llama-7B decode shapes, the GEMV alone on its
    other workloads (both kernels), prefill GEMM, QLoRA input gradient and
    LLM.int8().  Each timed with CUDA events."""
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

    out["path_step"] = path_step(args, nq, L, synth, torch, dev, peaks, flush, E, stream)

    def gemv_timed(qw, x, M, y, fn=None):
        """Average GEMV time over launches that rotate through copies of the
        packed weight and its int8 scales (together > 400 MB, so every
        launch reads its weight from HBM), captured in a CUDA graph so that
        host launch cost does not count; best of three replays."""
        fn = fn or L.nf4q_gemv
        ncopy = max(4, -(-400_000_000 // (qw.rows * qw.cols // 2)))
        cps = [nq.QuantizedWeight(qw.packed.clone(), qw.absmax, qw.absmax_q.clone(), qw.scale2,
                                  qw.offset, qw.rows, qw.cols, qw.code, qw.double_quant,
                                  qw.compute_dtype)
               for _ in range(ncopy)]
        structs = [c.struct() for c in cps]
        n = 4 * ncopy
        gs = torch.cuda.Stream(dev)
        with torch.cuda.stream(gs):
            for st in structs:
                check(fn(R(st), x.data_ptr(), M, y.data_ptr(), gs.cuda_stream), "gemv")
            gs.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gs):
                for i in range(n):
                    fn(R(structs[i % ncopy]), x.data_ptr(), M, y.data_ptr(), gs.cuda_stream)
        torch.cuda.synchronize()
        best = None
        for _ in range(3):
            a, b = E(), E()
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b) / n
            best = ms if best is None else min(best, ms)
        del cps, g
        return best

    # GEMV alone on the three decode weights, both kernels
    gem = []
    tot_b, tot_ms, tot_ms_x = 0, 0.0, 0.0
    for i in range(3):
        w, x = synth.llama7b_decode(i, device=dev)
        qw = nq.quantize(w)
        y = torch.empty(1, w.shape[0], dtype=torch.bfloat16, device=dev)
        ms = gemv_timed(qw, x, 1, y)
        ms_x = gemv_timed(qw, x, 1, y, L.nf4q_gemv_exact)
        b = kernel_bytes(*w.shape)["gemv"]
        gem.append({"shape": list(w.shape), "us": round(ms * 1e3, 2),
                    "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                    "us_exact": round(ms_x * 1e3, 2)})
        tot_b += b
        tot_ms += ms
        tot_ms_x += ms_x
        del w, qw
    gbs = tot_b / (tot_ms * 1e-3) / 1e9
    out["gemv_llama7b"] = {
        "workload": "Llama-7B decode weights, M=1, each launch reads its weight from HBM "
                    "(rotating copies > L2), launches in a CUDA graph",
        "GB/s": round(gbs, 1), "frac_measured_hbm": round(gbs / peaks["hbm"], 4),
        "frac_8TBps": round(gbs / NS_HBM_GBS, 4),
        "GB/s_exact": round(tot_b / (tot_ms_x * 1e-3) / 1e9, 1), "per_weight": gem}

    # 70B-MLP weight, M sweep, NF4 and FP4, both kernels
    w = synth.mlp70b_weight(device=dev)
    sweep = []
    for code in ("nf4", "fp4"):
        qw = nq.quantize(w, code)
        for M in (1, 2, 4, 8, 16):
            x = synth.mlp70b_x(M, device=dev)
            y = torch.empty(M, w.shape[0], dtype=torch.bfloat16, device=dev)
            ms = gemv_timed(qw, x, M, y)
            ms_x = gemv_timed(qw, x, M, y, L.nf4q_gemv_exact)
            b = kernel_bytes(*w.shape, M=M)["gemv"]
            sweep.append({"code": code, "M": M, "us": round(ms * 1e3, 2),
                          "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                          "frac_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peaks["hbm"], 4),
                          "us_exact": round(ms_x * 1e3, 2)})
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
    out["gemv_70b_mlp"] = {"workload": "28672x8192 bf16 N(0,0.015), rotating copies > L2; "
                                       "us = nf4q_gemv, us_exact = nf4q_gemv_exact",
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

    return out


def path_step(args, nq, L, synth, torch, dev, peaks, flush, E, stream):
    """The whole decode-side path on the Llama-7B decode shapes: for each of
    [4096x4096], [11008x4096], [4096x11008] (bf16 N(0, 0.02) + 0.1 %
    outliers) nf4q_quantize_dq, nf4q_dequantize (bf16 out) and nf4q_gemv
    (M = 1).  The three weights are independent: each gets two streams
    (quantize + double quant then dequantize; the GEMV once the quantized
    state is ready), captured as one CUDA graph; L2 is flushed before every
    replay, outside the events.  Also the same work one kernel at a time,
    for the per-phase breakdown."""
    sp = stream.cuda_stream
    R = ctypes.byref

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what} failed with status {st}")

    mats = []
    for i in range(3):
        w, x = synth.llama7b_decode(i, device=dev)
        N, K = w.shape
        qw = nq.QuantizedWeight.empty(N, K, device=dev)
        mats.append(dict(w=w, x=x, N=N, K=K, qw=qw, s=qw.struct(),
                         ws=nq.dq_workspace(N * K // 64, dev),
                         out=torch.empty(N, K, dtype=torch.bfloat16, device=dev),
                         y=torch.empty(1, N, dtype=torch.bfloat16, device=dev),
                         bytes=kernel_bytes(N, K)))
    names = ["quantize_dq", "dequantize", "gemv"]

    def launch(m, k, st):
        s_ = m["s"]
        if k == 0:
            check(L.nf4q_quantize_dq(m["w"].data_ptr(), nq.IN_BF16, R(s_), m["ws"].data_ptr(),
                                     m["ws"].numel(), st), "quantize_dq")
        elif k == 1:
            check(L.nf4q_dequantize(R(s_), m["out"].data_ptr(), st), "dequantize")
        else:
            check(L.nf4q_gemv(R(s_), m["x"].data_ptr(), 1, m["y"].data_ptr(), st), "gemv")

    s_a = [torch.cuda.Stream(dev) for _ in mats]
    s_b = [torch.cuda.Stream(dev) for _ in mats]
    ev_go = torch.cuda.Event()
    ev_q = [torch.cuda.Event() for _ in mats]
    ev_end = [torch.cuda.Event() for _ in range(2 * len(mats))]

    def step(main):
        ev_go.record(main)
        for i, m in enumerate(mats):
            s_a[i].wait_event(ev_go)
            s_b[i].wait_event(ev_go)
            launch(m, 0, s_a[i].cuda_stream)
            ev_q[i].record(s_a[i])
            s_b[i].wait_event(ev_q[i])
            launch(m, 2, s_b[i].cuda_stream)
            launch(m, 1, s_a[i].cuda_stream)
        for i in range(len(mats)):
            ev_end[2 * i].record(s_a[i])
            ev_end[2 * i + 1].record(s_b[i])
        for e in ev_end:
            main.wait_event(e)

    for _ in range(3):
        step(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    n = 20
    ts = []
    for _ in range(n):
        flush()
        a, b = E(), E()
        a.record(stream)
        graph.replay()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    step_bytes = sum(m["bytes"][k] for m in mats for k in names)
    # one kernel at a time on one stream: per phase, a CUDA graph of
    # (L2 flush, kernel) for each weight, repeated, against a graph of the
    # flushes alone; device time only, so host pacing cannot leak in
    reps = 10

    def timed_graph(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                body(torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        best = None
        for _ in range(3):
            a, b = E(), E()
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            best = a.elapsed_time(b) if best is None else min(best, a.elapsed_time(b))
        del g
        return best

    def flushes_only(st):
        for _ in mats:
            flush()

    t_flush = timed_graph(flushes_only)
    kern_ms = {}
    for k in range(3):
        def body(st, k=k):
            for m in mats:
                flush()
                launch(m, k, st)
        kern_ms[names[k]] = max(0.0, timed_graph(body) - t_flush) / reps * n
    serial = sum(kern_ms.values())
    breakdown = {k: {"ms_per_step": round(kern_ms[k] / n, 4),
                     "GB/s": round(sum(m["bytes"][k] for m in mats) / (kern_ms[k] / n * 1e-3) / 1e9, 1),
                     "frac_measured_hbm": round(sum(m["bytes"][k] for m in mats)
                                                / (kern_ms[k] / n * 1e-3) / 1e9 / peaks["hbm"], 4),
                     "share": round(kern_ms[k] / serial, 3),
                     "bytes_per_call": sum(m["bytes"][k] for m in mats) // 3}
                 for k in names}
    del graph
    return {"workload": "Llama-7B decode shapes [4096x4096], [11008x4096], [4096x11008], "
                        "bf16 N(0,0.02) + 0.1% outliers, x bf16 N(0,1) M=1: quantize + double "
                        "quant, dequantize and GEMV per weight; one CUDA graph, L2 flushed "
                        "before each replay",
            "ms": round(ms, 4), "GB/s": round(step_bytes / (ms * 1e-3) / 1e9, 1),
            "bytes": step_bytes,
            "serial_breakdown": {"note": f"one kernel at a time, L2 flushed before each (CUDA "
                                         f"graphs of flush + kernel less graphs of the flushes), "
                                         f"{round(serial / n, 4)} ms per step", **breakdown}}


# ------------------------------------------------------------------ oracle (CPU)
def _limit_threads(n=1):
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(n)
    except Exception:
        return None


def _oracle_dequant_gemv_time(states, threads):
    """Seconds the oracle takes to dequantize (from the packed state) and
    multiply (fp64), like the GEMV does from the stored weight."""
    from oracle import nf4_oracle as o
    lim = _limit_threads(threads)
    t0 = time.perf_counter()
    for packed, scales, shape, xb in states:
        w_hat = o.dequantize(packed, scales).reshape(shape)
        o.matmul_ref(xb, w_hat)
    dt = time.perf_counter() - t0
    if lim is not None and hasattr(lim, "unregister"):
        lim.unregister()
    return dt


def _stack_states(items):
    """The oracle's stored state (packed codes, block scales) of stack
    matrices, built in spawned workers (untimed preparation)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(len(items), os.cpu_count() or 1)) as pool:
        return pool.map(_oracle_state_item, items)


def _oracle_state_item(item):
    import numpy as np
    import torch
    import synth
    from oracle import nf4_oracle as o
    layer, mid, rows = item
    w = synth.llama3_8b_matrix(layer, mid, device="cpu")
    x = synth.llama3_8b_x(layer, mid, device="cpu")
    wf = (w if rows is None else w[:rows]).float().numpy()
    packed, absmax = o.quantize(wf)
    q, s2, off = o.double_quant(absmax)
    scales = o.block_scales(q, s2, off)
    return packed, scales, wf.shape, x.contiguous().view(torch.int16).numpy().view(np.uint16)


def cpu_baselines():
    """The oracle timed on the host cores on bounded samples of the GPU
    workloads: the decode token's GEMVs (dequantize from the stored state +
    fp64 GEMV) over layer 0's seven matrices, with one thread and with all
    cores; and the prefill GEMM (fp64) at M = 64 and 256."""
    import numpy as np
    cores = len(os.sched_getaffinity(0))
    items = [(0, mid, None) for mid in range(7)]
    states = _stack_states(items)
    by = sum(kernel_bytes(sh[0], sh[1])["gemv"] for _, _, sh, _ in states)
    dt1 = _oracle_dequant_gemv_time(states, 1)
    dtn = _oracle_dequant_gemv_time(states, cores)
    sample = ("layer 0 of the token (its 7 GEMVs, 218 M weights): the oracle's dequantize "
              "from the stored NF4 state + fp64 GEMV (NumPy); the oracle's own quantization "
              "is prepared untimed")
    out = {"cpu_baseline": {"value": round(by / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                            "kind": "oracle", "seconds": round(dt1, 3), "host_cpus": os.cpu_count(),
                            "affinity": cores, "sample": sample},
           "cpu_baseline_all_cores": {"value": round(by / dtn / 1e9, 4), "unit": "GB/s",
                                      "cores": cores, "kind": "oracle", "seconds": round(dtn, 3),
                                      "sample": sample}}
    del states
    # prefill GEMM: 14336x4096 weight, X [M x 4096]
    import synth
    import torch
    from oracle import nf4_oracle as o
    w_hat = _prefill_w_hat_spawned()
    n_rows, n_cols = w_hat.shape
    pts = []
    for M in (64, 256):
        xb = synth.prefill_x(M, device="cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
        for threads in (1, cores):
            lim = _limit_threads(threads)
            t0 = time.perf_counter()
            o.matmul_ref(xb, w_hat)
            dt = time.perf_counter() - t0
            if lim is not None and hasattr(lim, "unregister"):
                lim.unregister()
            pts.append({"M": M, "cores": threads, "s": round(dt, 3),
                        "TFLOP/s": round(2.0 * M * n_rows * n_cols / dt / 1e12, 5)})
    out["cpu_baseline_gemm"] = {"kind": "oracle", "workload": "prefill 14336x4096 NF4 weight "
                                "(oracle-dequantized, untimed), fp64 X . w_hat^T", "points": pts}
    return out


def _prefill_w_hat(_):
    """The oracle's dequantized prefill weight (untimed preparation)."""
    import synth
    from oracle import nf4_oracle as o
    wf = synth.prefill_weight(device="cpu").float().numpy()
    return o.quantize_full(wf)["w_hat"].reshape(wf.shape)


def _prefill_w_hat_spawned():
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(1) as pool:
        return pool.map(_prefill_w_hat, [0])[0]


def token_bytes_per_step() -> int:
    """Algorithmic bytes of one decode token: per launch the packed codes,
    int8 scale codes, scale2 and offset of each weight, its y, and x once."""
    import synth
    shapes = [(n, k) for _, n, k in synth.LLAMA3_8B_LAYER]
    per_layer = 0
    for _, mids in GROUPS:
        per_layer += sum(nbytes_state(shapes[m][0] * shapes[m][1]) + 2 * shapes[m][0]
                         for m in mids) + 2 * shapes[mids[0]][1]
    return per_layer * synth.LLAMA3_8B_LAYERS


def token_config(world: int) -> dict:
    """The workload both arms report (the reference arm times a bounded
    sample of it, named in its cpu_baseline)."""
    import synth
    return {"workload": WORKLOAD, "M": 1, "bytes_per_step": token_bytes_per_step(),
            "gemv_launches_per_step": len(GROUPS) * synth.LLAMA3_8B_LAYERS,
            "groups": "per layer: q/k/v sharing one x, o, gate/up sharing one x, down; "
                      "each group one nf4q_gemv_multi_ex call with NF4Q_GEMV_WEIGHTS_STATIC "
                      "(weights quantized once, never rewritten)",
            "l2": "not flushed: the 3.61 GB of weights per step exceed L2 (126 MB)",
            "launch": "the launches captured once in a CUDA graph, replayed per step",
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    rank, world, _ = rank_env()
    if rank != 0:
        return
    import numpy as np
    import torch
    import synth
    from oracle import nf4_oracle as o
    lim = _limit_threads(1)
    rows = 256   # per step, so that a run of --steps 1000 ends in a few minutes
    w = synth.llama3_8b_matrix(0, 0, device="cpu")[:rows]
    x = synth.llama3_8b_x(0, 0, device="cpu")
    packed, absmax = o.quantize(w.float().numpy())
    q, s2, off = o.double_quant(absmax)
    scales = o.block_scales(q, s2, off)
    xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    by = kernel_bytes(rows, w.shape[1])["gemv"]

    def one():
        w_hat = o.dequantize(packed, scales).reshape(rows, -1)
        o.matmul_ref(xb, w_hat)

    for _ in range(max(3, args.warmup)):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    tot = time.perf_counter() - t0
    value = by * args.steps / tot / 1e9
    sample = (f"rows 0..{rows - 1} of layer 0's q weight (4096x4096) per step: the oracle's "
              "dequantize from the stored NF4 state + fp64 GEMV (NumPy, one thread)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": token_config(world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)
    if lim is not None and hasattr(lim, "unregister"):
        lim.unregister()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="only the token step and e2e")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
