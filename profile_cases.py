"""Single workloads for profiling one kernel at a time (ncu / nsight).

    python profile_cases.py CASE [CASE ...]

Each case builds its seeded synthetic input, runs the library call twice
(a warm-up and the one to capture) and synchronizes.  Cases:

    quant11008   nf4q_quantize_dq then nf4q_dequantize, 11008x4096 decode weight
    gemv70b      nf4q_gemv M=1 on the 28672x8192 weight (NF4)
    gemv70b_exact  nf4q_gemv_exact M=1 on the same weight
    token        one Llama-3-8B decode token twice over the 224-weight stack:
                 per layer the groups (q, k, v), (o), (gate, up), (down), each
                 one nf4q_gemv_multi_ex call with NF4Q_GEMV_WEIGHTS_STATIC -
                 128 launches per token, as the benchmark step issues them
    layer        the same four launches for layer 0 only, twice
    gateup       the (gate, up) launch of layer 0, twice
    gemv4096     nf4q_gemv M=1 on the 4096x4096 decode weight
    gemv4096_exact  nf4q_gemv_exact M=1 on the same weight
    gemv11008    nf4q_gemv M=1 on the 11008x4096 decode weight
    gemv70b_m16  nf4q_gemv M=16 on the 28672x8192 weight (NF4)
    gemm2048     nf4q_gemm M=2048 on the 14336x4096 prefill weight
    gemm64       nf4q_gemm M=64 on the 14336x4096 prefill weight
    dx2048       nf4q_matmul_dx M=2048 on the 14336x4096 prefill weight
    dx256        nf4q_matmul_dx M=256 on the same weight (128-row tiles, the
                 contraction split over a 2-CTA cluster)
    int8_m1      nf4q_int8_quantize_weight, then nf4q_int8_matmul M=1 and
                 M=16, on the fp16 28672x8192 weight (LLM.int8())

Kernel launches per case are listed so a capture can be aimed with ncu's
-k / -s / -c options.
"""
from __future__ import annotations

import ctypes
import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _run(case: str, torch, nq, synth) -> None:
    L = nq.lib()
    R = ctypes.byref
    dev = torch.device("cuda", 0)
    sp = torch.cuda.current_stream().cuda_stream

    def ok(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: status {st}")

    if case in ("token", "layer", "gateup"):
        groups = ((0, 1, 2), (3,), (4, 5), (6,)) if case != "gateup" else ((4, 5),)
        layers = synth.LLAMA3_8B_LAYERS if case == "token" else 1
        launches = []
        for layer in range(layers):
            for mids in groups:
                qws = [nq.quantize(synth.llama3_8b_matrix(layer, mid, device=dev)) for mid in mids]
                x = synth.llama3_8b_x(layer, mids[0], device=dev)
                ys = [torch.empty(1, q.rows, dtype=torch.bfloat16, device=dev) for q in qws]
                launches.append((qws, x, ys))
        torch.cuda.synchronize()
        for _ in range(2):
            for qws, x, ys in launches:
                nq.gemv_multi(qws, x, outs=ys, static_weights=True)
    elif case == "quant11008":
        w, _ = synth.llama7b_decode(1, device=dev)
        N, K = w.shape
        qw = nq.QuantizedWeight.empty(N, K, device=dev)
        s = qw.struct()
        ws = nq.dq_workspace(N * K // 64, dev)
        out = torch.empty_like(w)
        for _ in range(2):
            ok(L.nf4q_quantize_dq(w.data_ptr(), nq.IN_BF16, R(s), ws.data_ptr(), ws.numel(), sp),
               "quantize_dq")
            ok(L.nf4q_dequantize(R(s), out.data_ptr(), sp), "dequantize")
    elif case in ("gemv70b", "gemv70b_m16", "gemv70b_exact"):
        M = 16 if case.endswith("m16") else 1
        fn = L.nf4q_gemv_exact if case.endswith("exact") else L.nf4q_gemv
        qw = nq.quantize(synth.mlp70b_weight(device=dev))
        s = qw.struct()
        x = synth.mlp70b_x(M, device=dev)
        y = torch.empty(M, qw.rows, dtype=torch.bfloat16, device=dev)
        for _ in range(2):
            ok(fn(R(s), x.data_ptr(), M, y.data_ptr(), sp), "gemv")
    elif case in ("gemv4096", "gemv11008", "gemv4096_exact"):
        w, x = synth.llama7b_decode(1 if case == "gemv11008" else 0, device=dev)
        fn = L.nf4q_gemv_exact if case.endswith("exact") else L.nf4q_gemv
        qw = nq.quantize(w)
        s = qw.struct()
        y = torch.empty(1, qw.rows, dtype=torch.bfloat16, device=dev)
        for _ in range(2):
            ok(fn(R(s), x.data_ptr(), 1, y.data_ptr(), sp), "gemv")
    elif case in ("gemm2048", "gemm64"):
        M = 2048 if case == "gemm2048" else 64
        qw = nq.quantize(synth.prefill_weight(device=dev))
        s = qw.struct()
        x = synth.prefill_x(M, device=dev)
        y = torch.empty(M, qw.rows, dtype=torch.bfloat16, device=dev)
        for _ in range(2):
            ok(L.nf4q_gemm(R(s), x.data_ptr(), M, y.data_ptr(), sp), "gemm")
    elif case in ("dx2048", "dx256"):
        Md = 2048 if case == "dx2048" else 256
        qw = nq.quantize(synth.prefill_weight(device=dev))
        s = qw.struct()
        N, K = qw.rows, qw.cols
        dy = synth.activations(Md, N, seed=Md + N, device=dev)
        dx = torch.empty(Md, K, dtype=torch.bfloat16, device=dev)
        for _ in range(2):
            ok(L.nf4q_matmul_dx(R(s), dy.data_ptr(), N, Md, dx.data_ptr(), sp), "matmul_dx")
    elif case == "int8_m1":
        w = synth.int8_mlp70b_weight(device=dev)
        for _ in range(2):
            wq = nq.int8_quantize_weight(w)
        for M in (1, 16):
            x = synth.int8_mlp70b_x(M, device=dev)
            ws = nq.int8_workspace(M, wq.cols, dev)
            y = torch.empty(M, wq.rows, dtype=torch.float16, device=dev)
            for _ in range(2):
                nq.int8_matmul(wq, x, workspace=ws, out=y)
    else:
        raise SystemExit(f"unknown case {case!r}; see the module docstring")
    torch.cuda.synchronize()


def main(argv) -> None:
    import torch
    import dequant_matmul_quantize_b300 as nq
    import synth
    if not argv:
        raise SystemExit(__doc__)
    for case in argv:
        _run(case, torch, nq, synth)
    print("ok")


if __name__ == "__main__":
    main(sys.argv[1:])
