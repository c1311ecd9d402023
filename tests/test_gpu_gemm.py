"""Parity of the tcgen05 NF4 GEMM (through the C ABI) with the fp64 oracle:
|y - y_ref| <= 2e-3 * sum|x w_hat| + 1 bf16 ulp, per output element."""
import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
import synth
from oracle import nf4_oracle as o
from tests._util import CODE_ID, as_f32, bf16_bits, check_matmul, oracle_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available()
    from dequant_matmul_quantize_b300 import build
    build.build()
    nq.device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert nq.device_error() == 0, "a GEMM pipeline wait timed out"


def _oracle_what(w, code):
    ref = oracle_state(as_f32(w).reshape(-1), code, True)
    return o.dequantize(ref["packed"], ref["scales"], CODE_ID[code]).reshape(w.shape)


@pytest.mark.parametrize("M,N,K", [
    (1, 256, 64), (64, 256, 256), (128, 512, 512), (200, 300, 320), (129, 257, 192),
    (256, 1000, 1024), (383, 768, 2048), (512, 256, 4096),
    # one-accumulator CTAs (M <= 128) with ragged N and K
    (100, 300, 320), (128, 200, 4160), (1, 129, 64), (77, 1000, 192),
    # K split over a cluster: S = 4 with k ranges not aligned to 16 k-steps
    # (37 k-steps), S = 2 (17 k-steps), S = 4 on a ragged 130-row weight
    (33, 700, 2368), (128, 1000, 1088), (5, 130, 4096),
    # narrower W tiles for M <= 128 (one wave): BN = 80, 112, 208, each with
    # a ragged last tile and a partial 32-column chunk in the epilogue
    (33, 11008, 256), (7, 14376, 128), (100, 28600, 192)])
def test_gemm_small(M, N, K):
    w = synth.normal_weight(N, K, 0.02, seed=N + K, outlier_frac=1e-3)
    x = synth.activations(M, K, seed=M)
    qw = nq.quantize(w.cuda())
    y = nq.gemm(qw, x.cuda())
    torch.cuda.synchronize()
    check_matmul(bf16_bits(y), bf16_bits(x), _oracle_what(w, "nf4"), f"gemm {M}x{N}x{K}")


def test_gemm_fp4_and_no_dq():
    w = synth.normal_weight(384, 512, 0.015, seed=4)
    x = synth.activations(160, 512, seed=5)
    for code in ("nf4", "fp4"):
        for dq in (True, False):
            qw = nq.quantize(w.cuda(), code, dq)
            y = nq.gemm(qw, x.cuda())
            ref = oracle_state(as_f32(w).reshape(-1), code, dq)
            what = o.dequantize(ref["packed"], ref["scales"], CODE_ID[code]).reshape(w.shape)
            check_matmul(bf16_bits(y), bf16_bits(x), what, f"{code} dq={dq}")


@pytest.mark.parametrize("code,dq,dt", [("nf4", True, "f16"), ("fp4", True, "bf16"),
                                        ("nf4", False, "bf16"), ("fp4", False, "f16")])
def test_gemm_split_k_configs(code, dq, dt):
    """Split K (2 tiles, 32 k-steps: S = 4) for the other codes, without
    double quantization and with fp16; two calls give identical bits."""
    w = synth.normal_weight(200, 2048, 0.02, seed=21)
    x = synth.activations(40, 2048, seed=22)
    if dt == "f16":
        x = x.to(torch.float16)
    qw = nq.quantize(w.cuda(), code, dq, compute_dtype=dt)
    y1 = nq.gemm(qw, x.cuda())
    y2 = nq.gemm(qw, x.cuda())
    assert torch.equal(y1, y2)
    ref = oracle_state(as_f32(w).reshape(-1), code, dq)
    dt_id = o.DT_F16 if dt == "f16" else o.DT_BF16
    what = o.dequantize(ref["packed"], ref["scales"], CODE_ID[code], dtype=dt_id).reshape(w.shape)
    if dt == "f16":
        check_matmul(y1.cpu().view(torch.int16).numpy().view(np.uint16),
                     x.view(torch.int16).numpy().view(np.uint16), what, f"split {code}", o.DT_F16)
    else:
        check_matmul(bf16_bits(y1), bf16_bits(x), what, f"split {code} dq={dq}")


@pytest.mark.parametrize("code,dq,dt", [("fp4", True, "bf16"), ("nf4", False, "f16")])
def test_gemm_narrow_tiles_configs(code, dq, dt):
    """One-wave narrow W tiles (BN = 80 for 11008 rows) with FP4, without
    double quantization and with fp16; and 128-row tiles at M = 200."""
    w = synth.normal_weight(11008, 128, 0.02, seed=23)
    qw = nq.quantize(w.cuda(), code, dq, compute_dtype=dt)
    ref = oracle_state(as_f32(w).reshape(-1), code, dq)
    dt_id = o.DT_F16 if dt == "f16" else o.DT_BF16
    what = o.dequantize(ref["packed"], ref["scales"], CODE_ID[code], dtype=dt_id).reshape(w.shape)
    for M in (9, 200):
        x = synth.activations(M, 128, seed=24 + M)
        if dt == "f16":
            x = x.to(torch.float16)
        y = nq.gemm(qw, x.cuda())
        if dt == "f16":
            check_matmul(y.cpu().view(torch.int16).numpy().view(np.uint16),
                         x.view(torch.int16).numpy().view(np.uint16), what, f"{code} M={M}",
                         o.DT_F16)
        else:
            check_matmul(bf16_bits(y), bf16_bits(x), what, f"{code} dq={dq} M={M}")


def test_gemm_matches_gemv_and_cublas():
    w = synth.normal_weight(512, 1024, 0.02, seed=8)
    qw = nq.quantize(w.cuda())
    what = _oracle_what(w, "nf4")
    for M in (1, 7, 16):
        x = synth.activations(M, 1024, seed=9 + M).cuda()
        y_gemm = nq.gemm(qw, x)
        y_gemv = nq.gemv(qw, x)
        check_matmul(bf16_bits(y_gemm), bf16_bits(x), what, "gemm small M")
        check_matmul(bf16_bits(y_gemv), bf16_bits(x), what, "gemv")
    x = synth.activations(256, 1024, seed=3).cuda()
    y_cublas = torch.matmul(x, nq.dequantize(qw).T)
    check_matmul(bf16_bits(y_cublas), bf16_bits(x), what, "cublas")
    check_matmul(bf16_bits(nq.matmul(qw, x)), bf16_bits(x), what, "matmul dispatch")


def test_matmul_dispatch():
    """nf4q_matmul: the GEMV up to M = 16, except M = 9..16 on weights of
    20000 rows or more, which take the GEMM (bitwise the same call)."""
    for rows, K in ((300, 256), (20000, 128)):
        qw = nq.quantize(synth.normal_weight(rows, K, 0.02, seed=rows).cuda())
        for M in (1, 8, 9, 16, 17):
            x = synth.activations(M, K, seed=M).cuda()
            gemm = M > 16 or (M > 8 and rows >= 20000)
            want = nq.gemm(qw, x) if gemm else nq.gemv(qw, x)
            assert torch.equal(nq.matmul(qw, x), want), (rows, M)


def test_gemm_one_hot_rows_exact():
    w = synth.normal_weight(256, 256, 0.02, seed=12)
    qw = nq.quantize(w.cuda())
    what = _oracle_what(w, "nf4")
    x = torch.zeros(128, 256, dtype=torch.bfloat16)
    for m in range(128):
        x[m, (m * 37) % 256] = 1.0
    y = bf16_bits(nq.gemm(qw, x.cuda()))
    for m in range(128):
        assert np.array_equal(y[m], what[:, (m * 37) % 256])


@pytest.mark.parametrize("M", [64, 256, 512, 2048])
def test_prefill_full_size_sampled(M):
    """The 14336 x 4096 prefill weight at full size; every output row, on 40
    sampled output columns (each recomputed by the oracle from W)."""
    w = synth.prefill_weight(device="cuda")
    x = synth.prefill_x(M, device="cuda")
    qw = nq.quantize(w)
    y = nq.gemm(qw, x)
    torch.cuda.synchronize()
    N, K = w.shape
    cols = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(M).integers(0, N, 40)]))
    w_rows = as_f32(w[torch.from_numpy(cols).cuda()])
    # scales need the whole tensor's mean: recompute the state from all of W
    absmax = o.absmax_blocks(as_f32(w).reshape(-1))
    q, s2, off = o.double_quant(absmax)
    scales = o.block_scales(q, s2, off).reshape(N, K // 64)
    what = np.stack([o.dequantize(o.quantize(w_rows[i])[0], scales[c]) for i, c in enumerate(cols)])
    y_cols = bf16_bits(y[:, torch.from_numpy(cols).cuda()])
    check_matmul(y_cols, bf16_bits(x), what, f"prefill M={M}")
