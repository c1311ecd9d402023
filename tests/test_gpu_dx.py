"""Parity of the input-gradient kernel dX = dY . w_hat (nf4q_matmul_dx,
tcgen05, through the C ABI) with the fp64 oracle: |dX - dX_ref| <= 2e-3 *
sum_n |dY_n w_hat_nk| + one ulp of the compute dtype, per output element."""
import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
import synth
from oracle import nf4_oracle as o
from tests._util import CODE_ID, as_f32, bf16_bits, oracle_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available()
    from dequant_matmul_quantize_b300 import build
    build.build()
    nq.device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert nq.device_error() == 0, "a dX pipeline wait timed out"


def _what(w, code="nf4", dq=True, dtype=o.DT_BF16):
    ref = oracle_state(as_f32(w).reshape(-1), code, dq)
    return o.dequantize(ref["packed"], ref["scales"], CODE_ID[code], dtype=dtype).reshape(w.shape)


def check_dx(dx_bits, dy_bits, what_bits, what="", dtype=o.DT_BF16):
    ref, bound = o.matmul_dx_ref(dy_bits, what_bits, dtype)
    got = o.from_bits(dx_bits, dtype).astype(np.float64)
    err = np.abs(got - ref)
    tol = o.matmul_tolerance(ref, bound, dtype)
    worst = float(np.max(err / tol)) if err.size else 0.0
    assert np.all(err <= tol), f"{what}: worst err/tol = {worst:.3f}"
    return worst


# (M, N, K): N = the weight's rows (the contraction), K = its columns (dX's
# width).  Ragged N and K tails, several M tiles, and shapes that select
# each tile width (128 for the small ones, 256 for 2048 x 256 x 4096, 192
# for 3000 x 136 x 4096).
SHAPES = [(1, 64, 64), (5, 200, 320), (64, 256, 256), (300, 1000, 1024), (129, 136, 4160),
          (513, 512, 512), (2048, 256, 4096), (3000, 136, 4096),
          # the contraction split over a cluster: S = 4 over 65 stages (ragged
          # last stage) and over 37 stages, one-accumulator tiles
          (200, 4160, 320), (77, 2368, 960),
          # 256-row tiles (two accumulators) split over a 2-CTA cluster: their
          # 128-row tiles would fill one wave with no room for a split
          # (148 SMs); ragged M and a ragged last stage
          (500, 1024, 4096), (512, 4160, 4096)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_dx_small(M, N, K):
    w = synth.normal_weight(N, K, 0.02, seed=N + K, outlier_frac=1e-3)
    dy = synth.activations(M, N, seed=M + 7)
    qw = nq.quantize(w.cuda())
    dx = nq.matmul_dx(qw, dy.cuda())
    torch.cuda.synchronize()
    assert dx.shape == (M, K)
    check_dx(bf16_bits(dx), bf16_bits(dy), _what(w), f"dx {M}x{N}x{K}")


@pytest.mark.parametrize("code", ["nf4", "fp4"])
@pytest.mark.parametrize("dq", [True, False])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_dx_codes_dq_and_dtypes(code, dq, dt):
    w = synth.normal_weight(384, 640, 0.015, seed=41)
    dtype = o.DT_BF16 if dt == "bf16" else o.DT_F16
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    dy = synth.activations(260, 384, seed=42).to(tdt)
    qw = nq.quantize(w.cuda(), code, dq, compute_dtype=dt)
    dx = nq.matmul_dx(qw, dy.cuda())
    torch.cuda.synchronize()
    assert dx.dtype == tdt
    check_dx(bf16_bits(dx), bf16_bits(dy), _what(w, code, dq, dtype), f"{code} dq={dq} {dt}",
             dtype)


def test_dx_one_hot_rows_are_weight_rows():
    """A one-hot row of dY picks one row of w_hat: exact, for every row n."""
    N, K = 192, 512
    w = synth.normal_weight(N, K, 0.02, seed=43)
    qw = nq.quantize(w.cuda())
    what = _what(w)
    dy = torch.zeros(N, N, dtype=torch.bfloat16)
    perm = np.random.default_rng(44).permutation(N)
    for m in range(N):
        dy[m, perm[m]] = 1.0
    dx = bf16_bits(nq.matmul_dx(qw, dy.cuda()))
    for m in range(N):
        assert np.array_equal(dx[m], what[perm[m]]), m


def test_dx_row_pitch_reads_only_the_rows():
    """dY as a column slice of a wider tensor (row pitch 104 > rows = 100):
    the padding holds NaN and must not be read."""
    N, K, M = 100, 256, 70
    w = synth.normal_weight(N, K, 0.02, seed=45)
    qw = nq.quantize(w.cuda())
    dy = synth.activations(M, N, seed=46)
    wide = torch.full((M, 104), float("nan"), dtype=torch.bfloat16)
    wide[:, :N] = dy
    wide = wide.cuda()
    dx = nq.matmul_dx(qw, wide[:, :N])
    torch.cuda.synchronize()
    assert torch.isfinite(dx.float()).all()
    check_dx(bf16_bits(dx), bf16_bits(dy), _what(w), "row pitch 104")


def test_dx_agrees_with_dequantize_then_cublas():
    w = synth.normal_weight(512, 1024, 0.02, seed=47)
    qw = nq.quantize(w.cuda())
    dy = synth.activations(256, 512, seed=48).cuda()
    what = _what(w)
    dx = nq.matmul_dx(qw, dy)
    ref_torch = dy @ nq.dequantize(qw)
    torch.cuda.synchronize()
    check_dx(bf16_bits(dx), bf16_bits(dy), what, "kernel")
    check_dx(bf16_bits(ref_torch), bf16_bits(dy), what, "cublas")


def test_dx_edge_cases():
    w = synth.normal_weight(64, 128, 0.02, seed=49)
    qw = nq.quantize(w.cuda())
    # M = 0: nothing launched
    out = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    nq.matmul_dx(qw, torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"), out=out)
    import ctypes
    L, s = nq.lib(), qw.struct()
    stream = torch.cuda.current_stream().cuda_stream
    dy = synth.activations(3, 64, seed=50).cuda()
    dx = torch.empty(3, 128, dtype=torch.bfloat16, device="cuda")
    # row pitch below rows or not a multiple of 8: invalid argument
    assert L.nf4q_matmul_dx(ctypes.byref(s), dy.data_ptr(), 60, 3, dx.data_ptr(), stream) == 1
    assert L.nf4q_matmul_dx(ctypes.byref(s), dy.data_ptr(), 65, 3, dx.data_ptr(), stream) == 1
    # misaligned dX: alignment error, nothing launched
    assert L.nf4q_matmul_dx(ctypes.byref(s), dy.data_ptr(), 64, 3, dx.data_ptr() + 2,
                            stream) == 2
    # rows = 0: dX is all zeros
    q0 = nq.QuantizedWeight.empty(0, 128, device="cuda")
    dx0 = torch.full((3, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    s0 = q0.struct()
    assert L.nf4q_matmul_dx(ctypes.byref(s0), dy.data_ptr(), 64, 3, dx0.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    assert (dx0 == 0).all()


def _columns_of_what(w_gpu, cols_blocks):
    """w_hat[:, 64b .. 64b+63] for the given block columns b of a full-size
    weight: codes from the oracle on those blocks, scales from the double
    quantization of every absmax of W."""
    N, K = w_gpu.shape
    absmax = o.absmax_blocks(as_f32(w_gpu).reshape(-1))
    q, s2, off = o.double_quant(absmax)
    scales = o.block_scales(q, s2, off).reshape(N, K // 64)
    out = []
    for b in cols_blocks:
        part = as_f32(w_gpu[:, 64 * b:64 * b + 64]).reshape(-1)
        packed, _ = o.quantize(part)
        out.append(o.dequantize(packed, scales[:, b].copy()).reshape(N, 64))
    return np.concatenate(out, axis=1)


@pytest.mark.parametrize("which,M", [("prefill", 2048), ("prefill", 256), ("down", 512)])
def test_dx_full_size_sampled(which, M):
    """Full-size weights (14336 x 4096 prefill; the 4096 x 11008 Llama-7B
    down projection): every row of dX on sampled 64-column blocks, each
    recomputed by the oracle from W."""
    if which == "prefill":
        w = synth.prefill_weight(device="cuda")
    else:
        w, _ = synth.llama7b_decode(2, device="cuda")
    N, K = w.shape
    dy = synth.activations(M, N, seed=M + N, device="cuda")
    qw = nq.quantize(w)
    dx = nq.matmul_dx(qw, dy)
    torch.cuda.synchronize()
    blocks = sorted(set([0, K // 64 - 1] + list(np.random.default_rng(M).integers(0, K // 64, 3))))
    what = _columns_of_what(w, blocks)
    idx = torch.tensor([64 * b + j for b in blocks for j in range(64)], device="cuda")
    check_dx(bf16_bits(dx[:, idx]), bf16_bits(dy), what, f"{which} M={M}")
