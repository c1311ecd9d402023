"""LLM.int8() through the C ABI against the oracle: weight and activation
codes, scales and the outlier columns bit for bit; the decomposition matmul
within |y - y_ref| <= 2e-3 * (the same sums over absolute values) + one fp16
ulp."""
import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
import synth
from oracle import llm_int8_oracle as q8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available()
    from dequant_matmul_quantize_b300 import build
    build.build()
    yield
    torch.cuda.synchronize()


def _bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def _check_y(y_gpu, x, wq_np, sw_np, threshold, what=""):
    y_ref, bound, _, _, _ = q8.matmul_ref(_bits16(x), wq_np, sw_np, threshold)
    y = _f32(y_gpu).astype(np.float64)
    err = np.abs(y - y_ref)
    tol = q8.tolerance(y_ref, bound)
    worst = float(np.max(err / tol)) if err.size else 0.0
    assert np.all(err <= tol), f"{what}: worst err/tol = {worst:.3f}"
    return worst


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", [(1, 16), (37, 320), (300, 4096), (5, 8208)])
def test_weight_codes_bit_exact(dtype, shape):
    w = synth.normal_weight(*shape, 0.02, seed=shape[0], dtype=dtype, outlier_frac=1e-3)
    w[min(2, shape[0] - 1)] = 0                           # an all-zero row: scale 0, codes 0
    wq = nq.int8_quantize_weight(w.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref = q8.quantize_rows(_f32(w))
    assert np.array_equal(wq.scale.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(wq.q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("M", [1, 5, 16, 40])
@pytest.mark.parametrize("threshold", [6.0, 0.0, 2.5])
def test_activation_side_bit_exact(M, threshold):
    K = 1024
    x = synth.outlier_activations(M, K, seed=M, outlier_frac=0.01)
    x[0, 7] = 6.0                                         # exactly at the threshold: not an outlier
    w = synth.normal_weight(64, K, 0.02, seed=3, dtype=torch.float16)
    wq = nq.int8_quantize_weight(w.cuda())
    ws = nq.int8_workspace(M, K)
    nq.int8_matmul(wq, x.cuda(), threshold, workspace=ws)
    torch.cuda.synchronize()
    flags, count, lst, sx, xq = nq.int8_workspace_views(ws, M, K)
    xf = _f32(x)
    outl = q8.outlier_columns(xf, threshold)
    xq_ref, sx_ref = q8.quantize_rows(xf, outl)
    assert np.array_equal(flags.cpu().numpy().astype(bool), outl)
    assert count == int(outl.sum())
    assert np.array_equal(lst.cpu().numpy(), np.nonzero(outl)[0])
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(_f32(xq).astype(np.int32), xq_ref.astype(np.int32))


@pytest.mark.parametrize("M,N,K", [(1, 64, 128), (3, 100, 320), (8, 37, 4160), (9, 256, 1024),
                                   (16, 130, 2048), (40, 96, 512), (1, 4096, 4096)])
def test_matmul_small(M, N, K):
    x = synth.outlier_activations(M, K, seed=N + K, outlier_frac=0.005)
    w = synth.normal_weight(N, K, 0.02, seed=N, dtype=torch.float16, outlier_frac=1e-3)
    wq = nq.int8_quantize_weight(w.cuda())
    y = nq.int8_matmul(wq, x.cuda())
    torch.cuda.synchronize()
    _check_y(y, x, wq.q.cpu().numpy(), wq.scale.cpu().numpy(), 6.0, f"{M}x{N}x{K}")


@pytest.mark.parametrize("threshold", [0.0, 1e-3, 6.0, float("nan")])
def test_matmul_thresholds(threshold):
    """No decomposition (0, NaN), every nonzero column an outlier (1e-3), and
    the default."""
    M, N, K = 6, 80, 640
    x = synth.outlier_activations(M, K, seed=9, outlier_frac=0.02)
    w = synth.normal_weight(N, K, 0.02, seed=10, dtype=torch.float16)
    wq = nq.int8_quantize_weight(w.cuda())
    y = nq.int8_matmul(wq, x.cuda(), threshold)
    torch.cuda.synchronize()
    t = 0.0 if threshold != threshold else threshold
    _check_y(y, x, wq.q.cpu().numpy(), wq.scale.cpu().numpy(), t, f"threshold {threshold}")


def test_matmul_zero_rows_and_edges():
    K, N = 256, 48
    w = synth.normal_weight(N, K, 0.02, seed=11, dtype=torch.float16)
    wq = nq.int8_quantize_weight(w.cuda())
    x = synth.outlier_activations(4, K, seed=12, outlier_frac=0.0)
    x[1] = 0                                              # sx = 0: codes 0, y = 0
    y = nq.int8_matmul(wq, x.cuda())
    torch.cuda.synchronize()
    assert (y[1] == 0).all()
    _check_y(y, x, wq.q.cpu().numpy(), wq.scale.cpu().numpy(), 6.0, "zero row")
    # M = 0: nothing launched
    out = torch.empty(0, N, dtype=torch.float16, device="cuda")
    nq.int8_matmul(wq, torch.empty(0, K, dtype=torch.float16, device="cuda"), out=out)
    # a workspace that is too small is refused
    import ctypes
    L, s = nq.lib(), wq.struct()
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    xs = x.cuda()
    assert L.nf4q_int8_matmul(ctypes.byref(s), xs.data_ptr(), 4, 6.0, y.data_ptr(),
                              ws.data_ptr(), 64, torch.cuda.current_stream().cuda_stream) == 4
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [1, 16])
def test_mlp70b_full_size_sampled(M):
    """The fp16 28672 x 8192 weight: whole weight quantized on the GPU; codes
    and scales of sampled rows, and all outputs of those rows, against the
    oracle."""
    w = synth.int8_mlp70b_weight(device="cuda")
    x = synth.int8_mlp70b_x(M, device="cuda")
    wq = nq.int8_quantize_weight(w)
    y = nq.int8_matmul(wq, x)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, w.shape[0] - 1],
                                     np.random.default_rng(M).integers(0, w.shape[0], 30)]))
    idx = torch.from_numpy(rows).cuda()
    q_ref, s_ref = q8.quantize_rows(_f32(w[idx]))
    assert np.array_equal(wq.q[idx].cpu().numpy(), q_ref)
    assert np.array_equal(wq.scale[idx].cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    _check_y(y[:, idx], x.cpu(), q_ref, s_ref, 6.0, f"70B MLP M={M}")
