"""fp16 compute dtype (tutorial sec. 四, bnb_4bit_compute_dtype = float16)
through the C ABI, against the oracle: fp16 weights into nf4q_quantize,
dequantization to fp16 bit for bit, and the GEMV / GEMM with fp16 x and y
within the matmul tolerance."""
import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
import synth
from oracle import nf4_oracle as o
from tests._util import (CODE_ID, as_f32, assert_bits_equal, bf16_bits, check_matmul,
                         gpu_state, oracle_state)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available()
    from dequant_matmul_quantize_b300 import build
    build.build()
    nq.device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert nq.device_error() == 0


def _f16_check(w: torch.Tensor, code: str, double_quant=True, what=""):
    """Quantize for the fp16 compute dtype; the stored state is the same as
    for bf16 and w_hat is the fp16 rounding of code * s."""
    qw = nq.quantize(w.cuda(), code, double_quant, compute_dtype="f16")
    out = nq.dequantize(qw)
    torch.cuda.synchronize()
    assert out.dtype == torch.float16
    g = gpu_state(qw)
    ref = oracle_state(as_f32(w).reshape(-1), code, double_quant)
    for k in ("packed", "absmax") + (("absmax_q", "scale2") if double_quant else ()):
        assert_bits_equal(g[k], ref[k], f"{what} {k}")
    w_hat = o.dequantize(ref["packed"], ref["scales"], CODE_ID[code], dtype=o.DT_F16)
    assert_bits_equal(bf16_bits(out).reshape(-1), w_hat, what + " w_hat f16")
    return qw, w_hat.reshape(w.shape)


@pytest.mark.parametrize("code", ["nf4", "fp4"])
@pytest.mark.parametrize("shape", [(3, 64), (37, 320), (129, 4160), (300, 2048)])
def test_f16_dequantize_bit_exact(code, shape):
    w = synth.normal_weight(*shape, 0.02, seed=shape[0], outlier_frac=2e-3)
    _f16_check(w, code, True, f"{code} {shape}")
    _f16_check(w, code, False, f"{code} {shape} no-dq")


def test_f16_weights_into_quantize():
    """fp16 input widens exactly; codes and scales equal the oracle's on the
    widened values, with and without the fused double quant."""
    w = synth.normal_weight(96, 1024, 0.05, seed=7).to(torch.float16)
    for dq in (True, False):
        qw = nq.quantize(w.cuda(), "nf4", dq)
        torch.cuda.synchronize()
        g = gpu_state(qw)
        ref = oracle_state(as_f32(w).reshape(-1), "nf4", dq)
        for k in ("packed", "absmax") + (("absmax_q", "scale2", "offset") if dq else ()):
            a = np.atleast_1d(g[k])
            assert_bits_equal(a, np.atleast_1d(ref[k]), f"f16 input dq={dq} {k}")


def test_f16_dequantize_overflows_to_infinity():
    """Scales large enough that code * s exceeds fp16's range give +-inf, as
    IEEE rounding to fp16 does (the oracle rounds the same way)."""
    rng = np.random.default_rng(4)
    w = (rng.uniform(-1, 1, (4, 256)) * 1e5).astype(np.float32)
    _, w_hat = _f16_check(torch.from_numpy(w), "nf4", False, "overflow")
    assert np.isinf(o.f16_bits_to_f32(w_hat)).any()


@pytest.mark.parametrize("code", ["nf4", "fp4"])
@pytest.mark.parametrize("M", [1, 5, 8, 16])
def test_f16_gemv(code, M):
    w = synth.normal_weight(200, 1536, 0.02, seed=M + 40, outlier_frac=1e-3)
    qw, w_hat = _f16_check(w, code, True, "gemv")
    x = synth.activations(M, 1536, seed=M).to(torch.float16)
    y = nq.gemv(qw, x.cuda())
    torch.cuda.synchronize()
    assert y.dtype == torch.float16
    check_matmul(bf16_bits(y), bf16_bits(x), w_hat, f"f16 gemv {code} M={M}", o.DT_F16)


@pytest.mark.parametrize("code", ["nf4", "fp4"])
@pytest.mark.parametrize("M", [64, 300])
def test_f16_gemm(code, M):
    w = synth.normal_weight(320, 1024, 0.02, seed=M + 50)
    qw, w_hat = _f16_check(w, code, True, "gemm")
    x = synth.activations(M, 1024, seed=M + 1).to(torch.float16)
    y = nq.gemm(qw, x.cuda())
    torch.cuda.synchronize()
    assert y.dtype == torch.float16
    check_matmul(bf16_bits(y), bf16_bits(x), w_hat, f"f16 gemm {code} M={M}", o.DT_F16)
    assert torch.equal(nq.matmul(qw, x.cuda()), y)
