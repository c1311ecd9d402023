"""Helpers shared by the GPU parity tests: move tensors to NumPy, run the
oracle on the same inputs, compare."""
import numpy as np
import torch

from oracle import nf4_oracle as o

CODE_ID = {"nf4": o.CODE_NF4, "fp4": o.CODE_FP4}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def as_f32(t: torch.Tensor) -> np.ndarray:
    """A CPU float32 copy of an fp32 or bf16 tensor (widening is exact)."""
    return t.detach().float().cpu().numpy()


def gpu_state(qw):
    out = dict(packed=qw.packed.cpu().numpy(), absmax=qw.absmax.cpu().numpy())
    if qw.double_quant:
        out.update(absmax_q=qw.absmax_q.cpu().numpy(), scale2=qw.scale2.cpu().numpy(),
                   offset=np.float32(qw.offset.cpu().numpy()[0]))
    return out


def oracle_state(w_f32: np.ndarray, code: str, double_quant: bool = True):
    c = CODE_ID[code]
    packed, absmax = o.quantize(w_f32, c)
    st = dict(packed=packed, absmax=absmax)
    if double_quant:
        q, s2, off = o.double_quant(absmax)
        st.update(absmax_q=q, scale2=s2, offset=off)
        scales = o.block_scales(q, s2, off)
    else:
        scales = absmax
    st["scales"] = scales
    return st


def assert_bits_equal(a, b, what):
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    if a.dtype.kind == "f":
        a = a.view(np.uint32 if a.itemsize == 4 else np.uint16)
        b = b.view(np.uint32 if b.itemsize == 4 else np.uint16)
    bad = np.nonzero(a != b)[0] if a.ndim == 1 else np.argwhere(a != b)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}"


def check_matmul(y_gpu_bits: np.ndarray, x_bits: np.ndarray, what_bits: np.ndarray, what="",
                 dtype: int = o.DT_BF16):
    """|y - y_ref| <= 2e-3 * sum|x w_hat| + one ulp of y_ref in the compute
    dtype, per output."""
    y_ref, bound = o.matmul_ref(x_bits, what_bits, dtype)
    y = o.from_bits(y_gpu_bits, dtype).astype(np.float64)
    err = np.abs(y - y_ref)
    tol = o.matmul_tolerance(y_ref, bound, dtype)
    worst = np.max(err / tol) if err.size else 0.0
    assert np.all(err <= tol), f"{what}: worst err/tol = {worst:.3f}"
    return worst


def full_check(w, code: str, double_quant=True, what=""):
    """Quantize on the GPU and in the oracle; compare every byte of the
    stored state and of the dequantized weights.  Returns the GPU weight and
    the ORACLE's w_hat (bit patterns, shaped like w)."""
    import dequant_matmul_quantize_b300 as nq
    qw = nq.quantize(w.cuda(), code, double_quant)
    what_gpu = nq.dequantize(qw)
    torch.cuda.synchronize()
    g = gpu_state(qw)
    ref = oracle_state(as_f32(w).reshape(-1), code, double_quant)
    assert_bits_equal(g["absmax"], ref["absmax"], what + " absmax")
    assert_bits_equal(g["packed"], ref["packed"], what + " packed")
    if double_quant:
        assert_bits_equal(np.array([g["offset"]]), np.array([ref["offset"]]), what + " offset")
        assert_bits_equal(g["scale2"], ref["scale2"], what + " scale2")
        assert_bits_equal(g["absmax_q"], ref["absmax_q"], what + " absmax_q")
    w_hat = o.dequantize(ref["packed"], ref["scales"], CODE_ID[code])
    assert_bits_equal(bf16_bits(what_gpu).reshape(-1), w_hat, what + " w_hat")
    return qw, w_hat.reshape(w.shape)
