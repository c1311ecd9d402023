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
