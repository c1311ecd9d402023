"""CPU oracle for LLM.int8(): vector-wise int8 quantization and the
mixed-precision decomposition matmul.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) imports, links or runs this file.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may use it.  It shares no code with the CUDA path.

Sources (web pages about the bitsandbytes library; cited by page title and
section):

* "bitsandbytes tutorial" (mlqm.cn/news/394670), section 3.1: LLM.int8()
  splits a matmul in three steps - the few outlier feature dimensions of the
  activations are computed exactly in FP16, the remaining dimensions are
  quantized to INT8 and computed there, and the two results are added;
  outlier dimensions are usually under 1 %.  Section 四 (key settings):
  ``llm_int8_threshold``, default 6.0, decides how large a value must be to
  count as an outlier.
* "bitsandbytes introduction" (modelers.csdn.net), core techniques item 2:
  weights and activations are quantized to 8 bits with a vector-wise
  strategy; the few outlier feature vectors keep 16-bit precision.
* "bitsandbytes: quantifier un modèle PyTorch sans quitter PyTorch"
  (hysenlabs.com): vector-wise quantization handles most features in 8 bits
  and isolates the outliers in a 16-bit matrix multiplication.

READINGS of what the pages leave open (each also listed in the design notes):

* outlier features: the columns k of the activations X [M x K] in which some
  row has |X[m, k]| > threshold (strictly greater); a threshold <= 0 turns
  the decomposition off;
* vector-wise scales: one per activation row (max |X[m, k]| over the
  non-outlier columns) and one per weight row, i.e. per output feature (max
  |W[n, k]| over all k: the weight is quantized once, when it is loaded,
  before any activation is seen);
* 8-bit code: symmetric linear with 127 levels per side,
  q = rint(RN(127 * v / s)) - 127 * v is exact in float32 for fp16 and bf16
  inputs, RN is the float32 rounding of the quotient, rint rounds half to
  even; s = 0 gives q = 0;
* "16-bit" is fp16; the outlier product uses the weight as the stored int8
  gives it back, w_hat = fp16(RN(RN(q * s) / 127));
* output y = fp16(C * sx * sw / 127^2 + sum over outlier k of x * w_hat),
  C = the exact integer sum of q_x * q_w over the non-outlier columns.
"""
from __future__ import annotations

import numpy as np

DEFAULT_THRESHOLD = 6.0   # llm_int8_threshold (tutorial section 四)
LEVELS = 127


def f16_to_f32(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) -> float32 (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> fp16 bit patterns, round to nearest even (NumPy's cast)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def outlier_columns(x: np.ndarray, threshold: float = DEFAULT_THRESHOLD) -> np.ndarray:
    """Boolean [K]: column k of x [M, K] holds a value with |x| > threshold."""
    x = np.asarray(x, dtype=np.float32)
    if threshold <= 0 or x.shape[0] == 0:
        return np.zeros(x.shape[1], dtype=bool)
    return np.any(np.abs(x) > np.float32(threshold), axis=0)


def quantize_rows(a: np.ndarray, exclude: np.ndarray | None = None):
    """Vector-wise int8 quantization of the rows of a [R, K] (float32 values
    of fp16 / bf16 numbers): scale s_r = max |a[r, k]| over the columns not
    in ``exclude``; q = rint(RN(127 * a / s_r)) there, 0 in the excluded
    columns and in rows with s_r = 0.  Returns (q int8 [R, K], s float32 [R])."""
    a = np.asarray(a, dtype=np.float32)
    keep = np.ones(a.shape[1], dtype=bool) if exclude is None else ~np.asarray(exclude)
    kept = np.where(keep[None, :], a, np.float32(0))
    s = np.max(np.abs(kept), axis=1).astype(np.float32) if a.shape[1] else \
        np.zeros(a.shape[0], np.float32)
    num = np.float32(LEVELS) * kept                       # exact for 16-bit inputs
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (num / s[:, None]).astype(np.float32)      # IEEE float32 division
    q = np.where(s[:, None] > 0, np.rint(quot), 0).astype(np.int8)
    return q, s


def dequantize_rows(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The 16-bit weight the stored int8 gives back, as fp16 bit patterns:
    fp16(RN(RN(q * s) / 127))."""
    prod = (np.asarray(q, dtype=np.float32) * np.asarray(s, np.float32)[:, None]).astype(np.float32)
    return f32_to_f16_bits((prod / np.float32(LEVELS)).astype(np.float32))


def matmul_ref(x_bits: np.ndarray, wq: np.ndarray, sw: np.ndarray,
               threshold: float = DEFAULT_THRESHOLD):
    """y_ref [M, N] (fp64) of the decomposition for fp16 activations x [M, K]
    (bit patterns) and the stored weight (wq int8 [N, K], sw float32 [N]),
    with the per-output error scale: the same sums taken over absolute
    values.  Also returns the outlier mask and the activation codes/scales."""
    x = f16_to_f32(x_bits)
    outl = outlier_columns(x, threshold)
    xq, sx = quantize_rows(x, outl)
    keep = ~outl
    c = xq[:, keep].astype(np.int64) @ wq[:, keep].astype(np.int64).T     # exact integers
    cabs = np.abs(xq[:, keep]).astype(np.int64) @ np.abs(wq[:, keep]).astype(np.int64).T
    scale = sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :] / (LEVELS * LEVELS)
    w_hat = f16_to_f32(dequantize_rows(wq, sw)).astype(np.float64)
    xo = x[:, outl].astype(np.float64)
    wo = w_hat[:, outl]
    y = c.astype(np.float64) * scale + xo @ wo.T
    bound = cabs.astype(np.float64) * scale + np.abs(xo) @ np.abs(wo).T
    return y, bound, outl, xq, sx


def ulp_f16(v: np.ndarray) -> np.ndarray:
    """Spacing of fp16 numbers at |v| (2^(e-10) for 2^e <= |v|, 2^-24 below
    the normal range)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -14, 2.0 ** (e - 10), 2.0 ** -24)


def tolerance(y_ref: np.ndarray, bound: np.ndarray) -> np.ndarray:
    """|y - y_ref| <= 2e-3 * bound + one fp16 ulp of y_ref."""
    return 2e-3 * bound + ulp_f16(y_ref)
