"""CPU oracle for NF4 / FP4 blockwise quantization, double quantization,
dequantization and the dequantize-then-multiply matmul.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) imports, links or runs this file.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may use it.  It shares no code, table or constant
generator with the CUDA path: it builds its own code tables from their
definitions, and it only shares the seeded input generators in ``synth``.

It is deliberately plain and slow: NumPy fp32 for the element-wise steps the
method defines in single precision (NumPy's float32 division, subtraction and
multiplication are IEEE round-to-nearest-even, no flush-to-zero), exact
integer / ``fractions.Fraction`` arithmetic where a step is a reduction, and
fp64 for the matmul reference.

Sources (web pages about the bitsandbytes library; cited by page title and
section):

* "bitsandbytes tutorial" (mlqm.cn/news/394670), section 2.3: data-free
  "absmax" quantization, one scale per block;
  section 3.2: NF4, 16 levels placed by the density of the normal
  distribution, dense near 0 and sparse in the tails;
  section 3.3: double quantization - the per-block scales are themselves
  quantized a second time;
  section 3.4: "4-bit stored, 16-bit computed" - weights are dequantized to
  the compute dtype (bf16) and an ordinary float matmul follows;
  section 四 (key settings): ``bnb_4bit_quant_type`` nf4 | fp4,
  ``bnb_4bit_use_double_quant``, ``bnb_4bit_compute_dtype``.
* "bitsandbytes introduction" (modelers.csdn.net), section 一, item 7: 4-bit
  quantization comes as FP4 or NF4; section 三, example 2: FP4 is the default
  4-bit type.
* "bitsandbytes: quantifier un modèle PyTorch sans quitter PyTorch"
  (hysenlabs.com): blockwise quantization of the weights.

The pages give the method in prose only.  The exact constants used here are
the ones stated for this workload: blocksize 64 with an fp32 absmax per
block; NF4 levels = Phi^-1 of 8 points evenly spaced from 0.9677083 down to
0.5 (0.5 excluded) on the positive side, -Phi^-1 of 7 such points on the
negative side, plus 0, all divided by the largest; double quantization =
absmax minus its mean, 8-bit blockwise in blocks of 256; FP4 = the E2M1
magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}/6 with a sign.  Readings of what the
pages leave open (tie rule, nibble order, the 8-bit map of the scales, the
rounding of the mean) are marked READING below.

Pins: every function is checked by ``tests/test_oracle_pins.py`` against
something other than itself (closed forms, invariants, brute force with exact
rational arithmetic, torch library routines for the bf16 cast and the
matmul).  One comparison is missing: the NF4 table is not compared against an
externally published list of its 16 values, because no such list is on the
pages or on this machine (parity unpinned for that comparison only; the table
is pinned by its definition and invariants).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import scipy.special

BLOCKSIZE = 64        # elements per absmax block
DQ_BLOCKSIZE = 256    # absmax values per double-quantization block
NF4_OFFSET = 0.9677083

CODE_NF4 = 0
CODE_FP4 = 1


# ------------------------------------------------------------------ fp helpers
def f32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even.

    Written out on the bit pattern: add 0x7FFF plus the lowest kept bit, then
    drop the low 16 bits.  NaN stays a quiet NaN with its sign.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        sign = ((u >> np.uint64(16)) & np.uint64(0x8000)).astype(np.uint16)
        r = np.where(nan, sign | np.uint16(0x7FC0), r)
    return r


# compute dtypes (the dequantized weights, x and y): tutorial section 四,
# bnb_4bit_compute_dtype; bf16 is the default
DT_BF16 = 0
DT_F16 = 1


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) -> float32 (exact widening)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> fp16 bit patterns, round to nearest, ties to even, with
    overflow to infinity and gradual underflow (NumPy's IEEE conversion)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    with np.errstate(over="ignore"):
        return x.astype(np.float16).view(np.uint16)


def to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """float32 -> bit patterns of the compute dtype."""
    return f32_to_bf16_bits(x) if dtype == DT_BF16 else f32_to_f16_bits(x)


def from_bits(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Bit patterns of the compute dtype -> float32 (exact)."""
    return bf16_bits_to_f32(bits) if dtype == DT_BF16 else f16_bits_to_f32(bits)


def round_fraction_to_f32(v: Fraction) -> np.float32:
    """Nearest float32 to the exact rational ``v`` (ties to even mantissa)."""
    if v == 0:
        return np.float32(0.0)
    c = np.float32(float(v))          # float(Fraction) is correctly rounded
    cands = [np.nextafter(c, np.float32(-np.inf)), c,
             np.nextafter(c, np.float32(np.inf))]
    best, best_d = None, None
    for cand in cands:
        if not np.isfinite(cand):
            continue
        d = abs(Fraction(float(cand)) - v)
        if best is None or d < best_d or (
                d == best_d and int(np.float32(cand).view(np.uint32)) % 2 == 0):
            best, best_d = np.float32(cand), d
    return best


def fma_f32(a, b, c) -> np.ndarray:
    """float32 fused multiply-add: nearest float32 to the exact a*b + c.

    a*b of two float32 is exact in fp64; the fp64 sum s may be inexact, so the
    exact remainder e (s + e == a*b + c) is taken with Knuth's TwoSum.  Only
    when s falls exactly on a midpoint between two float32 does e decide the
    direction; everywhere else rounding s is rounding a*b + c.
    """
    a = np.asarray(a, dtype=np.float32).astype(np.float64)
    b = np.asarray(b, dtype=np.float32).astype(np.float64)
    c = np.asarray(c, dtype=np.float32).astype(np.float64)
    p = a * b
    s = p + c
    bb = s - p
    e = (p - (s - bb)) + (c - bb)
    r = s.astype(np.float32)
    r64 = r.astype(np.float64)
    inexact = r64 != s
    toward = np.where(r64 < s, np.float32(np.inf), np.float32(-np.inf))
    other = np.nextafter(r, toward.astype(np.float32))
    midpoint = inexact & ((r64 + other.astype(np.float64)) * 0.5 == s)
    need = midpoint & (e != 0)
    if np.any(need):
        up = e > 0
        # pick the neighbour of s on the side of e
        hi = np.where(r64 > s, r, other)
        lo = np.where(r64 < s, r, other)
        r = np.where(need, np.where(up, hi, lo), r)
    return r.astype(np.float32)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (2^(e-7) for 2^e <= |v| < 2^(e+1)),
    never below the smallest bf16 subnormal 2^-133."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(v)               # v = f * 2^ex, f in [0.5, 1)
    u = np.ldexp(1.0, (ex - 8).astype(np.int64))
    return np.maximum(np.where(v == 0, 0.0, u), 2.0 ** -133)


# ------------------------------------------------------------------ code tables
def nf4_code_table() -> np.ndarray:
    """The 16 NF4 levels, ascending, as float32 (index 0..15 = code).

    Section 3.2 of the tutorial: levels follow the normal density.  Built from
    the stated construction in fp64: Phi^-1 (scipy.special.ndtri) of 8 points
    evenly spaced from 0.9677083 down to 0.5 (0.5 dropped) for the positive
    side, the negatives of Phi^-1 of 7 such points for the negative side,
    and 0; divided by the largest; sorted; rounded to float32.
    READING: "evenly spaced ... excluding 0.5" is numpy.linspace(offset, 0.5,
    n + 1) without its last point; codes are numbered in ascending order, so
    0 is code 7 and +1 is code 15.
    """
    pos = scipy.special.ndtri(np.linspace(NF4_OFFSET, 0.5, 9)[:-1])
    neg = -scipy.special.ndtri(np.linspace(NF4_OFFSET, 0.5, 8)[:-1])
    v = np.concatenate([pos, [0.0], neg])
    v = v / v.max()
    v.sort()
    return v.astype(np.float32)


FP4_MAGNITUDES = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64) / 6.0


def fp4_code_table() -> np.ndarray:
    """FP4 value of each 4-bit code, float32, indexed by code.

    E2M1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} / 6 with a sign.
    READING: code = (sign << 3) | j with j the magnitude index; code 8 is
    -0.0, never produced by the encoder.
    """
    m = FP4_MAGNITUDES.astype(np.float32)
    return np.concatenate([m, -m]).astype(np.float32)


def code_table(code: int) -> np.ndarray:
    return nf4_code_table() if code == CODE_NF4 else fp4_code_table()


# ------------------------------------------------------------------ quantize
def absmax_blocks(w: np.ndarray, blocksize: int = BLOCKSIZE) -> np.ndarray:
    """Per-block fp32 max |w| over consecutive ``blocksize`` elements of the
    row-major weight (tutorial section 2.3: one absmax scale per block).
    ``w`` is float32 (bf16 inputs are widened first, which is exact)."""
    w = np.asarray(w, dtype=np.float32).reshape(-1, blocksize)
    return np.abs(w).max(axis=1).astype(np.float32)


def normalize(w: np.ndarray, absmax: np.ndarray,
              blocksize: int = BLOCKSIZE) -> np.ndarray:
    """wn = fp32(w / absmax) per element; wn = 0 in an all-zero block."""
    w = np.asarray(w, dtype=np.float32).reshape(-1, blocksize)
    a = np.asarray(absmax, dtype=np.float32).reshape(-1, 1)
    safe = np.where(a == 0, np.float32(1), a)
    wn = np.where(a == 0, np.float32(0), w / safe)
    return wn.astype(np.float32).reshape(-1)


def _nearest(values: np.ndarray, levels: np.ndarray, chunk=1 << 20):
    """Index of the nearest level (fp64 distances); on an exact tie the lower
    index wins (numpy.argmin returns the first minimum)."""
    levels = np.asarray(levels, dtype=np.float64)
    out = np.empty(values.shape[0], dtype=np.uint8)
    for s in range(0, values.shape[0], chunk):
        v = values[s:s + chunk].astype(np.float64)[:, None]
        out[s:s + chunk] = np.argmin(np.abs(v - levels[None, :]), axis=1)
    return out


def encode(wn: np.ndarray, code: int = CODE_NF4) -> np.ndarray:
    """4-bit code of each normalized value (tutorial section 3.2: nearest
    level).

    NF4: the nearest of the 16 ascending levels; READING: an exact tie goes
    to the lower index (towards -1).
    FP4: the nearest magnitude of |wn| (a tie goes to the smaller magnitude),
    then the sign bit when wn < 0 and the magnitude is not 0.
    """
    wn = np.asarray(wn, dtype=np.float32).reshape(-1)
    if code == CODE_NF4:
        return _nearest(wn, nf4_code_table())
    j = _nearest(np.abs(wn), FP4_MAGNITUDES.astype(np.float32))
    sign = (wn < 0) & (j > 0)
    return (j | (sign.astype(np.uint8) << 3)).astype(np.uint8)


def pack_nibbles(idx: np.ndarray) -> np.ndarray:
    """Two codes per byte.  READING (no layout on the pages): element 2i goes
    to bits 7..4 and element 2i+1 to bits 3..0 of byte i."""
    idx = np.asarray(idx, dtype=np.uint8).reshape(-1, 2)
    return ((idx[:, 0] << 4) | (idx[:, 1] & 0x0F)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8).reshape(-1)
    out = np.empty(p.shape[0] * 2, dtype=np.uint8)
    out[0::2] = p >> 4
    out[1::2] = p & 0x0F
    return out


def quantize(w: np.ndarray, code: int = CODE_NF4, blocksize: int = BLOCKSIZE):
    """Blockwise 4-bit quantization: (packed uint8 [n/2], absmax fp32 [n/64])."""
    w = np.asarray(w, dtype=np.float32).reshape(-1)
    a = absmax_blocks(w, blocksize)
    idx = encode(normalize(w, a, blocksize), code)
    return pack_nibbles(idx), a


# ------------------------------------------------------------ double quant
def exact_sum_scaled(absmax: np.ndarray) -> int:
    """Exact sum of float32 values, returned as the integer sum * 2^149.

    Every float32 is m * 2^(E' - 150) with m < 2^24 and E' = max(E, 1) for
    the biased exponent E, so v * 2^149 = m << (E' - 1) is an integer; the
    mantissas are added per exponent (int64 cannot overflow: < 2^24 * 2^38)
    and the groups are combined as Python integers.
    """
    u = np.ascontiguousarray(absmax, dtype=np.float32).view(np.uint32).reshape(-1)
    e = ((u >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int64)
    frac = (u & np.uint32(0x7FFFFF)).astype(np.int64)
    m = np.where(e > 0, frac | (1 << 23), frac)
    ep = np.maximum(e, 1)
    total = 0
    for ev in np.unique(ep):
        total += int(m[ep == ev].sum()) << int(ev - 1)
    return total


def mean_f32(absmax: np.ndarray) -> np.float32:
    """READING of "the mean of the scales": the float32 nearest (ties to even)
    to the exact arithmetic mean of all absmax values of the tensor."""
    a = np.asarray(absmax, dtype=np.float32).reshape(-1)
    if a.size == 0:
        return np.float32(0.0)
    return round_fraction_to_f32(Fraction(exact_sum_scaled(a), a.size << 149))


def double_quant(absmax: np.ndarray, dq_blocksize: int = DQ_BLOCKSIZE):
    """Double quantization (tutorial section 3.3): the fp32 absmax scales are
    quantized a second time.

    offset = mean(absmax) (see ``mean_f32``); c = fp32(absmax - offset);
    per block d of 256 values scale2[d] = fp32(max|c| / 127);
    q = clamp(rint_half_even(fp32(c / scale2[d])), -127, 127), q = 0 where
    scale2 == 0.  The last block may be partial.
    READING: "8-bit blockwise" is the symmetric linear int8 map of the same
    absmax scheme (section 2.3), with ties to even and no -128.
    Returns (absmax_q int8 [n_b], scale2 fp32 [n_d], offset float32).
    """
    a = np.asarray(absmax, dtype=np.float32).reshape(-1)
    nb = a.size
    offset = mean_f32(a)
    c = (a - offset).astype(np.float32)
    nd = (nb + dq_blocksize - 1) // dq_blocksize
    scale2 = np.empty(nd, dtype=np.float32)
    q = np.empty(nb, dtype=np.int8)
    for d in range(nd):
        cb = c[d * dq_blocksize:(d + 1) * dq_blocksize]
        s2 = np.float32(np.abs(cb).max()) / np.float32(127)
        scale2[d] = s2
        if s2 == 0:
            q[d * dq_blocksize:(d + 1) * dq_blocksize] = 0
        else:
            r = np.rint((cb / s2).astype(np.float32))
            q[d * dq_blocksize:(d + 1) * dq_blocksize] = np.clip(r, -127, 127)
    return q, scale2, np.float32(offset)


def block_scales(absmax_q=None, scale2=None, offset=None, absmax=None,
                 dq_blocksize: int = DQ_BLOCKSIZE) -> np.ndarray:
    """Scale of each 64-block as the dequantizer sees it.

    With double quant: s_b = fp32 fma(q_b, scale2[b // 256], offset) (one
    rounding).  READING: quantization used the exact fp32 absmax; dequant uses
    the reconstructed s_b, following the order "quantize the weights, then
    quantize the scales" of section 3.3.  Without double quant: s_b = absmax.
    """
    if absmax_q is None:
        return np.asarray(absmax, dtype=np.float32).reshape(-1)
    q = np.asarray(absmax_q, dtype=np.int8).reshape(-1).astype(np.float32)
    d = np.arange(q.size) // dq_blocksize
    return fma_f32(q, np.asarray(scale2, dtype=np.float32)[d],
                   np.float32(offset))


def dequantize(packed: np.ndarray, scales: np.ndarray, code: int = CODE_NF4,
               blocksize: int = BLOCKSIZE, dtype: int = DT_BF16) -> np.ndarray:
    """Weights in the compute dtype (uint16 bit patterns):
    w_hat = round(fp32(code[idx] * s_b)) to bf16 or fp16 (tutorial section
    3.4: weights stored in 4 bits, dequantized to the compute dtype)."""
    idx = unpack_nibbles(packed)
    table = code_table(code)
    s = np.repeat(np.asarray(scales, dtype=np.float32), blocksize)
    prod = (table[idx] * s).astype(np.float32)
    return to_bits(prod, dtype)


def quantize_full(w, code=CODE_NF4, double_quant_on=True):
    """Whole path up to the stored state and its bf16 dequantization."""
    packed, absmax = quantize(w, code)
    if double_quant_on:
        q, s2, off = double_quant(absmax)
        scales = block_scales(q, s2, off)
    else:
        q, s2, off = None, None, None
        scales = absmax
    return dict(packed=packed, absmax=absmax, absmax_q=q, scale2=s2,
                offset=off, w_hat=dequantize(packed, scales, code))


# ------------------------------------------------------------------ matmul
def matmul_ref(x_bits: np.ndarray, w_hat_bits: np.ndarray, dtype: int = DT_BF16):
    """y_ref = x . w_hat^T in fp64 from compute-dtype inputs (section 3.4:
    dequantize to the compute dtype, then an ordinary matmul), and the
    per-output error scale sum_k |x_k * w_hat_k|.  x [M, K], w_hat [N, K] as
    bit patterns of the compute dtype."""
    x = from_bits(x_bits, dtype).astype(np.float64)
    w = from_bits(w_hat_bits, dtype).astype(np.float64)
    return x @ w.T, np.abs(x) @ np.abs(w).T


def matmul_dx_ref(dy_bits: np.ndarray, w_hat_bits: np.ndarray, dtype: int = DT_BF16):
    """dX_ref = dY . w_hat in fp64 from compute-dtype inputs, and the
    per-output error scale sum_n |dY_n * w_hat_nk|.  dY [M, N], w_hat [N, K]
    as bit patterns of the compute dtype.

    This is the gradient of y = x . w_hat^T with respect to x, the one
    gradient a frozen 4-bit base layer needs when only LoRA adapters train
    (tutorial section 5.4): dL/dx_k = sum_n dL/dy_n * w_hat[n, k]."""
    dy = from_bits(dy_bits, dtype).astype(np.float64)
    w = from_bits(w_hat_bits, dtype).astype(np.float64)
    return dy @ w, np.abs(dy) @ np.abs(w)


def ulp_f16(v: np.ndarray) -> np.ndarray:
    """Spacing of fp16 numbers at |v| (2^(e-10) for 2^e <= |v| < 2^(e+1),
    2^-24 below the normal range)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -14, 2.0 ** (e - 10), 2.0 ** -24)


def matmul_tolerance(y_ref: np.ndarray, bound: np.ndarray, dtype: int = DT_BF16) -> np.ndarray:
    """|y - y_ref| <= 2e-3 * sum_k |x_k w_hat_k| + one ulp of y_ref in the
    compute dtype."""
    return 2e-3 * bound + (ulp_bf16(y_ref) if dtype == DT_BF16 else ulp_f16(y_ref))


def bits_per_parameter(n: int, k: int, double_quant_on: bool = True) -> float:
    """Stored bits per weight: 4-bit codes plus the scale state."""
    nb = n * k // BLOCKSIZE
    if double_quant_on:
        nd = (nb + DQ_BLOCKSIZE - 1) // DQ_BLOCKSIZE
        total = n * k * 4 + nb * 8 + nd * 32 + 32
    else:
        total = n * k * 4 + nb * 32
    return total / (n * k)
