"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself (closed forms, invariants, exact rational brute force,
independent library routines), so that a dropped term, a wrong sign, a wrong
index or a swapped operand in the oracle fails here.  CPU only."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

from oracle import nf4_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def f32_from_bits(b):
    return np.asarray(b, dtype=np.uint32).view(np.float32)


# ------------------------------------------------------------ bf16 rounding
def test_bf16_rounding_matches_torch_cast():
    x = RNG.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # exact ties, values around the bf16 grid, specials
    ties = f32_from_bits(RNG.integers(0, 1 << 31, 5000).astype(np.uint32)
                         & np.uint32(0xFFFF8000) | np.uint32(0x8000))
    sub = f32_from_bits(RNG.integers(1, 1 << 23, 5000).astype(np.uint32))
    spec = np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, -3.4028235e38,
                     1.0, -1.0, 1.00390625, 1.001953125], dtype=np.float32)
    allx = np.concatenate([x, ties, -ties, sub, spec])
    ours = o.f32_to_bf16_bits(allx)
    ref = torch.from_numpy(allx).to(torch.bfloat16).view(torch.int16).numpy()
    ref = ref.view(np.uint16)
    nan = np.isnan(allx)            # NaN payloads are a convention; only
    assert nan.sum() > 0            # NaN-ness has to agree
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(o.bf16_bits_to_f32(ours[nan])))


def test_bf16_widen_is_exact():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = o.bf16_bits_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (f == ref) | (np.isnan(f) & np.isnan(ref))
    assert same.all()


# ------------------------------------------------------------ fp16 compute dtype
def _f16_grid():
    """Every finite fp16 value, ascending, as exact float64 with its bits:
    built from the IEEE half format definition (sign, 5-bit exponent with
    bias 15, 10-bit fraction; exponent 0 = subnormal), not from a cast."""
    vals, bits = [], []
    for e in range(31):
        for f in range(1024):
            v = (f / 1024.0) * 2.0 ** -14 if e == 0 else (1 + f / 1024.0) * 2.0 ** (e - 15)
            vals.append(v); bits.append((e << 10) | f)
    pos_v, pos_b = np.array(vals), np.array(bits, dtype=np.uint32)
    v = np.concatenate([-pos_v[::-1][:-1], pos_v])          # drop -0
    b = np.concatenate([(pos_b[::-1][:-1] | 0x8000), pos_b]).astype(np.uint16)
    return v, b


def _f16_nearest_even(x64: np.ndarray) -> np.ndarray:
    """Brute force round-to-nearest-even onto the fp16 grid with overflow to
    infinity at |x| >= 65520 (the midpoint past the largest finite value)."""
    v, b = _f16_grid()
    out = np.empty(x64.shape, dtype=np.uint16)
    for i, x in enumerate(x64):
        if abs(x) >= 65520.0:
            out[i] = 0x7C00 | (0x8000 if x < 0 else 0)
            continue
        j = np.searchsorted(v, x)
        cands = [k for k in (j - 1, j) if 0 <= k < len(v)]
        d = [abs(v[k] - x) for k in cands]
        best = min(d)
        ks = [k for k, dd in zip(cands, d) if dd == best]
        k = ks[0] if len(ks) == 1 else min(ks, key=lambda q: b[q] & 1)  # even mantissa
        out[i] = b[k]
        if out[i] == 0 and np.signbit(x):   # rounding to zero keeps the sign
            out[i] = 0x8000
    return out


def test_f16_rounding_matches_brute_force_grid():
    x = np.concatenate([
        RNG.standard_normal(3000).astype(np.float32) * np.float32(100.0),
        (RNG.standard_normal(1000) * 1e-5).astype(np.float32),          # subnormal range
        np.array([65504.0, 65519.0, 65520.0, 65536.0, 1e6, -65520.0, 0.0, -0.0,
                  2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 1.0 + 2.0 ** -11,
                  1.0 + 3 * 2.0 ** -11], dtype=np.float32)])
    # exact midpoints between neighbouring fp16 values (representable in fp32)
    v, _ = _f16_grid()
    mids = ((v[:-1] + v[1:]) / 2)[::37].astype(np.float32)
    x = np.concatenate([x, mids])
    got, want = o.f32_to_f16_bits(x), _f16_nearest_even(x.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(repr(x[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_f16_widen_is_exact():
    v, b = _f16_grid()
    assert np.array_equal(o.f16_bits_to_f32(b).astype(np.float64), v)


def test_dequant_f16_closed_form():
    # unit scale: w_hat is the code value rounded once to fp16
    t = o.nf4_code_table()
    packed = o.pack_nibbles(np.arange(16, dtype=np.uint8).repeat(4))
    got = o.f16_bits_to_f32(o.dequantize(packed, np.ones(1, np.float32), dtype=o.DT_F16))
    want = np.array([np.float16(float(c)) for c in t.repeat(4)], dtype=np.float32)
    assert np.array_equal(got, want)
    # a scale that overflows fp16 gives infinities, as IEEE rounding does
    big = o.f16_bits_to_f32(o.dequantize(packed, np.full(1, 1e5, np.float32), dtype=o.DT_F16))
    assert np.isinf(big[-1]) and big[-1] > 0 and big[28] == 0.0


def test_ulp_f16_spacing():
    v, b = _f16_grid()
    pos = v[v > 0][:-1]
    nxt = v[v > 0][1:]
    assert np.array_equal(o.ulp_f16(pos), nxt - pos)


# ------------------------------------------------------------ fma / rounding
def _exact_f32_round(v: Fraction) -> np.float32:
    """Brute force: scan the float32 neighbourhood and pick the nearest,
    ties to even.  Independent of round_fraction_to_f32's candidate logic."""
    approx = np.float32(float(v))
    cands = [approx]
    for _ in range(3):
        cands.append(np.nextafter(cands[-1], np.float32(np.inf)))
    c = approx
    for _ in range(3):
        c = np.nextafter(c, np.float32(-np.inf))
        cands.append(c)
    best = None
    for c in cands:
        d = abs(Fraction(float(c)) - v)
        key = (d, int(np.float32(c).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return np.float32(best[1])


def test_fma_f32_exact_on_random_and_midpoints():
    a = RNG.standard_normal(3000).astype(np.float32)
    b = RNG.standard_normal(3000).astype(np.float32)
    c = RNG.standard_normal(3000).astype(np.float32)
    # crafted: c in [1, 2), a*b = half an ulp of c, +/- a hair
    cc = (1 + RNG.random(600)).astype(np.float32)
    half = np.float32(2.0 ** -24)
    bb = np.concatenate([np.ones(200), 1 + 2.0 ** -23 * np.arange(1, 201),
                         1 - 2.0 ** -24 * np.arange(1, 201)]).astype(np.float32)
    aa = np.full(600, half, dtype=np.float32)
    # int8 q times a scale plus an offset, the way the scales use it
    q = RNG.integers(-127, 128, 2000).astype(np.float32)
    s2 = (RNG.random(2000) * 1e-3).astype(np.float32)
    off = np.float32(0.0513)
    A = np.concatenate([a, aa, q])
    B = np.concatenate([b, bb, s2])
    C = np.concatenate([c, cc, np.full(2000, off, np.float32)])
    got = o.fma_f32(A, B, C)
    for i in range(A.size):
        want = _exact_f32_round(Fraction(float(A[i])) * Fraction(float(B[i]))
                                + Fraction(float(C[i])))
        assert got[i] == want, (i, A[i], B[i], C[i], got[i], want)


def test_fma_differs_from_mul_then_add_somewhere():
    """a*b = 2^-24 (1 - 2^-26) is not a float32; rounded first it becomes
    2^-24, half an ulp of c in [1, 2), a tie.  Fused, c + a*b lies just below
    the midpoint and rounds to c; unfused, odd c rounds up to even."""
    cc = np.float32(1.0) + np.float32(2.0 ** -23) * np.arange(64, dtype=np.float32)
    aa = np.full(64, 1 - 2.0 ** -13, np.float32)
    bb = np.full(64, 2.0 ** -24 * (1 + 2.0 ** -13), np.float32)
    fused = o.fma_f32(aa, bb, cc)
    unfused = (aa * bb + cc).astype(np.float32)
    assert np.array_equal(fused, cc)
    odd = (cc.view(np.uint32) & 1) == 1
    assert np.all(unfused[odd] > cc[odd]) and np.array_equal(unfused[~odd], cc[~odd])


def test_round_fraction_to_f32_matches_numpy_cast_and_ties():
    v = np.concatenate([RNG.standard_normal(3000) * 10.0 ** RNG.integers(-40, 38, 3000),
                        np.abs(RNG.standard_normal(100)) * 1e-44])
    for x in np.abs(v):
        assert o.round_fraction_to_f32(Fraction(float(x))) == np.float32(x)
    # exact midpoints between consecutive float32: ties to even
    for k in range(200):
        lo = np.float32(1 + k * 2.0 ** -23)
        hi = np.nextafter(lo, np.float32(2))
        mid = (Fraction(float(lo)) + Fraction(float(hi))) / 2
        want = lo if int(lo.view(np.uint32)) % 2 == 0 else hi
        assert o.round_fraction_to_f32(mid) == want


# ------------------------------------------------------------ exact mean
def test_exact_sum_matches_fraction_sum():
    for trial in range(30):
        n = int(RNG.integers(1, 400))
        e = RNG.integers(-149, 120, n)
        v = (RNG.random(n) * np.exp2(e.astype(np.float64))).astype(np.float32)
        v[RNG.random(n) < 0.1] = 0
        v = np.abs(v)
        want = sum(Fraction(float(x)) for x in v) * (1 << 149)
        assert want.denominator == 1
        assert o.exact_sum_scaled(v) == want.numerator


def test_mean_closed_forms():
    assert o.mean_f32(np.array([1, 2, 3, 4], np.float32)) == np.float32(2.5)
    x = np.float32(0.0371)
    assert o.mean_f32(np.full(777, x, np.float32)) == x
    # mean of two neighbours is their midpoint: a tie, goes to the even one
    lo = np.float32(1.0)
    hi = np.nextafter(lo, np.float32(2))
    assert o.mean_f32(np.array([lo, hi], np.float32)) == lo
    lo2, hi2 = hi, np.nextafter(hi, np.float32(2))
    assert o.mean_f32(np.array([lo2, hi2], np.float32)) == hi2
    # 1/3 rounds to the float32 nearest to one third
    assert o.mean_f32(np.array([1, 0, 0], np.float32)) == np.float32(1.0 / 3.0)
    # a dynamic range far beyond fp64 is still exact: huge + 2 tiny values
    big = np.float32(3e38)
    tiny = np.float32(1e-45)
    m = o.mean_f32(np.array([big, tiny, tiny], np.float32))
    assert m == np.float32(1e38)


# ------------------------------------------------------------ code tables
def test_nf4_table_invariants():
    t = o.nf4_code_table()
    assert t.dtype == np.float32 and t.shape == (16,)
    assert np.all(np.diff(t) > 0)
    assert t[0] == -1.0 and t[15] == 1.0 and t[7] == 0.0
    assert (t < 0).sum() == 7 and (t > 0).sum() == 8
    gaps = np.diff(t.astype(np.float64))
    assert 0.0795 < gaps.min() < 0.0797 and 0.3037 < gaps.max() < 0.3039
    # dense near 0, sparse at the tails (normal density), on both sides
    assert np.all(np.diff(gaps[7:]) > 0) and np.all(np.diff(gaps[:7]) < 0)


def test_nf4_table_is_normal_quantiles_via_cdf():
    """Through the normal CDF (scipy.special.ndtr, not the inverse used to
    build the table) the levels map back onto the evenly spaced points."""
    t = o.nf4_code_table().astype(np.float64)
    scale = scipy.special.ndtri(o.NF4_OFFSET)
    p = scipy.special.ndtr(t * scale)
    pos = np.linspace(o.NF4_OFFSET, 0.5, 9)[:-1]
    neg = np.linspace(o.NF4_OFFSET, 0.5, 8)[:-1]
    assert np.allclose(np.sort(p[8:])[::-1], pos, atol=2e-8)
    assert np.allclose(np.sort(1 - p[:7])[::-1], neg, atol=2e-8)


def _phi_inv_bisect(p):
    lo, hi = 0.0, 10.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if 0.5 * math.erfc(-mid / math.sqrt(2.0)) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def test_nf4_table_matches_independent_bisection():
    pos = [_phi_inv_bisect(p) for p in np.linspace(o.NF4_OFFSET, 0.5, 9)[:-1]]
    neg = [-_phi_inv_bisect(p) for p in np.linspace(o.NF4_OFFSET, 0.5, 8)[:-1]]
    v = np.array(pos + [0.0] + neg)
    v = np.sort(v / v.max()).astype(np.float32)
    assert np.array_equal(v, o.nf4_code_table())


def test_nf4_offset_matches_closed_form():
    # 0.9677083 agrees to 7 digits with 1 - (1/32 + 1/30) / 2
    assert abs(o.NF4_OFFSET - (1 - 0.5 * (1 / 32 + 1 / 30))) < 1e-7


def test_fp4_table_closed_form():
    t = o.fp4_code_table()
    assert np.array_equal(t[:8] * np.float32(6),
                          np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32))
    assert np.array_equal(t[8:], -t[:8])
    assert t[7] == 1.0 and t[15] == -1.0


# ------------------------------------------------------------ encode / pack
def _brute_nearest(v: float, levels, tie_lower=True):
    fv = Fraction(v)
    best = None
    for j, c in enumerate(levels):
        d = abs(fv - Fraction(float(c)))
        if best is None or d < best[0]:
            best = (d, j)
    return best[1]


def test_encode_nf4_bruteforce_small():
    t = o.nf4_code_table()
    mids = [(Fraction(float(t[j])) + Fraction(float(t[j + 1]))) / 2 for j in range(15)]
    vals = list(RNG.uniform(-1, 1, 3000).astype(np.float32))
    for m in mids:   # planted exact ties where representable, and neighbours
        f = np.float32(float(m))
        vals += [f, np.nextafter(f, np.float32(2)), np.nextafter(f, np.float32(-2))]
    vals += [np.float32(0), np.float32(-0.0), np.float32(1), np.float32(-1)]
    vals = np.array(vals, dtype=np.float32)
    got = o.encode(vals, o.CODE_NF4)
    for v, g in zip(vals, got):
        assert g == _brute_nearest(float(v), t), (v, g)


def test_encode_fp4_bruteforce_small():
    mags = o.FP4_MAGNITUDES.astype(np.float32)
    vals = list(RNG.uniform(-1, 1, 3000).astype(np.float32))
    for j in range(7):
        m = (Fraction(float(mags[j])) + Fraction(float(mags[j + 1]))) / 2
        f = np.float32(float(m))
        for s in (1, -1):
            vals += [s * f, s * np.nextafter(f, np.float32(2)),
                     s * np.nextafter(f, np.float32(0))]
    vals += [np.float32(0), np.float32(-0.0)]
    vals = np.array(vals, dtype=np.float32)
    got = o.encode(vals, o.CODE_FP4)
    for v, g in zip(vals, got):
        j = _brute_nearest(abs(float(v)), mags)
        want = j | (8 if (v < 0 and j > 0) else 0)
        assert g == want, (v, g, want)


def test_encode_equals_midpoint_rule_near_every_threshold():
    """Exhaustive over all float32 within 4096 ulps of each NF4 midpoint:
    nearest-with-ties-lower equals counting exact midpoints strictly below."""
    t = o.nf4_code_table().astype(np.float64)
    mids = (t[:-1] + t[1:]) / 2          # exact in fp64
    vals = []
    for m in mids:
        b = np.float32(m).view(np.uint32).astype(np.int64)
        rng = np.arange(b - 4096, b + 4097)
        if m < 0:
            rng = rng[rng >= 0x80000000]
        vals.append(rng.astype(np.uint32).view(np.float32))
    v = np.concatenate(vals)
    want = np.searchsorted(mids, v.astype(np.float64), side="left")
    assert np.array_equal(o.encode(v, o.CODE_NF4), want.astype(np.uint8))


def test_encode_fixed_points_and_absmax_element():
    for code in (o.CODE_NF4, o.CODE_FP4):
        t = o.code_table(code)
        idx = o.encode(t, code)
        for j in range(16):
            if code == o.CODE_FP4 and j == 8:
                assert idx[j] == 0      # -0 encodes as +0
            else:
                assert idx[j] == j
    w = RNG.standard_normal(64 * 50).astype(np.float32)
    packed, a = o.quantize(w, o.CODE_NF4)
    idx = o.unpack_nibbles(packed).reshape(-1, 64)
    wb = w.reshape(-1, 64)
    arg = np.abs(wb).argmax(axis=1)
    top = idx[np.arange(50), arg]
    sgn = wb[np.arange(50), arg] > 0
    assert np.all(np.where(sgn, top == 15, top == 0))


def test_pack_layout_and_roundtrip():
    assert o.pack_nibbles(np.array([1, 2], np.uint8))[0] == 0x12
    assert o.pack_nibbles(np.array([15, 0, 0, 15], np.uint8)).tolist() == [0xF0, 0x0F]
    idx = RNG.integers(0, 16, 1000).astype(np.uint8)
    assert np.array_equal(o.unpack_nibbles(o.pack_nibbles(idx)), idx)


def test_all_zero_block():
    w = np.zeros(128, np.float32)
    w[64:] = RNG.standard_normal(64)
    packed, a = o.quantize(w)
    assert a[0] == 0
    assert np.all(o.unpack_nibbles(packed)[:64] == 7)
    packed, a = o.quantize(w, o.CODE_FP4)
    assert np.all(o.unpack_nibbles(packed)[:64] == 0)


def test_normalize_is_the_correctly_rounded_quotient():
    """wn = fp32(w / absmax) with IEEE division: the float32 nearest to the
    exact rational quotient, checked with Fraction arithmetic on values where
    multiplying by a rounded reciprocal gives a different float32."""
    g = np.random.default_rng(77)
    a = np.abs(g.standard_normal(400)).astype(np.float32) * np.float32(0.03) + np.float32(1e-4)
    w = (g.uniform(-1, 1, (400, 64)) * a[:, None]).astype(np.float32)
    wn = o.normalize(w.reshape(-1), a).reshape(400, 64)
    recip_differs = 0
    for i in range(400):
        r = np.float32(1) / a[i]
        for j in range(0, 64, 4):
            want = _exact_f32_round(Fraction(float(w[i, j])) / Fraction(float(a[i])))
            assert wn[i, j] == want, (i, j, w[i, j], a[i], wn[i, j], want)
            recip_differs += int(np.float32(w[i, j] * r) != want)
    assert recip_differs > 50     # the check can tell the two apart


# ------------------------------------------------------------ double quant
def test_double_quant_worked_example():
    a = np.array([0.5, 1.5], np.float32)
    q, s2, off = o.double_quant(a)
    assert off == np.float32(1.0)
    assert s2[0] == np.float32(0.5) / np.float32(127)
    assert q.tolist() == [-127, 127]
    # all equal: every centered value is 0, scale2 = 0, q = 0, s = offset
    q, s2, off = o.double_quant(np.full(300, 0.25, np.float32))
    assert off == np.float32(0.25) and np.all(s2 == 0) and np.all(q == 0)
    s = o.block_scales(q, s2, off)
    assert np.all(s == np.float32(0.25))


def test_double_quant_rounds_exact_halves_to_even():
    """Worked example with exact .5 quotients: absmax = 1 + c with c in
    {+-127, +-2.5, +-3.5, +-0.5, +-1.5}/128 has the exact mean 1, so
    c = fp32(absmax - 1) exactly, scale2 = (127/128)/127 = 1/128 exactly and
    c / scale2 lands on the halves; ties to even give 2, 4, 0, 2 (rounding
    half away from zero would give 3, 4, 1, 2)."""
    c = np.array([127, -127, 2.5, -2.5, 3.5, -3.5, 0.5, -0.5, 1.5, -1.5]) / 128
    a = (1.0 + c).astype(np.float32)
    assert np.array_equal(a.astype(np.float64) - 1.0, c)      # exact inputs
    q, s2, off = o.double_quant(a)
    assert off == np.float32(1.0) and s2[0] == np.float32(2.0 ** -7)
    assert q.tolist() == [127, -127, 2, -2, 4, -4, 0, 0, 2, -2]


def test_double_quant_invariants():
    a = np.abs(RNG.standard_normal(256 * 7 + 33)).astype(np.float32) * np.float32(0.05)
    q, s2, off = o.double_quant(a)
    assert q.dtype == np.int8 and s2.shape == (8,)
    exact_mean = sum(Fraction(float(x)) for x in a) / a.size
    assert abs(Fraction(float(off)) - exact_mean) <= Fraction(float(np.spacing(off))) / 2
    c = (a - off).astype(np.float32)
    for d in range(8):
        blk = q[d * 256:(d + 1) * 256]
        assert np.abs(blk.astype(np.int32)).max() == 127
        assert s2[d] == np.float32(np.abs(c[d * 256:(d + 1) * 256]).max()) / np.float32(127)
    s = o.block_scales(q, s2, off)
    d = np.arange(a.size) // 256
    err = np.abs(s.astype(np.float64) - a.astype(np.float64))
    bound = s2[d].astype(np.float64) / 2 * (1 + 2.0 ** -22) + 2 * np.spacing(np.abs(a)).astype(np.float64)
    assert np.all(err <= bound)


# ------------------------------------------------------------ dequant
def test_dequant_closed_form_unit_scale():
    for code in (o.CODE_NF4, o.CODE_FP4):
        idx = np.tile(np.arange(16, dtype=np.uint8), 4)
        packed = o.pack_nibbles(idx)
        w = o.dequantize(packed, np.ones(1, np.float32), code)
        want = torch.from_numpy(o.code_table(code)[idx]).to(torch.bfloat16)
        assert np.array_equal(w, want.view(torch.int16).numpy().view(np.uint16))


def test_dequant_single_rounding_with_scales():
    """w_hat = bf16(fp32(code * s)): the exact product rounded once to
    float32 (Fraction arithmetic), then to bf16 by torch's cast.  The scales
    cover many magnitudes; rounding the code to bf16 before the product (a
    double rounding) gives other bits on a good share of them."""
    g = np.random.default_rng(91)
    s = (np.abs(g.standard_normal(300)) * 10.0 ** g.integers(-6, 3, 300)).astype(np.float32)
    idx = np.tile(np.arange(16, dtype=np.uint8), 4 * 300)
    packed = o.pack_nibbles(idx)
    for code in (o.CODE_NF4, o.CODE_FP4):
        t = o.code_table(code)
        got = o.dequantize(packed, s, code).reshape(300, 64)
        f32 = np.empty((300, 16), np.float32)
        for b in range(300):
            for j in range(16):
                v = _exact_f32_round(Fraction(float(t[j])) * Fraction(float(s[b])))
                f32[b, j] = np.copysign(v, t[j])    # FP4 code 8 is -0: -0 * s = -0
        want = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got[:, :16], want)
        if code == o.CODE_NF4:
            tb = torch.from_numpy(t).to(torch.bfloat16).float().numpy()
            dbl = torch.from_numpy((tb[None, :] * s[:, None]).astype(np.float32)).to(
                torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.sum(dbl != want) > 100


def test_roundtrip_error_bound():
    w = (RNG.standard_normal(64 * 512) * 0.02).astype(np.float32)
    r = o.quantize_full(w)
    what = o.bf16_bits_to_f32(r["w_hat"]).astype(np.float64)
    a = np.repeat(r["absmax"], 64).astype(np.float64)
    s = np.repeat(o.block_scales(r["absmax_q"], r["scale2"], r["offset"]), 64)
    gap = np.diff(o.nf4_code_table().astype(np.float64)).max() / 2
    err = np.abs(what - w)
    bound = gap * a + np.abs(s - a) + np.abs(what) * 2.0 ** -8 + 1e-12
    assert np.all(err <= bound)


def test_nf4_beats_int4_error():
    """Section 3.2 of the tutorial: NF4 error is about 60 % of plain INT4 on
    normal weights.  Soft check: NF4 has the smaller RMSE."""
    w = (RNG.standard_normal(64 * 4096) * 0.02).astype(np.float32)
    packed, a = o.quantize(w)
    what = o.bf16_bits_to_f32(o.dequantize(packed, a)).astype(np.float64)
    rms_nf4 = np.sqrt(np.mean((what - w) ** 2))
    wb = w.reshape(-1, 64).astype(np.float64)
    s = np.abs(wb).max(axis=1, keepdims=True) / 7
    q = np.clip(np.rint(wb / s), -7, 7) * s
    rms_int4 = np.sqrt(np.mean((q - wb) ** 2))
    ratio = rms_nf4 / rms_int4
    assert 0.4 < ratio < 0.95, ratio


# ------------------------------------------------------------ matmul
def test_matmul_ref_against_torch_and_one_hot():
    x = torch.randn(3, 256, dtype=torch.float32).to(torch.bfloat16)
    w = (torch.randn(40, 256) * 0.02).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    y, bound = o.matmul_ref(xb, wb)
    yt = (x.double() @ w.double().T).numpy()
    assert np.allclose(y, yt, rtol=0, atol=1e-12)
    assert np.all(bound >= np.abs(y))
    e = np.zeros((1, 256), np.float32)
    e[0, 17] = 1.0
    eb = o.f32_to_bf16_bits(e)
    y1, _ = o.matmul_ref(eb, wb)
    assert np.array_equal(y1[0], o.bf16_bits_to_f32(wb[:, 17]).astype(np.float64))


def test_matmul_dx_ref_brute_force_one_hot_and_adjoint():
    """dX = dY . w_hat: a triple loop on a tiny case, a one-hot dY row picks
    a row of w_hat exactly, and <dY, x . w_hat^T> = <dY . w_hat, x> ties it
    to the forward reference on a non-square weight."""
    g = np.random.default_rng(5)
    w = o.f32_to_bf16_bits((g.standard_normal((6, 64)) * 0.1).astype(np.float32))
    dy = o.f32_to_bf16_bits(g.standard_normal((3, 6)).astype(np.float32))
    dx, bound = o.matmul_dx_ref(dy, w)
    assert dx.shape == (3, 64)
    W, D = o.bf16_bits_to_f32(w).astype(np.float64), o.bf16_bits_to_f32(dy).astype(np.float64)
    for i in range(3):
        for k in range(64):
            acc = sum(D[i, n] * W[n, k] for n in range(6))
            assert abs(dx[i, k] - acc) <= 1e-12 * max(1.0, abs(acc))
            assert abs(bound[i, k] - sum(abs(D[i, n] * W[n, k]) for n in range(6))) <= 1e-12
    e = np.zeros((1, 6), np.float32)
    e[0, 4] = 1.0
    dx1, _ = o.matmul_dx_ref(o.f32_to_bf16_bits(e), w)
    assert np.array_equal(dx1[0], W[4])
    x = o.f32_to_bf16_bits(g.standard_normal((3, 64)).astype(np.float32))
    y, _ = o.matmul_ref(x, w)
    X = o.bf16_bits_to_f32(x).astype(np.float64)
    assert abs(np.sum(D * y) - np.sum(dx * X)) <= 1e-9 * np.sum(np.abs(D) @ np.abs(W) * np.abs(X))


def test_tolerance_has_ulp_floor():
    y = np.array([0.0, 1.0, 3.0, -1e-3])
    tol = o.matmul_tolerance(y, np.zeros(4))
    assert tol[1] == 2.0 ** -7 and tol[2] == 2.0 ** -6 and tol[0] == 2.0 ** -133


# ------------------------------------------------------------ memory claims
def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=")
                vals[k.strip()] = float(v)
    return vals


def test_bits_per_param_and_page_memory_claims():
    g = _golden("memory_claims.txt")
    bpp = o.bits_per_parameter(4096, 4096, True)
    assert abs(bpp - (4 + 8 / 64 + 32 / 16384 + 32 / (4096 * 4096))) < 1e-12
    assert o.bits_per_parameter(4096, 4096, False) == 4.5
    saving = 4.5 - bpp
    assert 0.1 <= saving < 1.0        # "a few tenths of a bit" per parameter
    gb = 7e9 * bpp / 8 / 1e9
    assert abs(gb - g["nf4_dq_7b_gb"]) < 0.5  # page: 14 GB -> about 4 GB
    assert g["fp16_7b_gb"] == 14.0
    assert abs(bpp / 16 - 0.25) < 0.01       # 4-bit: about 3/4 saved


# ------------------------------------------------------------ planted mistakes
def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant typical slips in the oracle and check a pin above fails."""
    # (1) swapped nibble order
    orig_pack = o.pack_nibbles
    monkeypatch.setattr(o, "pack_nibbles",
                        lambda idx: orig_pack(np.asarray(idx).reshape(-1, 2)[:, ::-1]))
    with pytest.raises(AssertionError):
        test_pack_layout_and_roundtrip()
    monkeypatch.undo()
    # (2) dropped offset in the dequant scale
    orig_bs = o.block_scales
    monkeypatch.setattr(o, "block_scales",
                        lambda q=None, s2=None, off=None, absmax=None, **k:
                        orig_bs(q, s2, np.float32(0), absmax))
    with pytest.raises(AssertionError):
        test_double_quant_worked_example()
    monkeypatch.undo()
    # (3) ties to the upper level
    orig_near = o._nearest
    monkeypatch.setattr(o, "_nearest", lambda v, lv, chunk=1 << 20:
                        (len(lv) - 1 - orig_near(v, np.asarray(lv)[::-1], chunk)).astype(np.uint8))
    with pytest.raises(AssertionError):
        test_encode_equals_midpoint_rule_near_every_threshold()
    monkeypatch.undo()
    # (4) transposed operand in the matmul reference
    monkeypatch.setattr(o, "matmul_ref", lambda xb, wb: (
        o.bf16_bits_to_f32(xb).astype(np.float64)
        @ o.bf16_bits_to_f32(wb).astype(np.float64)[:, ::-1].T, None))
    with pytest.raises(AssertionError):
        test_matmul_ref_against_torch_and_one_hot()
    monkeypatch.undo()
    # (5) the backward reference with the output columns mis-indexed
    # (columns of w_hat reversed)
    monkeypatch.setattr(o, "matmul_dx_ref", lambda db, wb, dtype=0: (
        o.bf16_bits_to_f32(db).astype(np.float64)
        @ o.bf16_bits_to_f32(wb).astype(np.float64)[:, ::-1],
        np.abs(o.bf16_bits_to_f32(db).astype(np.float64))
        @ np.abs(o.bf16_bits_to_f32(wb).astype(np.float64))))
    with pytest.raises(AssertionError):
        test_matmul_dx_ref_brute_force_one_hot_and_adjoint()
    monkeypatch.undo()
    # (6) fp16 rounding by truncation instead of to nearest
    monkeypatch.setattr(o, "f32_to_f16_bits", lambda x: np.asarray(
        [np.float16(np.float32(v)) if abs(np.float16(np.float32(v))) <= abs(v) else
         np.nextafter(np.float16(np.float32(v)), np.float16(0)) for v in np.asarray(x, np.float32)],
        dtype=np.float16).view(np.uint16))
    with pytest.raises(AssertionError):
        test_f16_rounding_matches_brute_force_grid()
    monkeypatch.undo()
    # (7) division replaced by a multiply with the rounded reciprocal
    monkeypatch.setattr(o, "normalize", lambda w, a, blocksize=o.BLOCKSIZE: (
        np.asarray(w, np.float32).reshape(-1, blocksize)
        * (np.float32(1) / np.asarray(a, np.float32).reshape(-1, 1))).astype(np.float32).reshape(-1))
    with pytest.raises(AssertionError):
        test_normalize_is_the_correctly_rounded_quotient()
    monkeypatch.undo()
    # (8) int8 scale codes rounded half away from zero instead of to even
    monkeypatch.setattr(o.np, "rint", lambda v: np.trunc(v + np.copysign(0.5, v)))
    with pytest.raises(AssertionError):
        test_double_quant_rounds_exact_halves_to_even()
    monkeypatch.undo()
    # (9) the code value rounded to bf16 before the scale (double rounding)
    orig_table = o.code_table
    monkeypatch.setattr(o, "code_table", lambda code: torch.from_numpy(orig_table(code)).to(
        torch.bfloat16).float().numpy())
    with pytest.raises(AssertionError):
        test_dequant_single_rounding_with_scales()
    monkeypatch.undo()
