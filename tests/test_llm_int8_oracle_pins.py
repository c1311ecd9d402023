"""Pins of the LLM.int8() oracle against things other than itself: exact
rational arithmetic, a worked example whose codes follow by hand, closed
forms, a brute-force triple loop, invariants, and planted mistakes."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import llm_int8_oracle as q8
from oracle import nf4_oracle as o


def _f16(vals):
    return np.asarray(vals, dtype=np.float16).astype(np.float32)


def _rint_half_even(v: Fraction) -> int:
    f = v.numerator // v.denominator
    r = v - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def test_quantize_rows_worked_example():
    """Row 0: s = 12.7 (= 2 * 6.35 exactly in fp16), so 127 * 6.35 / 12.7 =
    63.5 is an exact tie -> the even 64; 3.175 gives 31.75 -> 32.  Row 1:
    s = 127/64, so (2k+1)/128 gives the exact tie k + 1/2: 62.5 -> 62 and
    2.5 -> 2 (half to even, not away from zero)."""
    a = _f16([[6.35, -12.7, 3.175, 0.0],
              [127 / 64, 125 / 128, 5 / 128, -5 / 128]])
    q, s = q8.quantize_rows(a)
    assert s[0] == np.float32(np.float16(12.7)) and s[1] == np.float32(127 / 64)
    assert q.tolist() == [[64, -127, 32, 0], [127, 62, 2, -2]]


def test_quantize_rows_against_exact_rationals():
    g = np.random.default_rng(1)
    a = _f16(g.standard_normal((6, 40)) * np.array([[0.01], [0.5], [1], [3], [20], [1000]]))
    excl = np.zeros(40, bool)
    excl[[3, 17]] = True
    q, s = q8.quantize_rows(a, excl)
    for r in range(a.shape[0]):
        sr = max(abs(Fraction(float(a[r, k]))) for k in range(40) if not excl[k])
        assert Fraction(float(s[r])) == sr
        for k in range(40):
            if excl[k]:
                assert q[r, k] == 0
                continue
            v = o.round_fraction_to_f32(127 * Fraction(float(a[r, k])) / sr)
            assert q[r, k] == _rint_half_even(Fraction(float(v))), (r, k)
    assert np.abs(q).max() == 127


def test_quantize_rows_zero_row_and_small_values():
    a = np.zeros((2, 8), np.float32)
    a[1, :] = _f16([1, -1, 0.5, 0.25, 3, 2, -2, 0])    # s = 3: 127/3 etc.
    q, s = q8.quantize_rows(a)
    assert s[0] == 0 and not q[0].any()
    assert q[1].tolist() == [42, -42, 21, 11, 127, 85, -85, 0]   # 42.33, 21.17, 10.58, 84.67


def test_outlier_threshold_is_strict_and_uses_magnitude():
    x = _f16([[6.0, 6.00390625, 0.0, -7.0, 1.0],
              [0.0, 0.0, 5.99, 0.0, -6.0]])
    assert q8.outlier_columns(x, 6.0).tolist() == [False, True, False, True, False]
    assert not q8.outlier_columns(x, 0.0).any()
    assert q8.outlier_columns(x, 0.5).tolist() == [True, True, True, True, True]


def test_dequantize_rows_against_exact_rationals():
    g = np.random.default_rng(2)
    qv = g.integers(-127, 128, (3, 50)).astype(np.int8)
    s = np.asarray([0.013, 1.7, 250.0], np.float32)
    w = q8.dequantize_rows(qv, s)
    for r in range(3):
        for k in range(50):
            p = o.round_fraction_to_f32(Fraction(int(qv[r, k])) * Fraction(float(s[r])))
            v = o.round_fraction_to_f32(Fraction(float(p)) / 127)
            assert w[r, k] == o.f32_to_f16_bits(np.asarray([v], np.float32))[0]


def test_matmul_no_outliers_closed_form():
    """Integer rows with |x| <= 127 and max 127 quantize to themselves
    (scale 127): y = x . w^T exactly."""
    g = np.random.default_rng(3)
    x = g.integers(-127, 128, (4, 64)).astype(np.float32)
    x[:, 0] = 127
    w = g.integers(-127, 128, (5, 64)).astype(np.float32)
    w[:, 1] = -127
    wq, sw = q8.quantize_rows(_f16(w))
    assert np.array_equal(wq, w.astype(np.int8)) and np.all(sw == 127)
    y, bound, outl, _, _ = q8.matmul_ref(q8.f32_to_f16_bits(x), wq, sw, threshold=0.0)
    assert not outl.any()
    assert np.array_equal(y, x.astype(np.float64) @ w.T.astype(np.float64))
    assert np.array_equal(bound, np.abs(x).astype(np.float64) @ np.abs(w).T.astype(np.float64))


def test_matmul_all_outliers_is_the_fp16_product():
    g = np.random.default_rng(4)
    x = _f16(g.standard_normal((3, 32)))
    w = _f16(g.standard_normal((6, 32)) * 0.1)
    wq, sw = q8.quantize_rows(w)
    w_hat = q8.f16_to_f32(q8.dequantize_rows(wq, sw)).astype(np.float64)
    y, _, outl, xq, _ = q8.matmul_ref(q8.f32_to_f16_bits(x), wq, sw, threshold=1e-6)
    assert outl.all() and not xq.any()
    assert np.allclose(y, x.astype(np.float64) @ w_hat.T, rtol=0, atol=1e-12)


def test_matmul_brute_force_with_one_outlier_column():
    g = np.random.default_rng(5)
    x = _f16(g.standard_normal((2, 8)))
    x[1, 5] = 9.5                                   # column 5 is an outlier
    w = _f16(g.standard_normal((3, 8)) * 0.2)
    wq, sw = q8.quantize_rows(w)
    y, _, outl, xq, sx = q8.matmul_ref(q8.f32_to_f16_bits(x), wq, sw)
    assert outl.tolist() == [k == 5 for k in range(8)]
    w_hat = q8.f16_to_f32(q8.dequantize_rows(wq, sw))
    for m in range(2):
        sm = max(abs(float(x[m, k])) for k in range(8) if k != 5)
        for n in range(3):
            acc = 0
            for k in range(8):
                if k == 5:
                    continue
                v = o.round_fraction_to_f32(127 * Fraction(float(x[m, k])) / Fraction(sm))
                acc += _rint_half_even(Fraction(float(v))) * int(wq[n, k])
            want = acc * sm * float(sw[n]) / 127 ** 2 + float(x[m, 5]) * float(w_hat[n, 5])
            assert abs(y[m, n] - want) <= 1e-12 * max(1.0, abs(want)), (m, n)


def test_matmul_power_of_two_row_scaling():
    """Doubling a row of x doubles its scale and leaves its codes: that row of
    y doubles exactly (no decomposition, so no outlier can appear)."""
    g = np.random.default_rng(6)
    x = _f16(g.standard_normal((3, 48)))
    w = _f16(g.standard_normal((7, 48)) * 0.05)
    wq, sw = q8.quantize_rows(w)
    y1, _, _, _, _ = q8.matmul_ref(q8.f32_to_f16_bits(x), wq, sw, threshold=0.0)
    x2 = x.copy()
    x2[1] *= 2
    y2, _, _, _, _ = q8.matmul_ref(q8.f32_to_f16_bits(x2), wq, sw, threshold=0.0)
    assert np.array_equal(y2[1], 2 * y1[1]) and np.array_equal(y2[[0, 2]], y1[[0, 2]])


def test_tolerance_floor_is_one_fp16_ulp():
    tol = q8.tolerance(np.array([1.0, 1000.0, 0.0]), np.zeros(3))
    assert tol.tolist() == [2.0 ** -10, 0.5, 2.0 ** -24]


def test_pins_catch_planted_mistakes(monkeypatch):
    # (1) threshold taken as >= instead of >
    monkeypatch.setattr(q8, "outlier_columns", lambda x, t=6.0: np.any(
        np.abs(np.asarray(x, np.float32)) >= np.float32(t), axis=0) if t > 0
        else np.zeros(np.asarray(x).shape[1], bool))
    with pytest.raises(AssertionError):
        test_outlier_threshold_is_strict_and_uses_magnitude()
    monkeypatch.undo()
    # (2) rounding half away from zero instead of half to even
    orig = q8.quantize_rows

    def away(a, exclude=None):
        q, s = orig(a, exclude)
        a = np.asarray(a, np.float32)
        quot = (np.float32(127) * a / np.where(s > 0, s, 1)[:, None]).astype(np.float32)
        return np.where(s[:, None] > 0, np.trunc(quot + np.copysign(0.5, quot)), 0).astype(np.int8), s
    monkeypatch.setattr(q8, "quantize_rows", away)
    with pytest.raises(AssertionError):
        test_quantize_rows_worked_example()
    monkeypatch.undo()
    # (3) outlier term dropped from the product
    orig_mm = q8.matmul_ref

    def no_outlier_term(x_bits, wq, sw, threshold=6.0):
        y, b, outl, xq, sx = orig_mm(x_bits, wq, sw, threshold)
        x = q8.f16_to_f32(x_bits).astype(np.float64)
        w_hat = q8.f16_to_f32(q8.dequantize_rows(wq, sw)).astype(np.float64)
        return y - x[:, outl] @ w_hat[:, outl].T, b, outl, xq, sx
    monkeypatch.setattr(q8, "matmul_ref", no_outlier_term)
    with pytest.raises(AssertionError):
        test_matmul_brute_force_with_one_outlier_column()
    monkeypatch.undo()
