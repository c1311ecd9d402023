"""The block-scale-folded GEMV against the oracle.  nf4q_gemv takes it for
M <= 6; nf4q_gemv_multi (here with a single weight) for M <= 8, which is
how the tests reach it at every M.

The folded kernel multiplies x by code_value * s_b (code values rounded to
fp16) instead of by w_hat = bf16(code_value * s_b); it is held to the same
tolerance as every matmul here, |y - y_ref| <= 2e-3 * sum|x w_hat| + one ulp
of y_ref, with y_ref the fp64 product of x and the ORACLE's w_hat.

The launch gives each CTA a contiguous range of 16-row tiles and cuts the
CTA's boxes (16 rows x 8 or 4 blocks) into equal runs over its 16 warps; a
tile whose boxes fall to several warps is summed by the last to arrive.
Shapes cover every regime of that split on a 148-SM B300: fewer boxes than
warps, one tile per CTA split over all 16 warps, runs that cross tile
boundaries (with and without 16-block scale chunks), and group launches
whose CTA ranges cross from one weight to the next; with ragged row tiles
and a K that is not a multiple of the 256-column boxes.  The error analysis of the fold is checked
on its own inputs: random activations, activations whose signs follow the
rounding of w_hat (the sign-adversarial case, inside the tolerance because
the mean relative bf16 rounding error is below 2e-3), and activations that
also sit only on the weights with the largest rounding error (bounded by the
per-term analytic bound 2^-8 + 2^-11, which exceeds the tolerance)."""
import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
import synth
from oracle import nf4_oracle as o
from tests._util import CODE_ID, bf16_bits, check_matmul, full_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_matmul_quantize_b300 import build
    build.build()
    nq.lib()
    yield
    torch.cuda.synchronize()
    assert nq.device_error() == 0


def folded(qw, x):
    """The folded kernel for any M <= 8: a one-weight group."""
    return nq.gemv_multi([qw], x)[0]


# (rows, cols): (37, 320) 3 CTAs of one box; (256, 1024) 16 CTAs, 4 boxes
# each; (129, 4160) 9 CTAs, one tile of 17 boxes over 16 warps; (4000, 256)
# 250 tiles of one box, 1-2 per CTA; (2400, 1024) 150 tiles, 1-2 per CTA;
# (700, 2112) 44 tiles of 5 boxes
SHAPES = [(37, 320), (256, 1024), (129, 4160), (4000, 256), (2400, 1024), (700, 2112)]


@pytest.mark.parametrize("code", ["nf4", "fp4"])
@pytest.mark.parametrize("M", [1, 2, 5, 8])
@pytest.mark.parametrize("shape", SHAPES)
def test_folded_gemv_parity(code, M, shape):
    w = synth.normal_weight(*shape, 0.02, seed=shape[0] + M, outlier_frac=1e-3)
    qw, w_hat = full_check(w, code, True, f"{code} {shape}")
    x = synth.activations(M, shape[1], seed=100 + M)
    y = folded(qw, x.cuda())
    check_matmul(bf16_bits(y), bf16_bits(x), w_hat, f"folded {code} M={M} {shape}")


@pytest.mark.parametrize("M", [1, 6])
def test_folded_gemv_fp16_and_no_double_quant(M):
    w = synth.normal_weight(300, 1088, 0.02, seed=7)
    # fp16 compute dtype (the stored state is the same; w_hat is fp16)
    qw = nq.quantize(w.cuda(), "nf4", True, compute_dtype="f16")
    ref = full_check(w, "nf4", True, "fp16 state")[0]
    assert torch.equal(qw.packed, ref.packed)
    st = o.quantize_full(w.float().numpy().reshape(-1), o.CODE_NF4)
    scales = o.block_scales(st["absmax_q"], st["scale2"], st["offset"])
    w_hat16 = o.dequantize(st["packed"], scales, o.CODE_NF4, dtype=o.DT_F16).reshape(300, 1088)
    x = synth.activations(M, 1088, seed=8).to(torch.float16)
    y = folded(qw, x.cuda())
    check_matmul(y.cpu().view(torch.int16).numpy().view(np.uint16),
                 x.view(torch.int16).numpy().view(np.uint16), w_hat16, "folded fp16", o.DT_F16)
    # no double quantization: the fp32 absmax is the scale
    qn, w_hat_n = full_check(w, "fp4", False, "no-dq")
    xb = synth.activations(M, 1088, seed=9)
    check_matmul(bf16_bits(folded(qn, xb.cuda())), bf16_bits(xb), w_hat_n, "folded no-dq")


def test_folded_gemv_rows_of_x_far_apart_in_magnitude():
    """Each row of x gets its own power-of-two scaling before it becomes
    fp16: rows at 2^-100 .. 2^100, an all-zero row, and a row whose values
    span 2^-30 .. 2^0 are all inside the tolerance."""
    K = 1024
    w = synth.normal_weight(200, K, 0.02, seed=11)
    qw, w_hat = full_check(w, "nf4", True, "x scales")
    base = synth.activations(7, K, seed=12).float()
    scale = torch.tensor([2.0 ** -100, 2.0 ** -20, 1.0, 2.0 ** 20, 2.0 ** 100, 0.0, 1.0])
    x = base * scale[:, None]
    g = torch.Generator().manual_seed(13)
    x[6] = x[6] * torch.exp2(-30.0 * torch.rand(K, generator=g))
    x = x.to(torch.bfloat16)
    y = folded(qw, x.cuda())
    assert torch.all(y[5] == 0)
    check_matmul(bf16_bits(y), bf16_bits(x), w_hat, "x row scales")


def test_folded_gemv_is_deterministic_and_near_the_exact_kernel():
    w = synth.normal_weight(1500, 2048, 0.02, seed=14, outlier_frac=1e-3)
    qw, w_hat = full_check(w, "nf4", True, "determinism")
    x = synth.activations(3, 2048, seed=15).cuda()
    y1 = folded(qw, x)
    y2 = folded(qw, x)
    assert torch.equal(y1, y2)
    ye = nq.gemv_exact(qw, x)
    check_matmul(bf16_bits(y1), bf16_bits(x), w_hat, "folded")
    check_matmul(bf16_bits(ye), bf16_bits(x), w_hat, "exact")


def _fold_error_terms(w_hat_bits, scales, packed, code):
    """Per weight: the value the folded kernel multiplies x by, fp16(code)
    * s (exact in fp64), and w_hat; both [N, K] float64."""
    idx = o.unpack_nibbles(packed)
    c16 = o.code_table(code).astype(np.float16).astype(np.float64)
    s = np.repeat(np.asarray(scales, np.float64), 64)
    folded = (c16[idx] * s).reshape(w_hat_bits.shape)
    return folded, o.bf16_bits_to_f32(w_hat_bits).astype(np.float64)


@pytest.mark.parametrize("code", ["nf4", "fp4"])
def test_folded_gemv_error_analysis(code):
    N, K = 512, 4096
    w = synth.normal_weight(N, K, 0.02, seed=16)
    qw, w_hat = full_check(w, code, True, "error analysis")
    st = o.quantize_full(w.float().numpy().reshape(-1), CODE_ID[code])
    scales = o.block_scales(st["absmax_q"], st["scale2"], st["offset"])
    folded, what = _fold_error_terms(w_hat, scales, st["packed"], CODE_ID[code])
    delta = folded - what

    # random activations: far inside the tolerance
    x = synth.activations(1, K, seed=17)
    worst_random = check_matmul(bf16_bits(nq.gemv(qw, x.cuda())), bf16_bits(x), w_hat,
                                "random x")
    assert worst_random < 0.2

    # signs of x follow the rounding of w_hat of row 0, |x| = 1
    xs = np.where(delta[0] >= 0, 1.0, -1.0).astype(np.float32)[None, :]
    xt = torch.from_numpy(xs).to(torch.bfloat16)
    y = nq.gemv(qw, xt.cuda())
    worst_sign = check_matmul(bf16_bits(y[:, :1]), bf16_bits(xt), w_hat[:1], "sign-adversarial")
    assert worst_sign < 1.0

    # x only on the weights of row 0 whose relative rounding error exceeds
    # 3e-3, signs aligned: beyond the 2e-3 tolerance by construction, but
    # within the per-term bound (2^-8 + 2^-11) * sum|x w_hat| + one ulp
    rel = np.abs(delta[0]) / np.maximum(np.abs(what[0]), 1e-300)
    sel = (rel > 3e-3) & (what[0] != 0)
    assert sel.sum() > 20
    xa = np.where(sel, np.sign(delta[0]), 0.0).astype(np.float32)[None, :]
    xat = torch.from_numpy(xa).to(torch.bfloat16)
    ya = nq.gemv(qw, xat.cuda()).float().cpu().numpy()[0, 0]
    y_ref, bound = o.matmul_ref(bf16_bits(xat), w_hat[:1])
    err = abs(ya - y_ref[0, 0])
    analytic = (2.0 ** -8 + 2.0 ** -11 + 2.0 ** -20) * bound[0, 0] + o.ulp_bf16(y_ref[0, 0])
    assert err <= analytic, (err, analytic)


# Larger splits (148 CTAs): (1600, 8192) one tile per CTA, 16 boxes, one per
# warp; (1600, 16384) 4-block boxes at M = 1 (x past the 8-block layout's
# room), 64 boxes per tile, 4 per warp; (7104, 3584) three tiles of 7 boxes
# per CTA, runs of 1-2 boxes crossing tiles, scales without chunks (K/64 =
# 56); (7104, 5120) the same with chunked scales (K/64 = 80, 10 boxes).
SPLITS = [(1600, 8192), (1600, 16384), (7104, 3584), (7104, 5120)]


@pytest.mark.parametrize("shape", SPLITS)
def test_folded_gemv_work_splits(shape):
    w = synth.normal_weight(*shape, 0.02, seed=shape[0] + shape[1], outlier_frac=1e-3)
    qw, w_hat = full_check(w, "nf4", True, f"split {shape}")
    for M in (1, 2):
        x = synth.activations(M, shape[1], seed=200 + M)
        y = folded(qw, x.cuda())
        check_matmul(bf16_bits(y), bf16_bits(x), w_hat, f"folded M={M} {shape}")


def test_grouped_gemv_ranges_cross_weights():
    """A group of 300 + 144 tiles (K = 5120): three tiles per CTA, so one
    CTA's range and some warps' runs start in the first weight and end in
    the second."""
    shapes = [(4800, 5120), (2304, 5120)]
    ws = [synth.normal_weight(n, k, 0.02, seed=80 + i) for i, (n, k) in enumerate(shapes)]
    checked = [full_check(w, "nf4", True, f"cross {i}") for i, w in enumerate(ws)]
    for M in (1, 2):
        x = synth.activations(M, 5120, seed=83 + M)
        ys = nq.gemv_multi([q for q, _ in checked], x.cuda())
        for (qw, w_hat), y in zip(checked, ys):
            check_matmul(bf16_bits(y), bf16_bits(x), w_hat, f"cross M={M}")


def test_static_weights_flag_changes_nothing_but_the_load_order():
    """nf4q_gemv_multi_ex with NF4Q_GEMV_WEIGHTS_STATIC loads the first
    weight tiles and scales before waiting for the preceding kernel; the
    results are the flag-free call's, bit for bit, in every regime of the
    kernel (3-D and 2-D weight views, chunked and per-box scales, no double
    quant, FP4, fp16, M = 1..6, groups), also when each launch directly
    follows another GEMV on the stream (so that it overlaps its tail), and
    they pass the oracle check."""
    cases = [([(4800, 5120), (2304, 5120)], "nf4", True, "bf16"),
             ([(4096, 4096), (1024, 4096), (1024, 4096)], "nf4", True, "bf16"),
             ([(700, 2112)], "nf4", True, "bf16"),
             ([(1000, 1024)], "nf4", False, "bf16"),
             ([(1500, 3072)], "fp4", True, "bf16"),
             ([(1200, 2048)], "nf4", True, "f16")]
    for i, (shapes, code, dq, cdt) in enumerate(cases):
        K = shapes[0][1]
        ws = [synth.normal_weight(n, k, 0.02, seed=120 + 7 * i + j)
              for j, (n, k) in enumerate(shapes)]
        qws = [nq.quantize(w.cuda(), code, dq, compute_dtype=cdt) for w in ws]
        for M in (1, 2, 6):
            x = synth.activations(M, K, seed=140 + M + i)
            x = x.to(torch.float16).cuda() if cdt == "f16" else x.cuda()
            want = nq.gemv_multi(qws, x)
            # back to back on one stream: each launch follows a GEMV
            outs = [nq.gemv_multi(qws, x, static_weights=True) for _ in range(3)]
            torch.cuda.synchronize()
            for got in outs:
                for a, b in zip(got, want):
                    assert torch.equal(a, b), (shapes, code, dq, cdt, M)
    shapes = [(4800, 5120), (2304, 5120)]
    ws = [synth.normal_weight(n, k, 0.02, seed=80 + i) for i, (n, k) in enumerate(shapes)]
    checked = [full_check(w, "nf4", True, f"static {i}") for i, w in enumerate(ws)]
    x = synth.activations(1, 5120, seed=84)
    ys = nq.gemv_multi([q for q, _ in checked], x.cuda(), static_weights=True)
    for (qw, w_hat), y in zip(checked, ys):
        check_matmul(bf16_bits(y), bf16_bits(x), w_hat, "static M=1")


def test_gemv_dispatch_by_m():
    """nf4q_gemv: the folded kernel for M <= 6 when x fits its staging room
    (M * K <= 30720 here), the exact one above."""
    w = synth.normal_weight(300, 1024, 0.02, seed=31)
    qw = nq.quantize(w.cuda())
    for M in (1, 2, 3, 6, 7, 8, 16):
        x = synth.activations(M, 1024, seed=32 + M).cuda()
        want = folded(qw, x) if M <= 6 else nq.gemv_exact(qw, x)
        assert torch.equal(nq.gemv(qw, x), want), M
    # x past the staging room (4 x 16384 > 30720): the exact kernel
    w = synth.normal_weight(64, 16384, 0.02, seed=39)
    qw = nq.quantize(w.cuda())
    x = synth.activations(4, 16384, seed=40).cuda()
    assert torch.equal(nq.gemv(qw, x), nq.gemv_exact(qw, x))


def test_grouped_gemv_matches_the_oracle_per_weight():
    """nf4q_gemv_multi: three weights sharing x (q, k, v shaped, rows not
    multiples of 16) in one launch; every output against the oracle, and
    each equal to its own nf4q_gemv within the tolerance."""
    shapes = [(300, 1024), (70, 1024), (64, 1024)]
    ws = [synth.normal_weight(n, k, 0.02, seed=60 + i) for i, (n, k) in enumerate(shapes)]
    checked = [full_check(w, "nf4", True, f"group {i}") for i, w in enumerate(ws)]
    for M in (1, 3):
        x = synth.activations(M, 1024, seed=63 + M)
        ys = nq.gemv_multi([q for q, _ in checked], x.cuda())
        for (qw, w_hat), y in zip(checked, ys):
            assert y.shape == (M, qw.rows)
            check_matmul(bf16_bits(y), bf16_bits(x), w_hat, f"grouped M={M}")
            check_matmul(bf16_bits(nq.gemv(qw, x.cuda())), bf16_bits(x), w_hat, "single")


def test_grouped_gemv_refuses_mixed_groups():
    a = nq.quantize(synth.normal_weight(64, 256, 0.02, seed=70).cuda())
    b = nq.quantize(synth.normal_weight(64, 320, 0.02, seed=71).cuda())
    c = nq.quantize(synth.normal_weight(64, 256, 0.02, seed=72).cuda(), "fp4")
    x = synth.activations(1, 256, seed=73).cuda()
    with pytest.raises(nq.Nf4qError):          # codes differ: refused by the C ABI
        nq.gemv_multi([a, c], x)
    with pytest.raises(ValueError):            # columns differ: refused by the binding
        nq.gemv_multi([a, b], x)
    with pytest.raises(ValueError):
        nq.gemv_multi([a] * 5, x)
