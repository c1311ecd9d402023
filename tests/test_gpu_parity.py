"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Quantize, double quant and dequantize are compared bit for bit; GEMV and
GEMM outputs within |y - y_ref| <= 2e-3 * sum|x w_hat| + 1 bf16 ulp of the
fp64 reference on the oracle's own dequantized weights.  Small cases span
several CTAs and ragged tails; the full workload sizes are checked on
sampled rows (each sampled row is recomputed by the oracle from scratch) and
on the complete scale state."""
import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
import synth
from oracle import nf4_oracle as o
from tests._util import (CODE_ID, as_f32, assert_bits_equal, bf16_bits, check_matmul,
                         full_check, gpu_state, oracle_state)

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


def _full_check(w: torch.Tensor, code: str, double_quant=True, what=""):
    """Quantize on the GPU and in the oracle; compare every byte."""
    return full_check(w, code, double_quant, what)


SMALL_SHAPES = [(1, 64), (3, 64), (5, 192), (37, 320), (64, 1024), (129, 4160), (300, 2048)]


@pytest.mark.parametrize("code", ["nf4", "fp4"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_quantize_dequant_small_bit_exact(code, dtype, shape):
    w = synth.normal_weight(*shape, 0.02, seed=hash(shape) % 1000, dtype=dtype,
                            outlier_frac=2e-3)
    _full_check(w, code, True, f"{code} {dtype} {shape}")


@pytest.mark.parametrize("code", ["nf4", "fp4"])
def test_no_double_quant_path(code):
    w = synth.normal_weight(77, 448, 0.02, seed=5)
    qw, w_hat = _full_check(w, code, False, "no-dq")
    x = synth.activations(3, 448, seed=6)
    y = nq.gemv(qw, x.cuda())
    check_matmul(bf16_bits(y), bf16_bits(x), w_hat, "no-dq gemv")


def test_single_fp32_1024_full():
    w, x = synth.single_fp32_1024()
    qw, w_hat = _full_check(w, "nf4", True, "1024x1024 fp32")
    y = nq.gemv(qw, x.cuda())
    check_matmul(bf16_bits(y), bf16_bits(x), w_hat, "1024 gemv")
    # secondary: cuBLAS on the dequantized weight, same tolerance
    y_cublas = torch.matmul(x.cuda(), nq.dequantize(qw).T)
    check_matmul(bf16_bits(y_cublas), bf16_bits(x), w_hat, "cublas")


# ---------------------------------------------------------------- code search
def _threshold_windows(code: str, n_scales: int, half: int, seed: int):
    """Blocks whose elements sweep every float32 within `half` ulps of
    (midpoint * absmax) for every decision midpoint, for many absmax values.
    Element 0 of each block is the absmax itself."""
    rng = np.random.default_rng(seed)
    lv = (o.nf4_code_table() if code == "nf4" else o.FP4_MAGNITUDES.astype(np.float32))
    lv = lv.astype(np.float64)
    mids = (lv[:-1] + lv[1:]) / 2
    if code == "fp4":
        mids = np.concatenate([mids, -mids])
    scales = np.concatenate([
        np.float32([1.0, 0.5, 2.0 ** -20, 3.0]),
        (10.0 ** rng.uniform(-30, 30, n_scales - 4)).astype(np.float32)])
    vals = []
    for a in scales:
        for m in mids:
            c = np.float32(m * float(a))
            b = np.int64(np.abs(c).view(np.uint32))
            win = np.arange(b - half, b + half + 1).astype(np.uint32).view(np.float32)
            win = win if c > 0 else -win
            win = win[np.abs(win) <= a]
            pad = (-win.size) % 63
            win = np.concatenate([win, np.zeros(pad, np.float32)]).reshape(-1, 63)
            blk = np.concatenate([np.full((win.shape[0], 1), a, np.float32), win], axis=1)
            vals.append(blk)
    return np.concatenate(vals).reshape(-1, 64)


@pytest.mark.parametrize("code", ["nf4", "fp4"])
def test_code_search_exact_near_every_threshold(code):
    blocks = _threshold_windows(code, 48, 1536, seed=11 if code == "nf4" else 12)
    nb8 = blocks.shape[0] // 8 * 8
    w = torch.from_numpy(np.ascontiguousarray(blocks[:nb8]).reshape(-1, 512))
    _full_check(w.contiguous(), code, True, f"{code} threshold sweep")


def test_edge_blocks():
    rng = np.random.default_rng(3)
    rows = []
    rows.append(np.zeros(64, np.float32))                               # all zero
    rows.append(np.concatenate([[1e-39], rng.uniform(-1e-39, 1e-39, 63)]))  # denormal absmax
    rows.append(np.concatenate([[2.0 ** -126], rng.uniform(-1, 1, 63) * 2.0 ** -126]))
    rows.append(np.concatenate([[-3e38], rng.uniform(-3e38, 3e38, 63)]))  # huge
    t = o.nf4_code_table().astype(np.float64)
    mids = (t[:-1] + t[1:]) / 2
    ties = [np.float32(m) for m in mids if float(np.float32(m)) == m]
    row = np.zeros(64, np.float32)
    row[0] = 1.0
    row[1:1 + len(ties)] = ties
    rows.append(row)                                                    # exact ties
    row = np.full(64, -0.0, np.float32)
    row[5] = -0.25
    rows.append(row)                                                    # negative absmax elt
    rows.append(np.float32(rng.standard_normal(64)))
    w = torch.from_numpy(np.stack(rows).astype(np.float32).reshape(1, -1))
    for code in ("nf4", "fp4"):
        _full_check(w.contiguous(), code, True, f"edge {code}")


# ---------------------------------------------------------------- double quant
def _dq_direct(absmax: np.ndarray):
    nb = absmax.size
    qw = nq.QuantizedWeight.empty(1, 64 * nb)
    qw.absmax.copy_(torch.from_numpy(absmax))
    nq.double_quant_into(qw)
    torch.cuda.synchronize()
    q, s2, off = o.double_quant(absmax)
    assert_bits_equal(qw.offset.cpu().numpy(), np.array([off], np.float32), "offset")
    assert_bits_equal(qw.scale2.cpu().numpy(), s2, "scale2")
    assert_bits_equal(qw.absmax_q.cpu().numpy(), q, "absmax_q")


@pytest.mark.parametrize("nb", [1, 2, 255, 256, 257, 1000, 65536 + 17])
def test_double_quant_ragged(nb):
    rng = np.random.default_rng(nb)
    _dq_direct(np.abs(rng.standard_normal(nb) * 0.05).astype(np.float32))


def test_double_quant_degenerate_and_wide_range():
    _dq_direct(np.full(777, 0.125, np.float32))                 # scale2 == 0
    _dq_direct(np.zeros(300, np.float32))                         # all zero
    rng = np.random.default_rng(9)
    wide = (10.0 ** rng.uniform(-38, 30, 5000)).astype(np.float32)  # exact re-sum path
    wide[::7] = 0
    _dq_direct(wide)
    _dq_direct(np.concatenate([np.full(3, 1e-45, np.float32), [3e38]]).astype(np.float32))


def _weight_with_absmax(absmax: np.ndarray, seed: int) -> np.ndarray:
    """One row whose 64-blocks have exactly the given absmax values."""
    rng = np.random.default_rng(seed)
    blocks = rng.uniform(-1, 1, (absmax.size, 64)).astype(np.float32)
    blocks *= absmax[:, None]
    blocks[:, 0] = absmax
    return blocks.reshape(1, -1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("code", ["nf4", "fp4"])
def test_quantize_dq_fused_matches_two_calls(code, dtype):
    """nf4q_quantize_dq == nf4q_quantize + nf4q_double_quant, bit for bit,
    including absmax sets that take the exact re-sum path of the mean."""
    rng = np.random.default_rng(5)
    cases = [np.abs(rng.standard_normal(3000) * 0.05).astype(np.float32),
             np.full(700, 0.125, np.float32),
             np.zeros(300, np.float32)]
    wide = (10.0 ** rng.uniform(-30, 30, 4000)).astype(np.float32)
    wide[::7] = 0
    cases.append(wide)
    for i, am in enumerate(cases):
        w = torch.from_numpy(_weight_with_absmax(am, i)).to(dtype).cuda()
        fused = nq.quantize(w, code)                       # the fused entry point
        two = nq.QuantizedWeight.empty(w.shape[0], w.shape[1], code, True, w.device)
        nq.quantize_into(two, w)
        nq.double_quant_into(two)
        torch.cuda.synchronize()
        a, b = gpu_state(fused), gpu_state(two)
        for k in a:
            assert_bits_equal(a[k], b[k], f"{code} case {i} {k}")
        ref = oracle_state(as_f32(w), code)
        for k in ("packed", "absmax", "absmax_q", "scale2", "offset"):
            assert_bits_equal(a[k], ref[k], f"{code} case {i} {k} vs oracle")


def test_double_quant_workspace_is_left_zero_and_reused():
    """The double-quant workspace is zero on entry and every call leaves it
    zero (the CTA that finalizes the mean clears it), so one workspace serves
    successive calls: nf4q_quantize_dq and nf4q_double_quant on one
    workspace, across tensors that take the fixed-point mean and the exact
    re-sum path (absmax outside [2^-32, 2^8)), give the bits of calls that
    each get a fresh workspace, which the oracle checks."""
    rng = np.random.default_rng(11)
    wide = (10.0 ** rng.uniform(-30, 30, 4000)).astype(np.float32)
    wide[::7] = 0
    cases = [np.abs(rng.standard_normal(3000) * 0.05).astype(np.float32), wide,
             np.full(700, 0.125, np.float32), np.abs(rng.standard_normal(20000)).astype(np.float32)]
    ws = nq.dq_workspace(1 << 20)
    for i, am in enumerate(cases * 2):
        w = torch.from_numpy(_weight_with_absmax(am, i)).to(torch.float32).cuda()
        fresh = nq.quantize(w, "nf4")
        reused = nq.quantize(w, "nf4", workspace=ws)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero()) == 0, f"case {i}: workspace left non-zero"
        two = nq.QuantizedWeight.empty(w.shape[0], w.shape[1], "nf4", True, w.device)
        nq.quantize_into(two, w)
        nq.double_quant_into(two, workspace=ws)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero()) == 0, f"case {i}: workspace left non-zero (two calls)"
        a, b, c = gpu_state(fresh), gpu_state(reused), gpu_state(two)
        for k in a:
            assert_bits_equal(b[k], a[k], f"case {i} {k} reused")
            assert_bits_equal(c[k], a[k], f"case {i} {k} two calls")
        if i < len(cases):
            ref = oracle_state(as_f32(w), "nf4")
            for k in ("absmax_q", "scale2", "offset"):
                assert_bits_equal(a[k], ref[k], f"case {i} {k} vs oracle")


def test_quantize_dq_chain_on_one_workspace():
    """Back-to-back nf4q_quantize_dq calls on one stream with no
    synchronisation between them share one workspace: each quantize kernel
    starts (a programmatic dependent launch) while the previous call's
    per-256 pass is still running, and relies on the previous call's last
    CTA having cleared the workspace.  Twelve weights of mixed sizes and
    absmax ranges (including the exact re-sum path), twice round: every
    stored byte equals a call with a fresh workspace of its own."""
    rng = np.random.default_rng(21)
    ws_ = []
    for i in range(12):
        rows, cols = [(96, 1024), (1000, 2048), (17, 64 * 40), (512, 4096)][i % 4]
        w = rng.standard_normal((rows, cols)).astype(np.float32) * (0.02 if i % 3 else 40.0)
        if i % 5 == 0:
            w[:, :64] *= 1e-12  # blocks with absmax below 2^-32
        ws_.append(torch.from_numpy(w).to(torch.bfloat16).cuda())
    fresh = [nq.quantize(w, "nf4") for w in ws_]
    torch.cuda.synchronize()
    want = [gpu_state(q) for q in fresh]
    ws = nq.dq_workspace(1 << 20)
    for _ in range(2):
        got = [nq.quantize(w, "nf4", workspace=ws) for w in ws_]
        torch.cuda.synchronize()
        assert int(ws.count_nonzero()) == 0
        for i, (q, ref) in enumerate(zip(got, want)):
            g = gpu_state(q)
            for k in ref:
                assert_bits_equal(g[k], ref[k], f"chain weight {i} {k}")


@pytest.mark.parametrize("shape", [(40, 64 * 33), (512, 1024)])
def test_dequantize_unaligned_fp32_scales(shape):
    """Without double quantization the fp32 absmax only has to be 4-byte
    aligned; a scale array that is not 16-byte aligned takes the direct-load
    path of the dequantizer and must give the same bits."""
    w = synth.normal_weight(*shape, 0.02, seed=shape[0])
    qw = nq.quantize(w.cuda(), "nf4", double_quant=False)
    ref = nq.dequantize(qw)
    nb = qw.absmax.numel()
    buf = torch.empty(nb + 4, dtype=torch.float32, device=qw.absmax.device)
    moved = buf[1:1 + nb]
    moved.copy_(qw.absmax)
    qw2 = nq.QuantizedWeight(qw.packed, moved, None, None, None, qw.rows, qw.cols, "nf4", False)
    out = nq.dequantize(qw2)
    torch.cuda.synchronize()
    assert_bits_equal(bf16_bits(out).ravel(), bf16_bits(ref).ravel(), "dequant unaligned scales")


# ---------------------------------------------------------------- GEMV
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16])
@pytest.mark.parametrize("shape", [(37, 320), (256, 1024), (129, 4160)])
def test_gemv_small(M, shape):
    w = synth.normal_weight(*shape, 0.02, seed=M * 7 + shape[0], outlier_frac=1e-3)
    qw, w_hat = _full_check(w, "nf4", True, "gemv")
    x = synth.activations(M, shape[1], seed=M)
    y = nq.gemv(qw, x.cuda())
    check_matmul(bf16_bits(y), bf16_bits(x), w_hat, f"gemv M={M} {shape}")
    if M == 1:
        y2 = nq.matmul(qw, x.cuda())
        assert torch.equal(y, y2)


def test_gemv_one_hot_column_is_exact():
    """A one-hot x picks a column of w_hat: bit for bit through the exact
    GEMV, within the matmul tolerance through the block-scale-folded one
    (which multiplies by code * s, not by its bf16 rounding)."""
    w = synth.normal_weight(200, 512, 0.02, seed=2)
    qw, w_hat = _full_check(w, "nf4", True, "onehot")
    for k in (0, 63, 64, 300, 511):
        x = torch.zeros(1, 512, dtype=torch.bfloat16)
        x[0, k] = 1.0
        y = nq.gemv_exact(qw, x.cuda())
        assert np.array_equal(bf16_bits(y)[0], w_hat[:, k])
        check_matmul(bf16_bits(nq.gemv(qw, x.cuda())), bf16_bits(x), w_hat, f"one-hot {k}")


@pytest.mark.parametrize("M", [1, 3, 8, 12, 16])
@pytest.mark.parametrize("shape", [(37, 320), (129, 4160)])
def test_gemv_exact_small(M, shape):
    w = synth.normal_weight(*shape, 0.02, seed=M * 5 + shape[0], outlier_frac=1e-3)
    qw, w_hat = _full_check(w, "nf4", True, "gemv exact")
    x = synth.activations(M, shape[1], seed=M + 40)
    check_matmul(bf16_bits(nq.gemv_exact(qw, x.cuda())), bf16_bits(x), w_hat,
                 f"gemv exact M={M} {shape}")


@pytest.mark.parametrize("M", [4, 7])
def test_gemv_fp4(M):
    w = synth.normal_weight(96, 768, 0.015, seed=21)
    qw, w_hat = _full_check(w, "fp4", True, "fp4 gemv")
    x = synth.activations(M, 768, seed=22)
    check_matmul(bf16_bits(nq.gemv(qw, x.cuda())), bf16_bits(x), w_hat, "fp4 gemv")


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_gemv_fp4_many_rows(M):
    """FP4 with enough rows (19001 > 148 SMs x 4 CTAs x 32 rows) that M = 2..4
    runs on 32-row CTAs: every output against the oracle, ragged last tile."""
    w = synth.normal_weight(19001, 192, 0.015, seed=23)
    qw, w_hat = _full_check(w, "fp4", True, "fp4 many rows")
    x = synth.activations(M, 192, seed=24 + M)
    check_matmul(bf16_bits(nq.gemv(qw, x.cuda())), bf16_bits(x), w_hat, f"fp4 19001 M={M}")


# ---------------------------------------------------------------- full sizes
def _sampled_full_size(w_gpu: torch.Tensor, code: str, xs, n_rows=48, seed=0):
    """Full-size weight: the whole scale state is compared exactly (the
    oracle recomputes absmax from the full weight and double-quantizes it);
    packed codes, w_hat and matmul outputs on sampled rows."""
    N, K = w_gpu.shape
    qw = nq.quantize(w_gpu, code, True)
    torch.cuda.synchronize()
    w_cpu = as_f32(w_gpu)
    absmax = o.absmax_blocks(w_cpu.reshape(-1))
    q, s2, off = o.double_quant(absmax)
    assert_bits_equal(qw.absmax.cpu().numpy(), absmax, "absmax")
    assert_bits_equal(qw.offset.cpu().numpy(), np.array([off], np.float32), "offset")
    assert_bits_equal(qw.scale2.cpu().numpy(), s2, "scale2")
    assert_bits_equal(qw.absmax_q.cpu().numpy(), q, "absmax_q")
    scales = o.block_scales(q, s2, off).reshape(N, K // 64)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(seed).integers(0, N, n_rows)]))
    packed_gpu = qw.packed.view(N, K // 2)[torch.from_numpy(rows).cuda()].cpu().numpy()
    what_rows = []
    for i, r in enumerate(rows):
        p, a = o.quantize(w_cpu[r], CODE_ID[code])
        assert_bits_equal(packed_gpu[i], p, f"packed row {r}")
        what_rows.append(o.dequantize(p, scales[r], CODE_ID[code]))
    what_rows = np.stack(what_rows)
    dq_gpu = nq.dequantize(qw)
    assert_bits_equal(bf16_bits(dq_gpu[torch.from_numpy(rows).cuda()]).reshape(-1),
                      what_rows.reshape(-1), "w_hat rows")
    del dq_gpu
    worst = 0.0
    for x in xs:
        y = nq.matmul(qw, x)
        y_rows = bf16_bits(y[:, torch.from_numpy(rows).cuda()])
        worst = max(worst, check_matmul(y_rows, bf16_bits(x), what_rows,
                                        f"{code} M={x.shape[0]} {N}x{K}"))
    return worst


@pytest.mark.parametrize("index", [0, 1, 2])
def test_llama7b_decode_full_size(index):
    w, x = synth.llama7b_decode(index, device="cuda")
    _sampled_full_size(w, "nf4", [x], seed=index)


@pytest.mark.parametrize("code", ["nf4", "fp4"])
def test_mlp70b_full_size(code):
    w = synth.mlp70b_weight(device="cuda")
    xs = [synth.mlp70b_x(m, device="cuda") for m in (1, 4, 8, 16)]
    _sampled_full_size(w, code, xs, n_rows=24, seed=7)


@pytest.mark.parametrize("layer,mid", [(0, 0), (0, 1), (0, 4), (0, 6), (31, 5)])
def test_llama3_stack_matrices(layer, mid):
    w = synth.llama3_8b_matrix(layer, mid, device="cuda")
    x = synth.llama3_8b_x(layer, mid, device="cuda")
    _sampled_full_size(w, "nf4", [x], n_rows=16, seed=layer * 10 + mid)


def test_beyond_2_31_elements():
    """A 32768 x 65536 weight (2^31 elements, 4 GB bf16): every index above
    2^31 must be 64-bit.  Codes and absmax of sampled rows against the oracle;
    their dequantized rows against the oracle's formula on the GPU's stored
    scales; the GEMV on those rows within the matmul tolerance."""
    N, K = 32768, 65536
    w = synth.normal_weight(N, K, 0.02, seed=77, device="cuda")
    qw = nq.quantize(w)
    x = synth.activations(1, K, seed=78, device="cuda")
    y = nq.gemv(qw, x)
    torch.cuda.synchronize()
    kb = K // 64
    rows = np.unique(np.concatenate([[0, 1, N // 2, N - 1],
                                     np.random.default_rng(79).integers(0, N, 8)]))
    idx = torch.from_numpy(rows).cuda()
    packed = qw.packed.view(N, K // 2)[idx].cpu().numpy()
    absmax = qw.absmax.view(N, kb)[idx].cpu().numpy()
    aq = qw.absmax_q.view(N, kb)[idx].cpu().numpy()
    s2 = qw.scale2.cpu().numpy()
    off = np.float32(qw.offset.cpu().numpy()[0])
    w_rows = as_f32(w[idx])
    del w
    what = []
    for i, r in enumerate(rows):
        p_ref, a_ref = o.quantize(w_rows[i])
        assert_bits_equal(packed[i], p_ref, f"packed row {r}")
        assert_bits_equal(absmax[i], a_ref, f"absmax row {r}")
        b = np.arange(kb, dtype=np.int64) + int(r) * kb      # global block indices
        sc = o.fma_f32(aq[i].astype(np.float32), s2[b // 256], off)
        what.append(o.dequantize(p_ref, sc))
    what = np.stack(what)
    dq = nq.dequantize(qw)
    assert_bits_equal(bf16_bits(dq[idx]).reshape(-1), what.reshape(-1), "w_hat rows")
    del dq
    check_matmul(bf16_bits(y[:, idx]), bf16_bits(x), what, "gemv 32768x65536")


# ---------------------------------------------------------------- errors
def test_bad_arguments_leave_gpu_usable():
    w = synth.normal_weight(64, 256, 0.02, seed=1).cuda()
    qw = nq.quantize(w)
    s = qw.struct()
    L = nq.lib()
    import ctypes
    stream = torch.cuda.current_stream().cuda_stream
    assert L.nf4q_gemv(ctypes.byref(s), w.data_ptr() + 2, 1, w.data_ptr(), stream) == 2
    assert L.nf4q_gemv(ctypes.byref(s), w.data_ptr(), 40, w.data_ptr(), stream) == 3
    ws = nq.dq_workspace(4)
    assert L.nf4q_double_quant(ctypes.byref(s), ws.data_ptr(), 4, stream) == 4
    x = synth.activations(1, 256, seed=3).cuda()
    y = nq.gemv(qw, x)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()


@pytest.mark.parametrize("op", ["quantize", "dequantize", "gemv1", "gemv9", "gemm"])
def test_first_call_on_a_fresh_host_thread(op):
    """Each entry point works as the FIRST library call on a new host thread
    (autograd runs backward on such a thread, where no CUDA context need be
    current): the same bytes / outputs as on the main thread."""
    import threading
    w = synth.normal_weight(160, 256, 0.02, seed=21).cuda()
    qw = nq.quantize(w)
    xs = {"gemv1": synth.activations(1, 256, seed=22).cuda(),
          "gemv9": synth.activations(9, 256, seed=23).cuda(),
          "gemm": synth.activations(80, 256, seed=24).cuda()}

    def run():
        if op == "quantize":
            q = nq.quantize(w)
            return (q.packed, q.absmax_q, q.scale2, q.offset)
        if op == "dequantize":
            return (nq.dequantize(qw),)
        return (nq.matmul(qw, xs[op]),)

    main = run()
    torch.cuda.synchronize()
    out, err = {}, []

    def worker():
        try:
            out["r"] = run()
            torch.cuda.synchronize()
        except Exception as e:      # noqa: BLE001 - reported below
            err.append(e)

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert not err, err
    for a, b in zip(main, out["r"]):
        assert torch.equal(a, b)
