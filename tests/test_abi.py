"""The C-ABI library loads on a machine without a GPU, exports every function
declared in include/nf4q.h, and its host-only calls (sizes, code tables,
argument checks) behave as documented.  No compute call is made."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
from oracle import nf4_oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nf4q.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nf4q_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from dequant_matmul_quantize_b300 import build
    build.build()
    return nq.lib()


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert len(names) >= 13
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def _prototypes():
    """{name: number of parameters} of every function declared in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(nf4q_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_signatures_match_the_header(L):
    """Every function the binding declares has the header's parameter count
    (a drifted binding would pass wrong arguments silently)."""
    protos = _prototypes()
    assert len(protos) == len(_declared_functions())
    for name, n in protos.items():
        f = getattr(L, name)
        if f.argtypes is not None:
            assert len(f.argtypes) == n, (name, len(f.argtypes), n)


def test_header_is_plain_c(tmp_path):
    """include/nf4q.h compiles as C99 and as C++ (no CUDA or torch types)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "use.c"
    src.write_text('#include "nf4q.h"\nint main(void) { nf4q_weight w = {0}; '
                   'nf4q_int8_weight q = {0}; (void)w; (void)q; '
                   'return (int)nf4q_sizes(64, 64, 64, 256, 0, 0, 0); }\n')
    for cmd in ([gcc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only"],
                [shutil.which("g++") or gcc, "-x", "c++", "-std=c++17", "-Wall", "-Werror",
                 "-fsyntax-only"]):
        r = subprocess.run(cmd + ["-I", os.path.dirname(HEADER), str(src)],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_version_and_status_strings(L):
    assert L.nf4q_version() >> 16 == 1
    for s in range(7):
        assert L.nf4q_status_string(s)
    assert L.nf4q_status_string(99) == b"unknown status"


def test_last_cuda_error_is_empty_before_any_failure(L):
    # a fresh thread has no recorded failure; the call itself needs no GPU
    import threading
    out = {}

    def probe():
        buf = ctypes.create_string_buffer(8)
        out["n"] = L.nf4q_last_cuda_error(buf, 8)
        out["text"] = buf.value
        out["n_null"] = L.nf4q_last_cuda_error(None, 0)

    t = threading.Thread(target=probe)
    t.start()
    t.join()
    assert out == {"n": 0, "text": b"", "n_null": 0}


def test_int8_workspace_layout_and_checks(L):
    """Workspace bytes follow the header's layout; bad arguments are refused
    before anything is launched."""
    def a(v):
        return (v + 255) // 256 * 256
    for M, K in [(1, 16), (3, 320), (16, 4096), (40, 8192)]:
        want = a(K) + 256 + a(4 * K) + a(4 * M) + a(2 * M * K)
        assert L.nf4q_int8_workspace_bytes(M, K) == want
    assert L.nf4q_int8_workspace_bytes(-1, 16) == 0
    w = nq.NF4QInt8Weight(None, None, 8, 24)                 # cols % 16 != 0
    assert L.nf4q_int8_quantize_weight(None, nq.IN_F16, ctypes.byref(w), None) == 1
    assert L.nf4q_int8_matmul(ctypes.byref(w), None, 1, 6.0, None, None, 0, None) == 1
    w = nq.NF4QInt8Weight(None, None, 8, 32)
    assert L.nf4q_int8_quantize_weight(None, nq.IN_F32, ctypes.byref(w), None) == 1
    assert L.nf4q_int8_matmul(ctypes.byref(w), None, 0, 6.0, None, None, 0, None) == 0
    assert L.nf4q_int8_matmul(ctypes.byref(w), None, -1, 6.0, None, None, 0, None) == 1
    assert L.nf4q_int8_matmul(ctypes.byref(w), None, 2, 6.0, None, None, 0, None) == 1
    assert L.nf4q_int8_matmul(None, None, 2, 6.0, None, None, 0, None) == 1
    # cols beyond 2^30 would overflow the kernels' int column counters
    w = nq.NF4QInt8Weight(0x1000, 0x2000, 8, (1 << 30) + 16)
    assert L.nf4q_int8_quantize_weight(0x3000, nq.IN_F16, ctypes.byref(w), None) == 3
    assert L.nf4q_int8_matmul(ctypes.byref(w), 0x3000, 1, 6.0, 0x4000, 0x5000, 1 << 40,
                              None) == 3


def test_sizes(L):
    assert nq.sizes(4096, 4096) == (4096 * 4096 // 2, 4096 * 4096 // 64, 1024)
    assert nq.sizes(28672, 8192)[2] == 14336
    assert nq.sizes(3, 64) == (96, 3, 1)          # partial last DQ block
    assert nq.sizes(0, 64) == (0, 0, 0)
    with pytest.raises(nq.Nf4qError):
        nq.sizes(4, 100)                           # cols % 64 != 0
    big = (2 ** 63 - 1) // 64                      # rows * 64 still fits in int64
    assert nq.sizes(big, 64) == (big * 32, big, (big + 255) // 256)
    for rows, cols in ((big + 1, 64), (2 ** 40, 2 ** 40), (2 ** 62, 2 ** 6 * 3)):
        with pytest.raises(nq.Nf4qError, match="UNSUPPORTED"):
            nq.sizes(rows, cols)                   # rows * cols overflows int64


def test_code_values_match_oracle_bit_exact(L):
    """The library builds its tables itself (Newton on erfc); the oracle uses
    scipy's ndtri.  Both must give the same float32 bits."""
    for code, ref in (("nf4", o.nf4_code_table()), ("fp4", o.fp4_code_table())):
        got = np.array(nq.code_values(code), dtype=np.float32)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), code


def test_thresholds_are_round_down_midpoints(L):
    for code in ("nf4", "fp4"):
        t = nq.thresholds(code)
        lv = (o.nf4_code_table() if code == "nf4" else o.FP4_MAGNITUDES.astype(np.float32))
        lv = lv.astype(np.float64)
        mids = (lv[:-1] + lv[1:]) / 2
        assert len(t) == len(mids)
        for ti, m in zip(t, mids):
            f = np.float32(ti)
            assert float(f) <= m < float(np.nextafter(f, np.float32(2)))


def test_argument_checks_launch_nothing(L):
    s = nq.NF4QWeight(None, None, None, None, None, 64, 64, 64, 256, 0, 1, 0)
    bad = nq.NF4QWeight(None, None, None, None, None, 64, 100, 64, 256, 0, 1, 0)
    wrongbs = nq.NF4QWeight(None, None, None, None, None, 64, 64, 128, 256, 0, 1, 0)
    R = ctypes.byref
    assert L.nf4q_quantize(None, 0, R(s), None) == 1
    assert L.nf4q_quantize(None, 0, R(bad), None) == 1
    assert L.nf4q_quantize(None, 0, R(wrongbs), None) == 1
    assert L.nf4q_quantize(16, 7, R(s), None) == 1               # dtype
    assert L.nf4q_double_quant(R(s), None, 0, None) == 1          # no outputs
    assert L.nf4q_dequantize(R(s), None, None) == 1
    assert L.nf4q_gemv(R(s), 16, 0, 16, None) == 3               # M out of range
    assert L.nf4q_gemv(R(s), 16, 17, 16, None) == 3
    assert L.nf4q_gemm(R(s), 16, -1, 16, None) == 1
    assert L.nf4q_gemv(None, 16, 1, 16, None) == 1
    # nf4q_gemv_multi_ex: unknown flag bits, then the group checks
    W1 = (ctypes.POINTER(nq.NF4QWeight) * 1)(ctypes.pointer(s))
    Y1 = (ctypes.c_void_p * 1)(16)
    assert L.nf4q_gemv_multi_ex(W1, 1, 16, 1, Y1, 2, None) == 1
    assert L.nf4q_gemv_multi_ex(W1, 1, 16, 1, Y1, -1, None) == 1
    assert L.nf4q_gemv_multi_ex(W1, 0, 16, 1, Y1, nq.GEMV_WEIGHTS_STATIC, None) == 1
    assert L.nf4q_gemv_multi_ex(W1, 1, 16, 0, Y1, nq.GEMV_WEIGHTS_STATIC, None) == 3
    # an unknown compute dtype is refused by every call on the weight
    dt = nq.NF4QWeight(None, None, None, None, None, 64, 64, 64, 256, 0, 1, 2)
    assert L.nf4q_quantize(16, 1, R(dt), None) == 1
    assert L.nf4q_dequantize(R(dt), 16, None) == 1
    assert L.nf4q_gemv(R(dt), 16, 1, 16, None) == 1
    assert L.nf4q_gemm(R(dt), 16, 64, 16, None) == 1
    # misaligned device pointers are refused before any launch
    sp = nq.NF4QWeight(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 64, 64, 64, 256, 0, 1, 0)
    assert L.nf4q_quantize(0x1008, 1, R(sp), None) == 2
    assert L.nf4q_gemv(R(sp), 0x1004, 1, 0x2000, None) == 2
    # a too-small double-quant workspace
    assert L.nf4q_double_quant(R(sp), 0x6000, 8, None) == 4
    # empty weights are a no-op that succeeds
    e = nq.NF4QWeight(None, None, None, None, None, 0, 64, 64, 256, 0, 1, 0)
    assert L.nf4q_quantize(None, 0, R(e), None) == 0
    assert L.nf4q_dequantize(R(e), None, None) == 0


def test_workspace_size(L):
    assert L.nf4q_double_quant_workspace_bytes(1 << 20) >= 64


def test_binding_rejects_bad_tensors_before_any_call():
    """Host tensors, wrong dtypes and shapes raise ValueError in the binding
    (no GPU needed: nothing reaches the library)."""
    qw = nq.QuantizedWeight(*(torch.empty(0) for _ in range(5)), 4, 64, "nf4", True)
    with pytest.raises(ValueError):
        nq.quantize_into(qw, torch.zeros(4, 64))                     # not on a GPU
    with pytest.raises(ValueError):
        nq.gemv(qw, torch.zeros(1, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        nq.matmul_dx(qw, torch.zeros(3, 4, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        nq.int8_quantize_weight(torch.zeros(4, 64, dtype=torch.float16))
    with pytest.raises(ValueError):
        nq.int8_matmul(nq.Int8Weight(torch.empty(0), torch.empty(0), 4, 64),
                       torch.zeros(1, 64, dtype=torch.float16))


def test_bench_traffic_digest_ignores_comments():
    """bench.py's measured DRAM traffic is tied to the step kernel's code:
    the digest must not move on a comment or blank-space edit, and must move
    on a code edit."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_digest", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    src = "int f(int a) { // the sum\n  return a + 1; /* one\n more */ }\n"
    assert b.code_of(src) == b.code_of("int f(int a) {\n\n   return a + 1;   }")
    assert b.code_of(src) != b.code_of(src.replace("a + 1", "a + 2"))
