"""nf4q: NF4 / FP4 blockwise quantization with double quantization and the
"4-bit stored, 16-bit computed" matmul, as hand-written CUDA for B300.

This module is a thin ctypes binding over ``libnf4q.so`` (the C ABI declared
in ``include/nf4q.h``): it marshals torch tensors' device pointers and the
current CUDA stream, nothing else.  Every step runs in the library's kernels.
There is no CPU or PyTorch fallback: if the library is missing the import of
the first op raises.

The user-facing knobs mirror ``BitsAndBytesConfig`` as the bitsandbytes
pages describe it (tutorial at mlqm.cn/news/394670, section 四): the 4-bit
type ``nf4`` or ``fp4``, ``double_quant`` on or off, and the compute dtype,
which is bf16 (or fp16) here.  The LLM.int8() path (``int8_*``) quantizes
fp16 weights and activations to int8 vector-wise and runs the
mixed-precision decomposition matmul.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnf4q.so")

CODES = {"nf4": 0, "fp4": 1}
IN_F32, IN_BF16, IN_F16 = 0, 1, 2
DTYPES = {"bf16": 0, "f16": 1}          # compute dtype codes of nf4q_weight
BLOCKSIZE, DQ_BLOCKSIZE = 64, 256
GEMV_MAX_M = 16
GEMV_WEIGHTS_STATIC = 1                  # nf4q_gemv_multi_ex flag (nf4q.h)

STATUS = {
    0: "NF4Q_OK", 1: "NF4Q_ERR_INVALID_ARG", 2: "NF4Q_ERR_ALIGNMENT",
    3: "NF4Q_ERR_UNSUPPORTED", 4: "NF4Q_ERR_WORKSPACE", 5: "NF4Q_ERR_CUDA",
    6: "NF4Q_ERR_TIMEOUT",
}


class Nf4qError(RuntimeError):
    def __init__(self, func: str, status: int, detail: str = ""):
        self.status = status
        self.detail = detail
        msg = f"{func} failed: {STATUS.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


def last_cuda_error() -> str:
    """Text of the last failing CUDA call of the library on this thread."""
    L = lib()
    n = L.nf4q_last_cuda_error(None, 0)
    buf = ctypes.create_string_buffer(n + 1)
    L.nf4q_last_cuda_error(buf, n + 1)
    return buf.value.decode(errors="replace")


class NF4QWeight(ctypes.Structure):
    """Mirror of ``nf4q_weight`` in include/nf4q.h."""
    _fields_ = [
        ("packed", ctypes.c_void_p),
        ("absmax_q", ctypes.c_void_p),
        ("absmax", ctypes.c_void_p),
        ("scale2", ctypes.c_void_p),
        ("offset", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("blocksize", ctypes.c_int32),
        ("dq_blocksize", ctypes.c_int32),
        ("code", ctypes.c_int32),
        ("double_quant", ctypes.c_int32),
        ("compute_dtype", ctypes.c_int32),
    ]


class NF4QInt8Weight(ctypes.Structure):
    """Mirror of ``nf4q_int8_weight`` in include/nf4q.h."""
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("scale", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libnf4q.so (built in-tree); raise if it is not there."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m dequant_matmul_quantize_b300.build` (no fallback exists)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    W = ctypes.POINTER(NF4QWeight)
    sig = {
        "nf4q_version": (i32, []),
        "nf4q_status_string": (ctypes.c_char_p, [i32]),
        "nf4q_last_cuda_error": (i32, [ctypes.c_char_p, i32]),
        "nf4q_sizes": (i32, [i64, i64, i32, i32, ctypes.POINTER(sz),
                             ctypes.POINTER(i64), ctypes.POINTER(i64)]),
        "nf4q_code_values": (i32, [i32, ctypes.POINTER(ctypes.c_float)]),
        "nf4q_thresholds": (i32, [i32, ctypes.POINTER(ctypes.c_float),
                                  ctypes.POINTER(i32)]),
        "nf4q_quantize": (i32, [vp, i32, W, vp]),
        "nf4q_double_quant_workspace_bytes": (sz, [i64]),
        "nf4q_double_quant": (i32, [W, vp, sz, vp]),
        "nf4q_quantize_dq": (i32, [vp, i32, W, vp, sz, vp]),
        "nf4q_dequantize": (i32, [W, vp, vp]),
        "nf4q_gemv": (i32, [W, vp, i32, vp, vp]),
        "nf4q_gemv_exact": (i32, [W, vp, i32, vp, vp]),
        "nf4q_gemv_multi": (i32, [ctypes.POINTER(W), i32, vp, i32,
                                  ctypes.POINTER(vp), vp]),
        "nf4q_gemv_multi_ex": (i32, [ctypes.POINTER(W), i32, vp, i32,
                                     ctypes.POINTER(vp), i32, vp]),
        "nf4q_gemm": (i32, [W, vp, i64, vp, vp]),
        "nf4q_matmul": (i32, [W, vp, i64, vp, vp]),
        "nf4q_matmul_dx": (i32, [W, vp, i64, i64, vp, vp]),
        "nf4q_device_error": (i32, [ctypes.POINTER(ctypes.c_uint32), i32]),
        "nf4q_double_quant_noalloc": (i32, [W, vp]),
        "nf4q_int8_quantize_weight": (i32, [vp, i32, ctypes.POINTER(NF4QInt8Weight), vp]),
        "nf4q_int8_workspace_bytes": (sz, [i64, i64]),
        "nf4q_int8_matmul": (i32, [ctypes.POINTER(NF4QInt8Weight), vp, i64, ctypes.c_float, vp,
                                   vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


_IN_DTYPES = {torch.float32: IN_F32, torch.bfloat16: IN_BF16, torch.float16: IN_F16}


def _require(cond: bool, what: str):
    """Argument check of the binding (raised even under python -O)."""
    if not cond:
        raise ValueError(what)


def _check(func: str, status: int):
    if status != 0:
        raise Nf4qError(func, status, last_cuda_error() if status == 5 else "")


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


# ------------------------------------------------------------------ host-only
def sizes(rows: int, cols: int):
    """(packed_bytes, n_b, n_d) of a [rows x cols] weight."""
    pb, nb, nd = ctypes.c_size_t(), ctypes.c_int64(), ctypes.c_int64()
    _check("nf4q_sizes", lib().nf4q_sizes(rows, cols, BLOCKSIZE, DQ_BLOCKSIZE,
                                          ctypes.byref(pb), ctypes.byref(nb),
                                          ctypes.byref(nd)))
    return pb.value, nb.value, nd.value


def code_values(code: str = "nf4"):
    out = (ctypes.c_float * 16)()
    _check("nf4q_code_values", lib().nf4q_code_values(CODES[code], out))
    return list(out)


def thresholds(code: str = "nf4"):
    out = (ctypes.c_float * 15)()
    n = ctypes.c_int32()
    _check("nf4q_thresholds", lib().nf4q_thresholds(CODES[code], out, ctypes.byref(n)))
    return list(out)[: n.value]


# ------------------------------------------------------------------ state
@dataclass
class QuantizedWeight:
    """Device buffers of one quantized weight (see the layout in nf4q.h)."""
    packed: torch.Tensor
    absmax: torch.Tensor
    absmax_q: Optional[torch.Tensor]
    scale2: Optional[torch.Tensor]
    offset: Optional[torch.Tensor]
    rows: int
    cols: int
    code: str = "nf4"
    double_quant: bool = True
    compute_dtype: str = "bf16"

    def struct(self) -> NF4QWeight:
        return NF4QWeight(_ptr(self.packed), _ptr(self.absmax_q), _ptr(self.absmax),
                          _ptr(self.scale2), _ptr(self.offset), self.rows, self.cols,
                          BLOCKSIZE, DQ_BLOCKSIZE, CODES[self.code],
                          1 if self.double_quant else 0, DTYPES[self.compute_dtype])

    @property
    def torch_dtype(self):
        """torch dtype of the dequantized weights, x and y."""
        return torch.bfloat16 if self.compute_dtype == "bf16" else torch.float16

    @staticmethod
    def empty(rows: int, cols: int, code: str = "nf4", double_quant: bool = True,
              device=None, compute_dtype: str = "bf16") -> "QuantizedWeight":
        device = device or torch.device("cuda", torch.cuda.current_device())
        pb, nb, nd = sizes(rows, cols)
        u8 = dict(dtype=torch.uint8, device=device)
        return QuantizedWeight(
            packed=torch.empty(max(pb, 1), **u8)[:pb],
            absmax=torch.empty(max(nb, 1), dtype=torch.float32, device=device)[:nb],
            absmax_q=torch.empty(max(nb, 1), dtype=torch.int8, device=device)[:nb],
            scale2=torch.empty(max(nd, 1), dtype=torch.float32, device=device)[:nd],
            offset=torch.empty(1, dtype=torch.float32, device=device),
            rows=rows, cols=cols, code=code, double_quant=double_quant,
            compute_dtype=compute_dtype)


# ------------------------------------------------------------------ ops
def quantize_into(qw: QuantizedWeight, w: torch.Tensor, stream=None):
    """nf4q_quantize: writes qw.packed and qw.absmax from w (fp32, bf16 or fp16)."""
    _require(w.is_cuda and w.is_contiguous() and tuple(w.shape) == (qw.rows, qw.cols),
             "w must be a contiguous CUDA tensor of the weight's shape")
    _require(w.dtype in _IN_DTYPES, "w must be fp32, bf16 or fp16")
    dt = _IN_DTYPES[w.dtype]
    s = qw.struct()
    _check("nf4q_quantize", lib().nf4q_quantize(_ptr(w), dt, ctypes.byref(s), _stream(stream)))


def dq_workspace(n_b: int, device=None) -> torch.Tensor:
    """A zero-filled double-quant workspace (every call leaves it zero, so
    it may be reused by successive calls on one stream)."""
    nbytes = lib().nf4q_double_quant_workspace_bytes(n_b)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def double_quant_into(qw: QuantizedWeight, workspace: Optional[torch.Tensor] = None,
                      stream=None):
    """nf4q_double_quant: writes qw.absmax_q, qw.scale2, qw.offset from qw.absmax."""
    if workspace is None:
        workspace = dq_workspace(qw.absmax.numel(), qw.absmax.device)
    s = qw.struct()
    _check("nf4q_double_quant", lib().nf4q_double_quant(
        ctypes.byref(s), _ptr(workspace), workspace.numel(), _stream(stream)))


def quantize_dq_into(qw: QuantizedWeight, w: torch.Tensor,
                     workspace: Optional[torch.Tensor] = None, stream=None):
    """nf4q_quantize_dq: quantize and double-quantize w into qw in one call."""
    _require(w.is_cuda and w.is_contiguous() and tuple(w.shape) == (qw.rows, qw.cols),
             "w must be a contiguous CUDA tensor of the weight's shape")
    _require(w.dtype in _IN_DTYPES, "w must be fp32, bf16 or fp16")
    dt = _IN_DTYPES[w.dtype]
    if workspace is None:
        workspace = dq_workspace(qw.absmax.numel(), qw.absmax.device)
    s = qw.struct()
    _check("nf4q_quantize_dq", lib().nf4q_quantize_dq(
        _ptr(w), dt, ctypes.byref(s), _ptr(workspace), workspace.numel(), _stream(stream)))


def quantize(w: torch.Tensor, code: str = "nf4", double_quant: bool = True,
             workspace: Optional[torch.Tensor] = None, stream=None,
             compute_dtype: str = "bf16") -> QuantizedWeight:
    """Quantize a [rows x cols] fp32/bf16/fp16 CUDA weight (cols % 64 == 0);
    `compute_dtype` ("bf16" or "f16") is the dtype it will be dequantized and
    multiplied in."""
    rows, cols = w.shape
    qw = QuantizedWeight.empty(rows, cols, code, double_quant, w.device, compute_dtype)
    if double_quant:
        quantize_dq_into(qw, w, workspace, stream)
    else:
        quantize_into(qw, w, stream)
    return qw


def dequantize(qw: QuantizedWeight, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(qw.rows, qw.cols, dtype=qw.torch_dtype, device=qw.packed.device)
    s = qw.struct()
    _check("nf4q_dequantize", lib().nf4q_dequantize(ctypes.byref(s), _ptr(out), _stream(stream)))
    return out


def _mm(name: str, qw: QuantizedWeight, x: torch.Tensor, out, stream):
    _require(x.is_cuda and x.dtype == qw.torch_dtype and x.is_contiguous() and x.dim() == 2,
             "x must be a contiguous 2-D CUDA tensor of the compute dtype")
    _require(x.shape[-1] == qw.cols, "x must have the weight's number of columns")
    M = x.shape[0]
    if out is None:
        out = torch.empty(M, qw.rows, dtype=qw.torch_dtype, device=x.device)
    s = qw.struct()
    _check(name, getattr(lib(), name)(ctypes.byref(s), _ptr(x), M, _ptr(out), _stream(stream)))
    return out


def gemv(qw, x, out=None, stream=None):
    """y = x . w_hat^T for 1 <= M <= 16 (decode); for M <= 6 (when x fits the
    kernel's staging room) the block scale is folded after an fp16
    contraction with the code values (see nf4q.h)."""
    return _mm("nf4q_gemv", qw, x, out, stream)


def gemv_multi(qws, x, outs=None, stream=None, static_weights=False):
    """y_i = x . w_hat_i^T for a group of 1..4 weights sharing x (same cols,
    code, double quant and compute dtype), in one launch where possible.
    static_weights: the caller guarantees that no kernel still running when
    this one starts writes the weights (true for weights quantized once and
    reused); their first tiles then load before the wait for the preceding
    kernel (nf4q_gemv_multi_ex with NF4Q_GEMV_WEIGHTS_STATIC; same results)."""
    _require(1 <= len(qws) <= 4, "a group has 1 to 4 weights")
    _require(x.is_cuda and x.dtype == qws[0].torch_dtype and x.is_contiguous() and x.dim() == 2,
             "x must be a contiguous 2-D CUDA tensor of the compute dtype")
    _require(all(q.cols == x.shape[-1] for q in qws), "x must have the weights' columns")
    M = x.shape[0]
    if outs is None:
        outs = [torch.empty(M, q.rows, dtype=q.torch_dtype, device=x.device) for q in qws]
    structs = [q.struct() for q in qws]
    ptrs = (ctypes.POINTER(NF4QWeight) * len(qws))(*[ctypes.pointer(st) for st in structs])
    ys = (ctypes.c_void_p * len(qws))(*[_ptr(o) for o in outs])
    flags = GEMV_WEIGHTS_STATIC if static_weights else 0
    _check("nf4q_gemv_multi_ex", lib().nf4q_gemv_multi_ex(ptrs, len(qws), _ptr(x), M, ys, flags,
                                                           _stream(stream)))
    return outs


def gemv_exact(qw, x, out=None, stream=None):
    """y = x . w_hat^T for 1 <= M <= 16 with w_hat rebuilt bit for bit inside
    the contraction."""
    return _mm("nf4q_gemv_exact", qw, x, out, stream)


def gemm(qw, x, out=None, stream=None):
    """Y = X . w_hat^T on the tcgen05 tensor cores (prefill)."""
    return _mm("nf4q_gemm", qw, x, out, stream)


def matmul(qw, x, out=None, stream=None):
    """Dispatch on M: gemv for M <= 16 (gemm for M = 9..16 on weights of at
    least 20000 rows), gemm above."""
    return _mm("nf4q_matmul", qw, x, out, stream)


def matmul_dx(qw, dy, out=None, stream=None):
    """dX = dY . w_hat (the input gradient through the frozen 4-bit weight)
    on the tcgen05 tensor cores.  dy [M, rows] may have a row pitch larger
    than rows (a column slice of a wider tensor) if it is a multiple of 8."""
    _require(dy.is_cuda and dy.dtype == qw.torch_dtype and dy.dim() == 2,
             "dy must be a 2-D CUDA tensor of the compute dtype")
    _require(dy.shape[1] == qw.rows and dy.stride(1) == 1,
             "dy must have the weight's number of rows, contiguous along them")
    M = dy.shape[0]
    ld = dy.stride(0) if M > 1 else max(qw.rows, dy.stride(0))
    if out is None:
        out = torch.empty(M, qw.cols, dtype=qw.torch_dtype, device=dy.device)
    s = qw.struct()
    _check("nf4q_matmul_dx", lib().nf4q_matmul_dx(ctypes.byref(s), _ptr(dy), ld, M, _ptr(out),
                                                   _stream(stream)))
    return out


def device_error(clear: bool = True) -> int:
    flags = ctypes.c_uint32()
    _check("nf4q_device_error", lib().nf4q_device_error(ctypes.byref(flags), 1 if clear else 0))
    return flags.value


# ---------------------------------------------------------------- LLM.int8()
INT8_DEFAULT_THRESHOLD = 6.0


@dataclass
class Int8Weight:
    """int8 codes [rows, cols] and per-row fp32 absmax (``nf4q_int8_weight``)."""
    q: torch.Tensor
    scale: torch.Tensor
    rows: int
    cols: int

    def struct(self) -> NF4QInt8Weight:
        return NF4QInt8Weight(_ptr(self.q), _ptr(self.scale), self.rows, self.cols)


def int8_quantize_weight(w: torch.Tensor, stream=None) -> Int8Weight:
    """Vector-wise int8 quantization of an fp16 / bf16 weight [rows, cols]."""
    _require(w.is_cuda and w.dim() == 2 and w.is_contiguous(),
             "w must be a contiguous 2-D CUDA tensor")
    _require(w.dtype in (torch.float16, torch.bfloat16), "w must be fp16 or bf16")
    in_dt = _IN_DTYPES[w.dtype]
    rows, cols = w.shape
    wq = Int8Weight(torch.empty(rows, cols, dtype=torch.int8, device=w.device),
                    torch.empty(rows, dtype=torch.float32, device=w.device), rows, cols)
    s = wq.struct()
    _check("nf4q_int8_quantize_weight",
           lib().nf4q_int8_quantize_weight(_ptr(w), in_dt, ctypes.byref(s), _stream(stream)))
    return wq


def int8_workspace(M: int, cols: int, device=None) -> torch.Tensor:
    n = lib().nf4q_int8_workspace_bytes(M, cols)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def int8_workspace_views(ws: torch.Tensor, M: int, cols: int):
    """The sections of a workspace after nf4q_int8_matmul, as the header
    lays them out: (flags u8 [cols], count, list i32 [count], sx f32 [M],
    xq fp16 [M, cols])."""
    def a(v):
        return (v + 255) // 256 * 256
    o_count = a(cols)
    o_list = o_count + 256
    o_sx = o_list + a(4 * cols)
    o_xq = o_sx + a(4 * M)
    flags = ws[:cols]
    count = int(ws[o_count:o_count + 4].view(torch.int32).item())
    lst = ws[o_list:o_list + 4 * cols].view(torch.int32)[:count]
    sx = ws[o_sx:o_sx + 4 * M].view(torch.float32)
    xq = ws[o_xq:o_xq + 2 * M * cols].view(torch.float16).view(M, cols)
    return flags, count, lst, sx, xq


def int8_matmul(wq: Int8Weight, x: torch.Tensor, threshold: float = INT8_DEFAULT_THRESHOLD,
                workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """LLM.int8() decomposition matmul: y [M, rows] = x [M, cols] (fp16)
    against the int8 weight, outlier columns (|x| > threshold) in fp16."""
    _require(x.is_cuda and x.dtype == torch.float16 and x.is_contiguous() and x.dim() == 2,
             "x must be a contiguous 2-D fp16 CUDA tensor")
    _require(x.shape[-1] == wq.cols, "x must have the weight's number of columns")
    M = x.shape[0]
    if workspace is None:
        workspace = int8_workspace(M, wq.cols, x.device)
    if out is None:
        out = torch.empty(M, wq.rows, dtype=torch.float16, device=x.device)
    s = wq.struct()
    _check("nf4q_int8_matmul",
           lib().nf4q_int8_matmul(ctypes.byref(s), _ptr(x), M, float(threshold), _ptr(out),
                                  _ptr(workspace), workspace.numel(), _stream(stream)))
    return out
