"""A 4-bit linear layer and the library calls as PyTorch custom operators.

The pages describe bitsandbytes' 4-bit layer (a Linear layer whose weight is
stored as NF4/FP4 codes and multiplied in a 16-bit compute dtype; "bitsandbytes
tutorial", sec. 3.4 and 四) and, for release 0.46.0, the registration of its
kernels as ``torch.library`` custom operators so that ``torch.compile`` can
trace them without graph breaks ("Bitsandbytes 0.46.0" release notes, sec. 1).
This module does the same for libnf4q:

* ``torch.ops.nf4q.quantize``, ``nf4q.dequantize`` and ``nf4q.matmul`` are
  custom operators whose real implementations call the C ABI (through the
  ctypes binding in this package) and whose fake implementations give the
  output shapes and dtypes, so ``torch.compile(fullgraph=True)`` and
  ``torch.export`` trace through them.
* ``Linear4bit`` holds the quantized state as buffers and computes
  ``x @ w_hat.T (+ bias)`` with ``nf4q.matmul`` (GEMV for up to 16 rows of
  x, the tcgen05 GEMM above).  The bias, not part of the pages' contraction,
  is added by PyTorch.
* ``nf4q.matmul`` is differentiable in x (the weight is frozen): dX = dY .
  w_hat by ``nf4q.matmul_dx`` (nf4q_matmul_dx, a tcgen05 kernel that
  dequantizes w_hat tile by tile, as the forward GEMM does) - the backward
  of a 4-bit base layer under LoRA ("bitsandbytes tutorial", sec. 5.4).
* ``Linear8bitLt`` is the LLM.int8() layer the pages name beside
  ``Linear4bit`` ("bitsandbytes: quantifier un modele PyTorch sans quitter
  PyTorch"; "bitsandbytes tutorial", sec. 3.1 and ``llm_int8_threshold`` in
  sec. 四): an fp16 weight stored as per-row int8 codes, and the
  decomposition matmul through ``nf4q.int8_quantize_weight`` /
  ``nf4q.int8_matmul``.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch
from torch import Tensor

from . import (DTYPES, INT8_DEFAULT_THRESHOLD, Int8Weight, QuantizedWeight,
               dequantize as _dequantize, int8_matmul as _int8_matmul,
               int8_quantize_weight as _int8_quantize_weight, matmul as _matmul,
               matmul_dx as _matmul_dx, quantize as _quantize, sizes)

_TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16}


def _qw(packed, absmax, absmax_q, scale2, offset, rows, cols, code, double_quant,
        compute_dtype) -> QuantizedWeight:
    return QuantizedWeight(packed, absmax, absmax_q, scale2, offset, rows, cols, code,
                           double_quant, compute_dtype)


# ---------------------------------------------------------------- operators
@torch.library.custom_op("nf4q::quantize", mutates_args=())
def quantize_op(w: Tensor, code: str, double_quant: bool, compute_dtype: str
                ) -> Tuple[Tensor, Tensor, Tensor, Tensor, Tensor]:
    """w [rows x cols] (fp32 / bf16 / fp16, CUDA) -> (packed, absmax,
    absmax_q, scale2, offset) of nf4q_quantize_dq (or nf4q_quantize)."""
    qw = _quantize(w.contiguous(), code, double_quant, compute_dtype=compute_dtype)
    return (qw.packed.clone(), qw.absmax.clone(), qw.absmax_q.clone(), qw.scale2.clone(),
            qw.offset.clone())


@quantize_op.register_fake
def _(w, code, double_quant, compute_dtype):
    pb, nb, nd = sizes(w.shape[0], w.shape[1])
    return (w.new_empty(pb, dtype=torch.uint8), w.new_empty(nb, dtype=torch.float32),
            w.new_empty(nb, dtype=torch.int8), w.new_empty(nd, dtype=torch.float32),
            w.new_empty(1, dtype=torch.float32))


@torch.library.custom_op("nf4q::dequantize", mutates_args=())
def dequantize_op(packed: Tensor, absmax: Tensor, absmax_q: Tensor, scale2: Tensor,
                  offset: Tensor, rows: int, cols: int, code: str, double_quant: bool,
                  compute_dtype: str) -> Tensor:
    """w_hat [rows x cols] in the compute dtype (nf4q_dequantize)."""
    return _dequantize(_qw(packed, absmax, absmax_q, scale2, offset, rows, cols, code,
                           double_quant, compute_dtype))


@dequantize_op.register_fake
def _(packed, absmax, absmax_q, scale2, offset, rows, cols, code, double_quant, compute_dtype):
    return packed.new_empty(rows, cols, dtype=_TORCH_DT[compute_dtype])


@torch.library.custom_op("nf4q::matmul", mutates_args=())
def matmul_op(x: Tensor, packed: Tensor, absmax: Tensor, absmax_q: Tensor, scale2: Tensor,
              offset: Tensor, rows: int, cols: int, code: str, double_quant: bool,
              compute_dtype: str) -> Tensor:
    """y [M x rows] = x [M x cols] . w_hat^T (nf4q_matmul)."""
    return _matmul(_qw(packed, absmax, absmax_q, scale2, offset, rows, cols, code,
                       double_quant, compute_dtype), x.contiguous())


@matmul_op.register_fake
def _(x, packed, absmax, absmax_q, scale2, offset, rows, cols, code, double_quant,
      compute_dtype):
    return x.new_empty(x.shape[0], rows, dtype=_TORCH_DT[compute_dtype])


@torch.library.custom_op("nf4q::matmul_dx", mutates_args=())
def matmul_dx_op(dy: Tensor, packed: Tensor, absmax: Tensor, absmax_q: Tensor, scale2: Tensor,
                 offset: Tensor, rows: int, cols: int, code: str, double_quant: bool,
                 compute_dtype: str) -> Tensor:
    """dX [M x cols] = dY [M x rows] . w_hat (nf4q_matmul_dx)."""
    dy = dy.contiguous()
    if rows % 8:  # the kernel reads dY rows at a pitch of a multiple of 8 elements
        wide = dy.new_zeros(dy.shape[0], (rows + 7) // 8 * 8)
        wide[:, :rows] = dy
        dy = wide[:, :rows]
    return _matmul_dx(_qw(packed, absmax, absmax_q, scale2, offset, rows, cols, code,
                          double_quant, compute_dtype), dy)


@matmul_dx_op.register_fake
def _(dy, packed, absmax, absmax_q, scale2, offset, rows, cols, code, double_quant,
      compute_dtype):
    return dy.new_empty(dy.shape[0], cols, dtype=_TORCH_DT[compute_dtype])


# The frozen 4-bit weight gets no gradient; the input's is dX = dY . w_hat
# (QLoRA backward through the base layer, "bitsandbytes tutorial" sec. 5.4).
def _matmul_setup_context(ctx, inputs, output):
    ctx.state = inputs[1:]


def _matmul_backward(ctx, grad_y):
    grad_x = torch.ops.nf4q.matmul_dx(grad_y.to(_TORCH_DT[ctx.state[-1]]), *ctx.state)
    return (grad_x,) + (None,) * len(ctx.state)


matmul_op.register_autograd(_matmul_backward, setup_context=_matmul_setup_context)


@torch.library.custom_op("nf4q::int8_quantize_weight", mutates_args=())
def int8_quantize_weight_op(w: Tensor) -> Tuple[Tensor, Tensor]:
    """w [rows x cols] (fp16 / bf16, CUDA) -> (int8 codes, fp32 row absmax)."""
    wq = _int8_quantize_weight(w.contiguous())
    return wq.q, wq.scale


@int8_quantize_weight_op.register_fake
def _(w):
    return (w.new_empty(w.shape[0], w.shape[1], dtype=torch.int8),
            w.new_empty(w.shape[0], dtype=torch.float32))


@torch.library.custom_op("nf4q::int8_matmul", mutates_args=())
def int8_matmul_op(x: Tensor, q: Tensor, scale: Tensor, threshold: float) -> Tensor:
    """y [M x rows] = the LLM.int8() decomposition matmul of x [M x cols] (fp16)
    with the int8 weight (nf4q_int8_matmul)."""
    return _int8_matmul(Int8Weight(q, scale, q.shape[0], q.shape[1]), x.contiguous(), threshold)


@int8_matmul_op.register_fake
def _(x, q, scale, threshold):
    return x.new_empty(x.shape[0], q.shape[0], dtype=torch.float16)


# ---------------------------------------------------------------- module
class Linear4bit(torch.nn.Module):
    """y = x @ w_hat.T + bias with the weight stored as 4-bit codes.

    Build it from a float weight with :meth:`from_weight` (or an
    ``nn.Linear`` with :meth:`from_linear`); the weight is quantized once on
    its CUDA device.  ``x`` may have any leading dimensions and must be of
    the compute dtype.
    """

    def __init__(self, in_features: int, out_features: int, bias: bool = True,
                 code: str = "nf4", double_quant: bool = True, compute_dtype: str = "bf16",
                 device=None):
        super().__init__()
        if code not in ("nf4", "fp4") or compute_dtype not in DTYPES:
            raise ValueError("code must be nf4|fp4 and compute_dtype bf16|f16")
        if in_features % 64:
            raise ValueError("in_features must be a multiple of 64 (the block size)")
        self.in_features, self.out_features = in_features, out_features
        self.code, self.double_quant, self.compute_dtype = code, double_quant, compute_dtype
        pb, nb, nd = sizes(out_features, in_features)
        dev = torch.device(device) if device is not None else torch.device("cuda")
        self.register_buffer("packed", torch.zeros(pb, dtype=torch.uint8, device=dev))
        self.register_buffer("absmax", torch.zeros(nb, dtype=torch.float32, device=dev))
        self.register_buffer("absmax_q", torch.zeros(nb, dtype=torch.int8, device=dev))
        self.register_buffer("scale2", torch.zeros(nd, dtype=torch.float32, device=dev))
        self.register_buffer("offset", torch.zeros(1, dtype=torch.float32, device=dev))
        if bias:
            self.register_buffer("bias", torch.zeros(out_features, dtype=_TORCH_DT[compute_dtype],
                                                     device=dev))
        else:
            self.bias = None

    @classmethod
    def from_weight(cls, weight: Tensor, bias: Optional[Tensor] = None, code: str = "nf4",
                    double_quant: bool = True, compute_dtype: str = "bf16") -> "Linear4bit":
        out_f, in_f = weight.shape
        m = cls(in_f, out_f, bias is not None, code, double_quant, compute_dtype,
                device=weight.device)
        st = torch.ops.nf4q.quantize(weight, code, double_quant, compute_dtype)
        for name, t in zip(("packed", "absmax", "absmax_q", "scale2", "offset"), st):
            getattr(m, name).copy_(t)
        if bias is not None:
            m.bias.copy_(bias.to(_TORCH_DT[compute_dtype]))
        return m

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear, code: str = "nf4", double_quant: bool = True,
                    compute_dtype: str = "bf16") -> "Linear4bit":
        return cls.from_weight(linear.weight.detach(),
                               None if linear.bias is None else linear.bias.detach(),
                               code, double_quant, compute_dtype)

    def _state(self):
        return (self.packed, self.absmax, self.absmax_q, self.scale2, self.offset,
                self.out_features, self.in_features, self.code, self.double_quant,
                self.compute_dtype)

    def dequantized_weight(self) -> Tensor:
        return torch.ops.nf4q.dequantize(*self._state())

    def forward(self, x: Tensor) -> Tensor:
        lead = x.shape[:-1]
        y = torch.ops.nf4q.matmul(x.reshape(-1, self.in_features), *self._state())
        if self.bias is not None:
            y = y + self.bias
        return y.reshape(*lead, self.out_features)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"code={self.code}, double_quant={self.double_quant}, "
                f"compute_dtype={self.compute_dtype}, bias={self.bias is not None}")


class Linear8bitLt(torch.nn.Module):
    """y = x @ w_hat.T + bias with the weight stored as per-row int8 codes and
    the LLM.int8() decomposition: activation columns with a value above
    ``threshold`` (6.0 by default) in fp16, the rest in int8.  fp16 in and out;
    inference only (the int8 weight is frozen)."""

    def __init__(self, in_features: int, out_features: int, bias: bool = True,
                 threshold: float = INT8_DEFAULT_THRESHOLD, device=None):
        super().__init__()
        if in_features % 16:
            raise ValueError("in_features must be a multiple of 16")
        self.in_features, self.out_features, self.threshold = in_features, out_features, threshold
        dev = torch.device(device) if device is not None else torch.device("cuda")
        self.register_buffer("q", torch.zeros(out_features, in_features, dtype=torch.int8,
                                              device=dev))
        self.register_buffer("scale", torch.zeros(out_features, dtype=torch.float32, device=dev))
        if bias:
            self.register_buffer("bias", torch.zeros(out_features, dtype=torch.float16, device=dev))
        else:
            self.bias = None

    @classmethod
    def from_weight(cls, weight: Tensor, bias: Optional[Tensor] = None,
                    threshold: float = INT8_DEFAULT_THRESHOLD) -> "Linear8bitLt":
        out_f, in_f = weight.shape
        m = cls(in_f, out_f, bias is not None, threshold, device=weight.device)
        q, scale = torch.ops.nf4q.int8_quantize_weight(weight)
        m.q.copy_(q)
        m.scale.copy_(scale)
        if bias is not None:
            m.bias.copy_(bias.to(torch.float16))
        return m

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear,
                    threshold: float = INT8_DEFAULT_THRESHOLD) -> "Linear8bitLt":
        return cls.from_weight(linear.weight.detach().to(torch.float16),
                               None if linear.bias is None else linear.bias.detach(), threshold)

    def forward(self, x: Tensor) -> Tensor:
        lead = x.shape[:-1]
        y = torch.ops.nf4q.int8_matmul(x.reshape(-1, self.in_features), self.q, self.scale,
                                       float(self.threshold))
        if self.bias is not None:
            y = y + self.bias
        return y.reshape(*lead, self.out_features)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"threshold={self.threshold}, bias={self.bias is not None}")
