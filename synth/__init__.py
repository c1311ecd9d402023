"""Seeded synthetic inputs for the NF4 quantize / dequantize / matmul path.

This module only draws random numbers.  It holds none of the method's
arithmetic (no absmax, no code search, no scales): both the CUDA path and the
CPU oracle receive the very same tensors from here.

The recipes follow the workloads the bitsandbytes pages talk about: Llama-
shaped linear weights drawn from a zero-mean normal (the tutorial at
mlqm.cn/news/394670, section 3.2, motivates NF4 by weights being close to a
normal distribution), a sprinkling of large outliers that stress the per-block
absmax, and N(0, 1) bf16 activations.  No dataset or trained checkpoint is
used anywhere; every tensor is random-init.

Every generator takes an explicit seed and a device.  On the CPU the draws
come from ``torch.Generator('cpu')``; on a GPU from a CUDA generator (used
for the very large stacks where only sampled rows are checked on the CPU).
"""
from __future__ import annotations

import torch

# (rows N, cols K) of the seven linear layers of one Llama-3-8B block, with
# the matrix ids used in the per-matrix seed (seed = 1000 * layer + id).
LLAMA3_8B_LAYER = (
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 14336, 4096),
    ("up", 14336, 4096),
    ("down", 4096, 14336),
)
LLAMA3_8B_LAYERS = 32

# Llama-7B decode shapes (rows, cols, seed).
LLAMA7B_DECODE = ((4096, 4096, 10), (11008, 4096, 11), (4096, 11008, 12))
LLAMA7B_X_SEED = 13


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal_weight(rows: int, cols: int, std: float, seed: int, *,
                  dtype=torch.bfloat16, device="cpu",
                  outlier_frac: float = 0.0) -> torch.Tensor:
    """W [rows x cols] ~ N(0, std^2), row-major, cast (RNE) to ``dtype``.

    With ``outlier_frac`` > 0, floor(outlier_frac * rows * cols) entries,
    picked by a random permutation, are replaced by sign * U(0.5, 2.0) with a
    fair random sign before the cast.
    """
    g = _gen(seed, device)
    w = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    w.mul_(std)
    n_out = int(outlier_frac * rows * cols)
    if n_out > 0:
        pos = torch.randperm(rows * cols, generator=g, device=device)[:n_out]
        mag = torch.rand(n_out, generator=g, device=device) * 1.5 + 0.5
        sgn = torch.where(torch.rand(n_out, generator=g, device=device) < 0.5,
                          -1.0, 1.0)
        w.view(-1)[pos] = mag * sgn
    return w.to(dtype).contiguous()


def activations(m: int, k: int, seed: int, *, device="cpu") -> torch.Tensor:
    """x [m x k] bf16 ~ N(0, 1)."""
    g = _gen(seed, device)
    x = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16).contiguous()


def uniform_weight(rows: int, cols: int, lo: float, hi: float, seed: int, *,
                   dtype=torch.float32, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    w = torch.rand(rows, cols, generator=g, device=device, dtype=torch.float32)
    return (w * (hi - lo) + lo).to(dtype).contiguous()


# ---------------------------------------------------------------- workloads
def single_fp32_1024(device="cpu"):
    """Single fp32 1024x1024 weight ~ N(0, 0.02) (seed 0) and x [1 x 1024]
    ~ N(0, 1) (seed 1)."""
    w = normal_weight(1024, 1024, 0.02, 0, dtype=torch.float32, device=device)
    x = activations(1, 1024, 1, device=device)
    return w, x


def llama7b_decode(index: int, device="cpu"):
    """One of the three Llama-7B decode GEMV weights, bf16 N(0, 0.02) with
    0.1 % outliers, and its M=1 activation row."""
    n, k, seed = LLAMA7B_DECODE[index]
    w = normal_weight(n, k, 0.02, seed, device=device, outlier_frac=1e-3)
    x = activations(1, k, LLAMA7B_X_SEED, device=device)
    return w, x


def mlp70b_weight(device="cpu"):
    """70B-MLP-shaped weight [28672 x 8192], bf16 N(0, 0.015), seed 20."""
    return normal_weight(28672, 8192, 0.015, 20, device=device)


def mlp70b_x(m: int, device="cpu"):
    return activations(m, 8192, 21, device=device)


def prefill_weight(device="cpu"):
    """Prefill weight [14336 x 4096], bf16 N(0, 0.02), seed 30."""
    return normal_weight(14336, 4096, 0.02, 30, device=device)


def prefill_x(m: int, device="cpu"):
    return activations(m, 4096, 31, device=device)


def llama3_8b_matrix(layer: int, mid: int, device="cpu"):
    name, n, k = LLAMA3_8B_LAYER[mid]
    return normal_weight(n, k, 0.02, 1000 * layer + mid, device=device)


# Matrices of a block that read the same activation row in a decoder layer:
# q, k and v read the normalized hidden state, gate and up the normalized
# attention output; o and down read their own inputs.
LLAMA3_8B_X_GROUP = (0, 0, 0, 3, 4, 4, 6)


def llama3_8b_x(layer: int, mid: int, device="cpu"):
    """x [1 x K] ~ N(0, 1) bf16 of a stack matrix, shared within a group
    (q/k/v, gate/up): seed 500000 + 1000 * layer + the group's first id."""
    _, n, k = LLAMA3_8B_LAYER[mid]
    return activations(1, k, 500000 + 1000 * layer + LLAMA3_8B_X_GROUP[mid], device=device)


# ---------------------------------------------------------------- LLM.int8()
def outlier_activations(m: int, k: int, seed: int, *, outlier_frac: float = 0.005,
                        outlier_scale: float = 20.0, device="cpu") -> torch.Tensor:
    """x [m x k] fp16 ~ N(0, 1) with a few "outlier feature" columns: a
    random floor(outlier_frac * k) of the columns (at least one when
    outlier_frac > 0) are scaled by ``outlier_scale``, so most of their
    values are far above 6 - the systematic large feature dimensions that
    LLM.int8() splits off (the tutorial at mlqm.cn/news/394670, section 3.1,
    puts them under 1 % of the dimensions)."""
    g = _gen(seed, device)
    x = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
    n_out = max(1, int(outlier_frac * k)) if outlier_frac > 0 else 0
    if n_out:
        cols = torch.randperm(k, generator=g, device=device)[:n_out]
        x[:, cols] *= outlier_scale
    return x.to(torch.float16).contiguous()


def int8_mlp70b_weight(device="cpu"):
    """fp16 [28672 x 8192] ~ N(0, 0.015), seed 40 (the 70B MLP shape)."""
    return normal_weight(28672, 8192, 0.015, 40, dtype=torch.float16, device=device)


def int8_mlp70b_x(m: int, device="cpu"):
    return outlier_activations(m, 8192, 41, device=device)
