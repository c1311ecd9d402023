"""Linear4bit and the nf4q custom operators.  CPU tests check registration,
fake (shape) propagation and that torch.export traces through the operators
without running them; GPU tests check the module's forward and input
gradient against the CPU oracle (fp64 on the oracle's own dequantized
weights, within the matmul tolerance), against the plain binding calls, and
torch.compile(fullgraph=True) against eager."""
import pytest
import torch

import numpy as np

import dequant_matmul_quantize_b300 as nq
import synth
from dequant_matmul_quantize_b300.nn import Linear4bit, Linear8bitLt
from oracle import nf4_oracle as o
from tests._util import CODE_ID, as_f32, oracle_state


def test_operators_are_registered():
    for name in ("quantize", "dequantize", "matmul", "matmul_dx", "int8_quantize_weight",
                 "int8_matmul"):
        assert hasattr(torch.ops.nf4q, name)


def test_fake_shapes_and_dtypes():
    from torch._subclasses.fake_tensor import FakeTensorMode
    with FakeTensorMode():
        w = torch.empty(96, 256, dtype=torch.bfloat16)
        st = torch.ops.nf4q.quantize(w, "nf4", True, "f16")
        assert [tuple(t.shape) for t in st] == [(96 * 256 // 2,), (384,), (384,), (2,), (1,)]
        assert [t.dtype for t in st] == [torch.uint8, torch.float32, torch.int8,
                                         torch.float32, torch.float32]
        w_hat = torch.ops.nf4q.dequantize(*st, 96, 256, "nf4", True, "f16")
        assert w_hat.shape == (96, 256) and w_hat.dtype == torch.float16
        x = torch.empty(5, 256, dtype=torch.float16)
        y = torch.ops.nf4q.matmul(x, *st, 96, 256, "nf4", True, "f16")
        assert y.shape == (5, 96) and y.dtype == torch.float16
        dx = torch.ops.nf4q.matmul_dx(y, *st, 96, 256, "nf4", True, "f16")
        assert dx.shape == (5, 256) and dx.dtype == torch.float16


def test_int8_fake_shapes_and_export():
    from torch._subclasses.fake_tensor import FakeTensorMode
    with FakeTensorMode():
        w = torch.empty(48, 64, dtype=torch.float16)
        q, sc = torch.ops.nf4q.int8_quantize_weight(w)
        assert q.shape == (48, 64) and q.dtype == torch.int8 and sc.shape == (48,)
        y = torch.ops.nf4q.int8_matmul(torch.empty(3, 64, dtype=torch.float16), q, sc, 6.0)
        assert y.shape == (3, 48) and y.dtype == torch.float16
    m = Linear8bitLt(64, 32, bias=True, device="cpu")
    ep = torch.export.export(m, (torch.empty(2, 5, 64, dtype=torch.float16),))
    targets = [str(n.target) for n in ep.graph.nodes if n.op == "call_function"]
    assert any("nf4q.int8_matmul" in t for t in targets), targets


def test_export_traces_through_the_operator():
    m = Linear4bit(128, 48, bias=True, device="cpu")
    ep = torch.export.export(m, (torch.empty(3, 7, 128, dtype=torch.bfloat16),))
    targets = [str(n.target) for n in ep.graph.nodes if n.op == "call_function"]
    assert any("nf4q.matmul" in t for t in targets), targets


def test_module_argument_checks():
    with pytest.raises(ValueError):
        Linear4bit(100, 8, device="cpu")             # not a multiple of 64
    with pytest.raises(ValueError):
        Linear4bit(128, 8, code="int4", device="cpu")


@pytest.mark.gpu
@pytest.mark.parametrize("compute_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M", [1, 9, 100])
def test_linear4bit_matches_binding(compute_dtype, M):
    dt = torch.bfloat16 if compute_dtype == "bf16" else torch.float16
    w = synth.normal_weight(192, 512, 0.02, seed=M).cuda()
    b = torch.randn(192, generator=torch.Generator().manual_seed(M)).to(dt).cuda()
    lin = Linear4bit.from_weight(w, b, "nf4", True, compute_dtype)
    qw = nq.quantize(w, "nf4", True, compute_dtype=compute_dtype)
    x = synth.activations(M, 512, seed=M + 1).to(dt).cuda()
    y = lin(x)
    ref = nq.matmul(qw, x) + b
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    assert torch.equal(lin.dequantized_weight(), nq.dequantize(qw))


@pytest.mark.gpu
def test_compile_fullgraph_matches_eager():
    torch.manual_seed(0)
    l1 = torch.nn.Linear(512, 256).cuda()
    l2 = torch.nn.Linear(256, 128).cuda()
    mlp = torch.nn.Sequential(Linear4bit.from_linear(l1), torch.nn.GELU(),
                              Linear4bit.from_linear(l2))
    x = synth.activations(24, 512, seed=3).cuda().reshape(2, 12, 512)
    eager = mlp(x)
    # fullgraph: the nf4q operators trace without graph breaks; the aot_eager
    # backend runs the traced graph as is (no code generation)
    compiled = torch.compile(mlp, fullgraph=True, backend="aot_eager")(x)
    torch.cuda.synchronize()
    assert compiled.shape == (2, 12, 128)
    assert torch.equal(compiled, eager)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _oracle_w_hat(w: torch.Tensor, code: str, dq: bool, dt: int) -> np.ndarray:
    """The oracle's dequantized weight (bit patterns of the compute dtype)."""
    st = oracle_state(as_f32(w).reshape(-1), code, dq)
    return o.dequantize(st["packed"], st["scales"], CODE_ID[code], dtype=dt).reshape(w.shape)


def _check_tol(got: torch.Tensor, ref: np.ndarray, bound: np.ndarray, dt: int, what: str):
    y = o.from_bits(_bits(got), dt).astype(np.float64)
    tol = o.matmul_tolerance(ref, bound, dt)
    err = np.abs(y - ref)
    assert np.all(err <= tol), f"{what}: worst err/tol {np.max(err / tol):.3f}"


CONFIGS = [("nf4", True, "bf16"), ("nf4", True, "f16"), ("fp4", True, "bf16"),
           ("nf4", False, "bf16"), ("fp4", False, "f16")]


@pytest.mark.gpu
@pytest.mark.parametrize("code,dq,compute_dtype", CONFIGS)
@pytest.mark.parametrize("M,rows", [(1, 160), (5, 100), (70, 160)])
def test_linear4bit_forward_and_backward_against_oracle(code, dq, compute_dtype, M, rows):
    """Linear4bit over the config matrix (NF4 / FP4, double quant on / off,
    bf16 / fp16 compute): its dequantized weight equals the oracle's bit for
    bit; the forward without bias and the input gradient dX = dY . w_hat of
    the frozen base match the oracle's fp64 products within the matmul
    tolerance (2e-3 * sum|a b| + one ulp); the bias is added in the compute
    dtype.  100 rows: dY is re-pitched to 104 columns for the backward."""
    tdt = torch.bfloat16 if compute_dtype == "bf16" else torch.float16
    odt = o.DT_BF16 if compute_dtype == "bf16" else o.DT_F16
    w = synth.normal_weight(rows, 256, 0.02, seed=11 + M).cuda()
    b = synth.normal_weight(1, rows, 0.5, seed=12 + M).reshape(-1).to(tdt).cuda()
    lin = Linear4bit.from_weight(w, None, code, dq, compute_dtype)
    lin_b = Linear4bit.from_weight(w, b, code, dq, compute_dtype)
    w_hat = _oracle_w_hat(w.cpu(), code, dq, odt)
    assert np.array_equal(_bits(lin.dequantized_weight()), w_hat)
    x = synth.activations(M, 256, seed=13 + M).to(tdt).cuda().requires_grad_(True)
    y = lin(x)
    y_ref, bound = o.matmul_ref(_bits(x), w_hat, odt)
    _check_tol(y, y_ref, bound, odt, f"forward {code} dq={dq} {compute_dtype} M={M}")
    assert torch.equal(lin_b(x.detach()), y.detach() + b)
    gy = synth.activations(M, rows, seed=14 + M).to(tdt).cuda()
    y.backward(gy)
    torch.cuda.synchronize()
    assert x.grad.dtype == tdt and x.grad.shape == x.shape
    dx_ref, dbound = o.matmul_dx_ref(_bits(gy), w_hat, odt)
    _check_tol(x.grad, dx_ref, dbound, odt, f"backward {code} dq={dq} {compute_dtype} M={M}")
    assert lin.packed.grad is None


@pytest.mark.gpu
def test_linear8bitlt_matches_binding_and_compiles():
    """Linear8bitLt gives the binding's int8 matmul (+ bias) bit for bit, in
    eager mode and under torch.compile(fullgraph=True)."""
    w = synth.normal_weight(96, 256, 0.02, seed=31, dtype=torch.float16).cuda()
    b = synth.normal_weight(1, 96, 0.1, seed=32, dtype=torch.float16).cuda().reshape(-1)
    lin = Linear8bitLt.from_weight(w, b)
    x = synth.outlier_activations(12, 256, seed=33, outlier_frac=0.02).cuda().reshape(3, 4, 256)
    y = lin(x)
    wq = nq.int8_quantize_weight(w)
    ref = nq.int8_matmul(wq, x.reshape(12, 256)) + b.to(torch.float16)
    torch.cuda.synchronize()
    assert torch.equal(lin.q, wq.q) and torch.equal(lin.scale, wq.scale)
    assert torch.equal(y.reshape(12, 96), ref)
    compiled = torch.compile(lin, fullgraph=True, backend="aot_eager")
    assert torch.equal(compiled(x), y)


@pytest.mark.gpu
@pytest.mark.parametrize("code,dq", [("fp4", True), ("nf4", False), ("fp4", False)])
def test_linear4bit_other_configs_match_binding(code, dq):
    """The module over the rest of the config matrix (FP4, no double quant)
    gives the binding's matmul bit for bit."""
    w = synth.normal_weight(128, 320, 0.02, seed=41).cuda()
    lin = Linear4bit.from_weight(w, None, code, dq, "bf16")
    qw = nq.quantize(w, code, dq)
    x = synth.activations(70, 320, seed=42).cuda()
    assert torch.equal(lin(x), nq.matmul(qw, x))


@pytest.mark.gpu
def test_from_linear_and_state_dict_round_trip():
    """Both modules built from an nn.Linear; their state (codes, scales, bias)
    survives a state_dict round trip into fresh modules bit for bit."""
    torch.manual_seed(0)
    lin = torch.nn.Linear(256, 96, bias=True).cuda()
    m4 = Linear4bit.from_linear(lin, "nf4", True, "bf16")
    fresh4 = Linear4bit(256, 96, True, "nf4", True, "bf16")
    fresh4.load_state_dict(m4.state_dict())
    x = synth.activations(5, 256, seed=51).cuda()
    assert torch.equal(fresh4(x), m4(x))
    ref = nq.matmul(nq.quantize(lin.weight.detach()), x) + lin.bias.detach().to(torch.bfloat16)
    assert torch.equal(m4(x), ref)
    m8 = Linear8bitLt.from_linear(lin)
    fresh8 = Linear8bitLt(256, 96, True)
    fresh8.load_state_dict(m8.state_dict())
    x16 = synth.outlier_activations(5, 256, seed=52, outlier_frac=0.02).cuda()
    torch.cuda.synchronize()
    assert torch.equal(fresh8(x16), m8(x16))
