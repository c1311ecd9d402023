"""Linear4bit and the nf4q custom operators.  CPU tests check registration,
fake (shape) propagation and that torch.export traces through the operators
without running them; GPU tests check the module against the plain binding
calls and torch.compile(fullgraph=True) against eager."""
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
import synth
from dequant_matmul_quantize_b300.nn import Linear4bit, Linear8bitLt


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


@pytest.mark.gpu
@pytest.mark.parametrize("compute_dtype,rows", [("bf16", 160), ("f16", 160), ("bf16", 100)])
def test_backward_through_frozen_base(compute_dtype, rows):
    """dX = dY . w_hat (w_hat exactly as nf4q_dequantize gives it); the 4-bit
    state gets no gradient.  100 rows: dY is re-pitched to 104 columns."""
    dt = torch.bfloat16 if compute_dtype == "bf16" else torch.float16
    w = synth.normal_weight(rows, 256, 0.02, seed=11).cuda()
    lin = Linear4bit.from_weight(w, None, "nf4", True, compute_dtype)
    x = synth.activations(6, 256, seed=12).to(dt).cuda().requires_grad_(True)
    gy = synth.activations(6, rows, seed=13).to(dt).cuda()
    lin(x).backward(gy)
    w_hat = lin.dequantized_weight().float()
    ref = gy.float() @ w_hat
    torch.cuda.synchronize()
    assert x.grad.dtype == dt and x.grad.shape == x.shape
    err = (x.grad.float() - ref).abs()
    # fp32 accumulation in the kernel plus one rounding of the output to 16 bits
    tol = 4e-3 * (gy.float().abs() @ w_hat.abs()) + 1e-30
    assert bool((err <= tol).all())
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
def test_linear4bit_other_configs_forward_and_backward(code, dq):
    """The module over the rest of the config matrix (FP4, no double quant):
    forward equals the binding; the input gradient is dY . w_hat."""
    w = synth.normal_weight(128, 320, 0.02, seed=41).cuda()
    lin = Linear4bit.from_weight(w, None, code, dq, "bf16")
    qw = nq.quantize(w, code, dq)
    x = synth.activations(70, 320, seed=42).cuda().requires_grad_(True)
    y = lin(x)
    assert torch.equal(y, nq.matmul(qw, x.detach()))
    gy = synth.activations(70, 128, seed=43).cuda()
    y.backward(gy)
    w_hat = nq.dequantize(qw).float()
    ref = gy.float() @ w_hat
    torch.cuda.synchronize()
    tol = 4e-3 * (gy.float().abs() @ w_hat.abs()) + 1e-30
    assert bool(((x.grad.float() - ref).abs() <= tol).all())


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
