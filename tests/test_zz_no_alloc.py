"""nf4q_double_quant_noalloc: the double quantization for callers that cannot
allocate device memory (their memory is all handed to a fixed pool, or a
cudaMalloc - with its implicit device synchronization - is not allowed on
their path).  It keeps its scratch in a small static device array instead of
a caller workspace.

Called through the C ABI and compared with nf4q_double_quant (which takes a
caller workspace) bit for bit - the tolerance every double-quant test here
uses - on two calls in a row, so that a second call that inherited the
first one's scratch contents would show up.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq

pytestmark = pytest.mark.gpu


def _noalloc():
    f = nq.lib().nf4q_double_quant_noalloc
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.POINTER(nq.NF4QWeight), ctypes.c_void_p]
    return f


def _state(absmax: np.ndarray):
    nb = absmax.size
    qw = nq.QuantizedWeight.empty(1, 64 * nb)
    qw.absmax.copy_(torch.from_numpy(absmax))
    return qw


def _outputs(qw):
    torch.cuda.synchronize()
    return (qw.absmax_q.cpu().numpy().copy(), qw.scale2.cpu().numpy().view(np.uint32).copy(),
            qw.offset.cpu().numpy().view(np.uint32).copy())


def test_noalloc_matches_workspace_entry_point_twice():
    assert torch.cuda.is_available()
    from dequant_matmul_quantize_b300 import build
    build.build()
    f = _noalloc()
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(2024)
    inputs = [np.abs(rng.standard_normal(70000) * 0.05).astype(np.float32),
              np.abs(rng.standard_normal(1 << 16) * 3.0).astype(np.float32) + 1.0]
    for absmax in inputs:                      # two calls in a row
        ref = _state(absmax)
        nq.double_quant_into(ref)              # caller-workspace entry point
        got = _state(absmax)
        s = got.struct()
        assert f(ctypes.byref(s), stream) == 0
        for a, b, what in zip(_outputs(got), _outputs(ref), ("absmax_q", "scale2", "offset")):
            assert np.array_equal(a, b), what
    assert nq.device_error() == 0


def test_noalloc_refuses_bad_arguments_without_launching():
    f = _noalloc()
    too_big = nq.NF4QWeight(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1 << 32, 1 << 10,
                            64, 256, 0, 1)
    assert f(ctypes.byref(too_big), None) == 3          # n_b beyond 2^31 - 1
    no_out = nq.NF4QWeight(0x1000, None, 0x3000, 0x4000, 0x5000, 64, 64, 64, 256, 0, 1)
    assert f(ctypes.byref(no_out), None) == 1
