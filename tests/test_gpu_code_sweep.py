"""Exhaustive sweep of the encoder's code search ("bitsandbytes tutorial",
sec. 3.2: every value goes to the nearest of the 16 levels).

For an absmax a, every float32 w with |w| <= a is quantized on the GPU, 63
to a 64-block whose first element is a (so the block's absmax is a and the
normalized value is fp32(w / a)).  Both the kernel's codes and the oracle's
are monotone step functions of w: fp32(w / a) is non-decreasing in w (IEEE
division by a positive number), and the oracle's nearest level with ties to
the lower index is non-decreasing in the normalized value (for FP4 this holds
for the magnitude index of |w|, the sign bit being set exactly for w < 0 and
a non-zero magnitude).  So the check is complete with far less host work
than comparing 2 x 10^9 codes one by one: the GPU's codes are checked to be
monotone over the whole sweep (on the device), and at every point where
they change, the two neighbouring values are encoded by the oracle and must
give the same two codes.  Two monotone step functions that agree at both
sides of every step of one of them agree everywhere.

Absmax values: 1 (every float32 in [-1, 1] is its own normalized value), a
value that is not a power of two (the kernel's reciprocal-based fast path
with non-trivial rounding), a large one, and one below 2^-100 (the kernel's
exact IEEE-division path, subnormal inputs included).  Device memory stays
near 2 GB per chunk."""
import numpy as np
import pytest
import torch

import dequant_matmul_quantize_b300 as nq
from oracle import nf4_oracle as o

pytestmark = pytest.mark.gpu

CHUNK_BLOCKS = 1 << 21          # 63 test values per block
ABSMAXES = [1.0, 0.012345678, 3.7e5, 1e-35]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_matmul_quantize_b300 import build
    build.build()
    nq.lib()
    yield
    torch.cuda.synchronize()
    assert nq.device_error() == 0


def _f32_bits(a: float) -> int:
    return int(np.float32(a).view(np.uint32))


def _oracle_codes(w: np.ndarray, a: np.float32, code: int) -> np.ndarray:
    """The oracle's code of each value w in a block of absmax a."""
    w = np.asarray(w, np.float32)
    wn = o.normalize(w, np.full(w.size, a, np.float32), blocksize=1)
    return o.encode(wn, code)


def _key(codes: torch.Tensor, code: str, sign: int) -> torch.Tensor:
    """A key that must be non-decreasing along the sweep (bits of |w| rising):
    the NF4 index (reversed for w < 0) or the FP4 magnitude index."""
    c = codes.to(torch.int16)
    if code == "fp4":
        return c & 7
    return -c if sign else c


def _sweep(code: str, a: float, dtype=torch.float32):
    a32 = np.float32(a)
    cid = o.CODE_NF4 if code == "nf4" else o.CODE_FP4
    if dtype == torch.float32:
        top = _f32_bits(a32)                     # bit patterns 0 .. top are |w| <= a
    else:
        top = int(np.float32(a32).view(np.uint32)) >> 16   # bf16 patterns <= a
        assert np.float32(np.uint32(top << 16).view(np.float32)) <= a32
    checked = 0
    edge_codes = {}
    for sign in (0, 1):
        n_total = top + 1
        prev = None                              # (bits, code) of the last value so far
        edges = []                               # bit patterns at both sides of a change
        for start in range(0, n_total, 63 * CHUNK_BLOCKS):
            n = min(63 * CHUNK_BLOCKS, n_total - start)
            nb = (n + 62) // 63
            bits = torch.arange(start, start + nb * 63, dtype=torch.int32, device="cuda")
            bits = bits.clamp_(max=top)           # pad the last block with a itself
            if dtype == torch.float32:
                pat = bits | (-(1 << 31) if sign else 0)
                vals = pat.view(torch.float32)
                aval = torch.tensor([a], dtype=torch.float32)
            else:
                pat = bits | (sign << 15)
                vals = pat.to(torch.int16).view(torch.bfloat16)
                aval = torch.tensor([a], dtype=torch.float32).to(torch.bfloat16)
            w = torch.empty(nb, 64, dtype=dtype, device="cuda")
            w[:, 0] = aval.to(dtype).cuda()[0]
            w[:, 1:] = vals.view(nb, 63)
            del vals
            qw = nq.quantize(w, code, double_quant=False)
            amax = qw.absmax.float()
            assert torch.all(amax == float(w[0, 0].float()))
            del w
            p = qw.packed.view(nb, 32)
            codes = torch.stack([p >> 4, p & 15], dim=2).view(nb, 64)[:, 1:].reshape(-1)[:n]
            del qw, p
            if code == "fp4":
                mag = codes & 7
                want_sign = torch.full_like(codes, sign, dtype=torch.uint8) & (mag > 0).to(torch.uint8)
                assert torch.equal((codes >> 3).to(torch.uint8), want_sign), "FP4 sign bit"
            key = _key(codes, code, sign)
            assert bool((key[1:] >= key[:-1]).all()), f"{code} a={a} sign={sign}: not monotone"
            bits_n = bits[:n]
            if prev is not None:
                k0 = _key(torch.tensor([prev[1]], dtype=torch.uint8), code, sign)
                assert int(key[0]) >= int(k0[0]), "not monotone across chunks"
                if int(codes[0]) != prev[1]:
                    edges += [prev[0], int(bits_n[0])]
            ch = torch.nonzero(codes[1:] != codes[:-1]).flatten()
            edges += bits_n[ch].tolist() + bits_n[ch + 1].tolist()
            edges += [int(bits_n[0]), int(bits_n[-1])]
            prev = (int(bits_n[-1]), int(codes[-1]))
            # GPU codes at the edge points, for the oracle comparison below
            sel = torch.cat([ch, ch + 1, torch.tensor([0, n - 1], device="cuda")])
            for b_, c_ in zip(bits_n[sel].tolist(), codes[sel].tolist()):
                edge_codes[(sign, b_)] = c_
            checked += n
            del codes, bits, bits_n
        # the oracle at every edge
        eb = np.array(sorted(set(edges)), dtype=np.int64)
        if dtype == torch.float32:
            wv = (eb | (sign << 31)).astype(np.uint32).view(np.float32)
            av = a32
        else:
            wv = ((eb | (sign << 15)).astype(np.uint32) << 16).view(np.float32)
            av = np.float32(torch.tensor([a]).to(torch.bfloat16).float().item())
        want = _oracle_codes(wv, av, cid)
        got = np.array([edge_codes[(sign, int(b))] for b in eb], dtype=np.uint8)
        bad = np.nonzero(want != got)[0]
        assert bad.size == 0, (f"{code} a={a} sign={sign}: {bad.size} edge mismatches, "
                               f"first w={wv[bad[:3]]}, gpu={got[bad[:3]]}, oracle={want[bad[:3]]}")
    return checked



@pytest.mark.parametrize("code", ["nf4", "fp4"])
@pytest.mark.parametrize("a", ABSMAXES)
def test_every_float32_up_to_absmax(code, a):
    n = _sweep(code, a)
    assert n == 2 * (_f32_bits(a) + 1)


@pytest.mark.parametrize("code", ["nf4", "fp4"])
def test_every_bf16_up_to_absmax(code):
    for a in (1.0, 0.0123, 3.7e5):
        _sweep(code, a, torch.bfloat16)
