"""GPU parity of fp8_mm (the FP8 scaled product, the forward of the page's
FP8 matmul) against the oracle (oracle/fp8.py), through the C ABI.

x_f8 and w_f8 are decisions taken in the same precision on both sides (the
quotient rounded once to bfloat16, then to E4M3 to nearest even): they must
equal the oracle's bit for bit.  out is the fp32-accumulated product scaled
by x_s w_s and rounded to bfloat16.  Products of E4M3 values are exact in
fp32, so it differs from the oracle's exact sum only by fp32 accumulation
rounding and the fp32 product of the scales: every entry is within one
bfloat16 spacing plus 2**-20 of the scaled sum of |products|, and at least
98 % are equal.  Cases span one tile, several tiles, ragged M, N and K
(K a multiple of 16, N of 8), a single row, and K beyond one 128-element
block.
"""

import numpy as np
import pytest
import torch

import oracle
from newton_schulz_08_gb300 import muon
from tests.gpu_helpers import bf16_ulp

pytestmark = pytest.mark.gpu

CASES = [(256, 256, 256), (300, 520, 384), (64, 136, 1040), (1000, 264, 96), (1, 8, 16), (513, 1024, 128)]


def same(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return bool(np.all((np.isnan(a) & np.isnan(b)) | ((a == b) & (np.signbit(a) == np.signbit(b)))))


def operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    x = oracle.round_to_bf16(rng.standard_normal((M, K)) * 2.0)
    w = oracle.round_to_bf16(rng.standard_normal((N, K)) * 0.05)
    # scales that fill E4M3 without overflow, as float32 (what the ABI takes)
    x_s = np.float32(np.abs(x).max() / 448.0 * 1.05)
    w_s = np.float32(np.abs(w).max() / 448.0 * 1.05)
    return x, w, x_s, w_s


@pytest.mark.parametrize("M,N,K", CASES)
def test_fp8_mm_matches_oracle(M, N, K):
    x, w, x_s, w_s = operands(M, N, K, M + 7 * N + 13 * K)
    dev = torch.device("cuda")
    X = torch.from_numpy(x.astype(np.float32)).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(w.astype(np.float32)).to(dev).to(torch.bfloat16)
    ws = muon.new_workspace(256)
    out, xq, wq = muon.fp8_mm(X, W, float(x_s), float(w_s), workspace=ws)
    torch.cuda.synchronize()
    assert muon.muon_device_status(ws) == muon.MUON_OK
    ref, xq_ref, wq_ref = oracle.fp8_mm(x, w, float(x_s), float(w_s))
    assert same(xq.to(torch.float64).cpu().numpy(), xq_ref)
    assert same(wq.to(torch.float64).cpu().numpy(), wq_ref)
    o = out.to(torch.float64).cpu().numpy()
    mag = (np.abs(xq_ref) @ np.abs(wq_ref).T) * (float(x_s) * float(w_s))
    bound = bf16_ulp(ref) + 2.0 ** -20 * mag
    assert np.all(np.abs(o - ref) <= bound), float(np.max(np.abs(o - ref) - bound))
    assert np.mean(o == ref) >= 0.98


def test_fp8_mm_outputs_view_as_float8():
    """The returned operands read back as PyTorch float8_e4m3fn values, the
    type the page's op returns."""
    x, w, x_s, w_s = operands(128, 64, 64, 5)
    dev = torch.device("cuda")
    X = torch.from_numpy(x.astype(np.float32)).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(w.astype(np.float32)).to(dev).to(torch.bfloat16)
    _, xq, wq = muon.fp8_mm(X, W, float(x_s), float(w_s))
    torch.cuda.synchronize()
    assert xq.dtype == torch.float8_e4m3fn and xq.shape == (128, 64) and wq.shape == (64, 64)
    # PyTorch's own cast of the bf16 quotient agrees here (no quotient lands
    # within float32 rounding of a bfloat16 midpoint in this case)
    want = X.div(float(x_s)).to(torch.float8_e4m3fn)
    assert torch.equal(xq.view(torch.uint8), want.view(torch.uint8))
