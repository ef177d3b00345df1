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


def test_fp8_mm_at_the_benchmarked_shape():
    """65536 x 3072 x 768 (the bench's workload, 3,072 tiles of 6 K blocks):
    both E4M3 operands bit for bit in full, and out on blocks of rows at the
    start, middle and end against the oracle on those rows."""
    M, N, K = 65536, 3072, 768
    rng = np.random.default_rng(11)
    x = oracle.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    w = oracle.round_to_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    x_s = np.float32(np.abs(x).max() / 448.0 * 1.05)
    w_s = np.float32(np.abs(w).max() / 448.0 * 1.05)
    dev = torch.device("cuda")
    X = torch.from_numpy(x.astype(np.float32)).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(w.astype(np.float32)).to(dev).to(torch.bfloat16)
    ws = muon.new_workspace(256)
    out, xq, wq = muon.fp8_mm(X, W, float(x_s), float(w_s), workspace=ws)
    torch.cuda.synchronize()
    assert muon.muon_device_status(ws) == muon.MUON_OK
    xq_ref = oracle.quantize(x, float(x_s), "e4m3")
    wq_ref = oracle.quantize(w, float(w_s), "e4m3")
    assert same(xq.to(torch.float64).cpu().numpy(), xq_ref)
    assert same(wq.to(torch.float64).cpu().numpy(), wq_ref)
    o = out.to(torch.float64).cpu().numpy()
    for r0 in (0, 32768 - 128, M - 300):
        rows = slice(r0, r0 + 300 if r0 + 300 <= M else M)
        ref, _, _ = oracle.fp8_mm(x[rows], w, float(x_s), float(w_s))
        mag = (np.abs(xq_ref[rows]) @ np.abs(wq_ref).T) * (float(x_s) * float(w_s))
        bound = bf16_ulp(ref) + 2.0 ** -20 * mag
        assert np.all(np.abs(o[rows] - ref) <= bound), r0
        assert np.mean(o[rows] == ref) >= 0.98


def test_fp8_mm_e4m3_overflow_is_nan():
    """Quotients past E4M3's rounding range become NaN; exactly 464 (the
    midpoint between 448 and the next step) rounds to 448 (even).  Rows and
    columns that meet a NaN operand are NaN in out; the others keep the
    bound."""
    M, N, K = 256, 136, 128
    rng = np.random.default_rng(12)
    x = oracle.round_to_bf16(rng.standard_normal((M, K)) * 2.0)
    w = oracle.round_to_bf16(rng.standard_normal((N, K)) * 0.05)
    x_s, w_s = 1.0, float(np.float32(np.abs(w).max() / 448.0 * 1.05))
    # with x_s = 1 the bf16 quotient is x itself
    specials = [464.0, -464.0, 466.0, -466.0, 1000.0, -65536.0, 448.0, 460.0]
    for j, v in enumerate(specials):
        x[3 * j, 5 + j] = v
    dev = torch.device("cuda")
    X = torch.from_numpy(x.astype(np.float32)).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(w.astype(np.float32)).to(dev).to(torch.bfloat16)
    out, xq, wq = muon.fp8_mm(X, W, x_s, w_s)
    torch.cuda.synchronize()
    ref, xq_ref, wq_ref = oracle.fp8_mm(x, w, x_s, w_s)
    got = xq.to(torch.float64).cpu().numpy()
    assert same(got, xq_ref) and same(wq.to(torch.float64).cpu().numpy(), wq_ref)
    assert got[0, 5] == 448.0 and got[3, 6] == -448.0
    assert np.isnan(got[6, 7]) and np.isnan(got[9, 8]) and np.isnan(got[12, 9]) and np.isnan(got[15, 10])
    assert got[18, 11] == 448.0 and got[21, 12] == 448.0
    # NaN codes are the format's: S.1111.111
    codes = xq.view(torch.uint8).cpu().numpy()
    assert all((codes[r, c] & 0x7F) == 0x7F for r, c in [(6, 7), (9, 8), (12, 9), (15, 10)])
    o = out.to(torch.float64).cpu().numpy()
    nan_rows = np.isnan(ref).any(axis=1)
    assert np.array_equal(np.isnan(o), np.isnan(ref)) and nan_rows.sum() == 4
    mag = (np.abs(xq_ref[~nan_rows]) @ np.abs(wq_ref).T) * (x_s * w_s)
    bound = bf16_ulp(ref[~nan_rows]) + 2.0 ** -20 * mag
    assert np.all(np.abs(o[~nan_rows] - ref[~nan_rows]) <= bound)


# ------------------------------------------------------------------ backward
# grad_x = (grad_s w_s)(g_f8 . w_f8) and grad_w = (grad_s x_s)(g_f8^T . x_f8)
# against oracle.fp8_mm_backward: g_f8 bit for bit (a decision taken in the
# same precision on both sides), the products within one bf16 spacing plus
# 2**-20 of the scaled sum of |products| (fp32 accumulation; a split
# contraction adds its fp32 slices in order).
BWD_CASES = [(256, 256, 256), (272, 528, 384), (64, 48, 1040), (1024, 96, 160), (16, 16, 16), (4096, 272, 64),
             (1040, 48, 1040)]


def bwd_operands(M, N, K, seed):
    x, w, x_s, w_s = operands(M, N, K, seed)
    rng = np.random.default_rng(seed + 1)
    g = oracle.round_to_bf16(rng.standard_normal((M, N)) * 1e-3)
    grad_s = np.float32(np.abs(g).max() / 57344.0 * 1.05)
    return x, w, g, x_s, w_s, grad_s


def check_bwd(g_dev, xq, wq, x_s, w_s, grad_s, g, xq_ref, wq_ref, rows_x=None, rows_w=None):
    gx, gw, gq = muon.fp8_mm_backward(g_dev, xq, wq, float(x_s), float(w_s), float(grad_s))
    torch.cuda.synchronize()
    gq_ref = oracle.quantize(g, float(grad_s), "e5m2")
    got_q = gq.to(torch.float64).cpu().numpy()
    assert same(got_q, gq_ref)
    rx = slice(None) if rows_x is None else rows_x
    cw = slice(None) if rows_w is None else rows_w
    ref_x = oracle.round_to_bf16((gq_ref[rx] @ wq_ref) * (float(grad_s) * float(w_s)))
    ref_w = oracle.round_to_bf16((gq_ref[:, cw].T @ xq_ref) * (float(grad_s) * float(x_s)))
    mag_x = (np.abs(gq_ref[rx]) @ np.abs(wq_ref)) * (float(grad_s) * float(w_s))
    mag_w = (np.abs(gq_ref[:, cw]).T @ np.abs(xq_ref)) * (float(grad_s) * float(x_s))
    for got, ref, mag, what in ((gx.to(torch.float64).cpu().numpy()[rx], ref_x, mag_x, "grad_x"),
                                (gw.to(torch.float64).cpu().numpy()[cw], ref_w, mag_w, "grad_w")):
        bound = bf16_ulp(ref) + 2.0 ** -20 * mag
        assert np.all(np.abs(got - ref) <= bound), (what, float(np.max(np.abs(got - ref) - bound)))
        assert np.mean(got == ref) >= 0.95, what


@pytest.mark.parametrize("M,N,K", BWD_CASES)
def test_fp8_mm_backward_matches_oracle(M, N, K):
    x, w, g, x_s, w_s, grad_s = bwd_operands(M, N, K, 3 * M + 5 * N + K)
    dev = torch.device("cuda")
    X = torch.from_numpy(x.astype(np.float32)).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(w.astype(np.float32)).to(dev).to(torch.bfloat16)
    _, xq, wq = muon.fp8_mm(X, W, float(x_s), float(w_s))
    G = torch.from_numpy(g.astype(np.float32)).to(dev).to(torch.bfloat16)
    xq_ref = oracle.quantize(x, float(x_s), "e4m3")
    wq_ref = oracle.quantize(w, float(w_s), "e4m3")
    check_bwd(G, xq, wq, x_s, w_s, grad_s, g, xq_ref, wq_ref)


def test_fp8_mm_backward_at_the_benchmarked_shape():
    """65536 x 3072 x 768: g_f8 in full; grad_x on blocks of rows and
    grad_w on a block of rows (the split contraction over all 65536)."""
    M, N, K = 65536, 3072, 768
    rng = np.random.default_rng(31)
    dev = torch.device("cuda")
    xq_ref = oracle.quantize(rng.standard_normal((M, K)).astype(np.float32) * 4, 1.0, "e4m3")
    wq_ref = oracle.quantize(rng.standard_normal((N, K)).astype(np.float32) * 4, 1.0, "e4m3")
    g = oracle.round_to_bf16(rng.standard_normal((M, N)).astype(np.float32) * np.float32(1e-3))
    grad_s = np.float32(np.abs(g).max() / 57344.0 * 1.05)
    xq = torch.from_numpy(xq_ref).to(dev).to(torch.float8_e4m3fn)
    wq = torch.from_numpy(wq_ref).to(dev).to(torch.float8_e4m3fn)
    G = torch.from_numpy(g.astype(np.float32)).to(dev).to(torch.bfloat16)
    gx, gw, gq = muon.fp8_mm_backward(G, xq, wq, 1.0, 1.0, float(grad_s))
    torch.cuda.synchronize()
    got_q = gq.view(torch.uint8)
    for r0 in range(0, M, 8192):  # g_f8 in full, in row blocks
        want = torch.from_numpy(oracle.quantize(g[r0:r0 + 8192], float(grad_s), "e5m2")).to(torch.float8_e5m2)
        assert torch.equal(got_q[r0:r0 + 8192].cpu(), want.view(torch.uint8)), r0
    gq_ref = np.concatenate([oracle.quantize(g[:, c0:c0 + 64], float(grad_s), "e5m2") for c0 in (0, 1536)], axis=1)
    gxn, gwn = gx.to(torch.float64).cpu().numpy(), gw.to(torch.float64).cpu().numpy()
    for r0 in (0, 40000, M - 256):
        gqr = oracle.quantize(g[r0:r0 + 256], float(grad_s), "e5m2")
        ref = oracle.round_to_bf16((gqr @ wq_ref) * float(grad_s))
        bound = bf16_ulp(ref) + 2.0 ** -20 * (np.abs(gqr) @ np.abs(wq_ref)) * float(grad_s)
        assert np.all(np.abs(gxn[r0:r0 + 256] - ref) <= bound), r0
    for j, c0 in enumerate((0, 1536)):
        gc = gq_ref[:, 64 * j:64 * j + 64]
        ref = oracle.round_to_bf16((gc.T @ xq_ref) * float(grad_s))
        bound = bf16_ulp(ref) + 2.0 ** -20 * (np.abs(gc).T @ np.abs(xq_ref)) * float(grad_s)
        assert np.all(np.abs(gwn[c0:c0 + 64] - ref) <= bound), c0


def all_bf16_patterns():
    """Every bfloat16 bit pattern, as a 256 x 256 float32 array (NaNs
    included)."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    return bits.view(np.float32).reshape(256, 256)


@pytest.mark.parametrize("scale", [1.0, 0.0137, 3.0e-5, 7.5])
def test_quantise_passes_on_every_bf16_value(scale):
    """Both quantise passes on all 65,536 bfloat16 inputs: E4M3 codes of the
    forward and E5M2 codes of the backward equal the oracle's bit for bit,
    including NaN, infinities, subnormals and the overflow boundaries; a
    scale other than 1 exercises the quotient's rounding."""
    dev = torch.device("cuda")
    v = all_bf16_patterns()
    V = torch.from_numpy(v).to(dev).to(torch.bfloat16)
    s = float(np.float32(scale))
    _, xq, _ = muon.fp8_mm(V, torch.zeros((16, 256), dtype=torch.bfloat16, device=dev), s, 1.0)
    z8 = torch.zeros((256, 16), dtype=torch.uint8, device=dev)
    _, _, gq = muon.fp8_mm_backward(V, z8, torch.zeros((256, 16), dtype=torch.uint8, device=dev), 1.0, 1.0, s)
    torch.cuda.synchronize()
    vb = oracle.round_to_bf16(v.astype(np.float64))
    with np.errstate(invalid="ignore", over="ignore"):
        assert same(xq.to(torch.float64).cpu().numpy(), oracle.quantize(vb, s, "e4m3"))
        assert same(gq.to(torch.float64).cpu().numpy(), oracle.quantize(vb, s, "e5m2"))
