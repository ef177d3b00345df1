"""Pins of the FP8 scaled-matmul oracle (oracle/fp8.py), CPU only.

The page "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术"
(reposource.net), section "自定义FP8矩阵乘法实现", casts x / x_s and w / w_s
to E4M3 with PyTorch's own conversion and multiplies in FP8; its backward
casts g / grad_s to E5M2.  The oracle restates those casts from the formats'
definitions; here they are checked against:

* PyTorch's float8 conversions (an independent implementation, the one the
  page's op calls) on all 65,536 bfloat16 values, on every midpoint between
  neighbouring FP8 values and its neighbours, and on random float32 values;
* a bit-field decoding of all 256 codes and rounding by exhaustive search in
  rational arithmetic (tests/pins.py);
* the page's own first step, ``x.div(x_s).to(torch.float8_e4m3fn)`` on a
  bfloat16 tensor.

The matmul is checked by closed forms (operands already representable:
the result is the bf16 rounding of the exact product), by power-of-two scale
invariance, and by brute force in rational arithmetic; planted mistakes each
fail one of these checks.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as of
from tests import pins

TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def torch_cast(x32, fmt):
    """PyTorch's float32 -> FP8 conversion, back to float64."""
    return torch.from_numpy(np.asarray(x32, np.float32)).to(TORCH_FP8[fmt]).to(torch.float64).numpy()


def same(a, b):
    """Equal values with equal signs of zero, NaN where NaN."""
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return bool(np.all(nan | eq))


def all_bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    return bits.view(np.float32)


def fp8_values(fmt):
    v = np.array([pins.fp8_decode(c, fmt) for c in range(256)])
    return v


# ------------------------------------------------------------------ casts
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_cast_matches_torch_on_all_bfloat16_values(fmt):
    x = all_bf16_values()
    with np.errstate(invalid="ignore"):  # the signalling NaN patterns
        assert same(oracle.round_to_fp8(x, fmt), torch_cast(x, fmt))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_cast_matches_torch_on_midpoints_and_neighbours(fmt):
    v = np.unique(fp8_values(fmt)[np.isfinite(fp8_values(fmt))])
    mids = (v[:-1] + v[1:]) / 2  # exact: FP8 values have at most 4 significant bits
    top = of.FP8_FORMATS[fmt]["max"]
    # midpoint above the largest value: half the spacing of its binade
    # (464 for E4M3, 61440 for E5M2)
    over = np.array([top + 2.0 ** (np.floor(np.log2(top)) - of.FP8_FORMATS[fmt]["frac"] - 1)])
    m = np.concatenate([mids, over, -over]).astype(np.float32)
    x = np.concatenate([m, np.nextafter(m, np.float32(np.inf)), np.nextafter(m, np.float32(-np.inf))])
    assert same(oracle.round_to_fp8(x, fmt), torch_cast(x, fmt))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_cast_matches_torch_on_random_float32(fmt):
    rng = np.random.default_rng(81)
    mag = np.exp2(rng.uniform(-30, 20, 200_000))
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, np.inf, -np.inf, np.nan], np.float32)])
    assert same(oracle.round_to_fp8(x, fmt), torch_cast(x, fmt))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_codes_decode_and_round_to_themselves(fmt):
    v = fp8_values(fmt)
    fin = np.isfinite(v)
    # E4M3 "fn": 2 NaN codes, no infinity; E5M2: 6 NaN codes and 2 infinities
    assert int(np.isnan(v).sum()) == (2 if fmt == "e4m3" else 6)
    assert int(np.isinf(v).sum()) == (0 if fmt == "e4m3" else 2)
    assert same(oracle.round_to_fp8(v[fin], fmt), v[fin])
    # PyTorch reads the same bits as the same values
    tv = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(TORCH_FP8[fmt]).to(torch.float64).numpy()
    assert same(v, tv)
    pos = v[fin & (v > 0)]
    assert pos.max() == of.FP8_FORMATS[fmt]["max"]
    assert pos.min() == (2.0 ** -9 if fmt == "e4m3" else 2.0 ** -16)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_cast_matches_exhaustive_search(fmt):
    rng = np.random.default_rng(82)
    top = of.FP8_FORMATS[fmt]["max"]
    x = np.concatenate([rng.uniform(-1.2 * top, 1.2 * top, 300),
                        np.exp2(rng.uniform(-20, 2, 300)) * rng.choice([-1, 1], 300)])
    want = [pins.fp8_nearest(float(a), fmt) for a in x]
    assert same(oracle.round_to_fp8(x, fmt), want)


def test_quantize_follows_the_page_cast_of_a_bfloat16_tensor():
    """x.div(x_s).to(float8_e4m3fn) on a bfloat16 tensor: the quotient is
    rounded to bfloat16 first (reading 2)."""
    rng = np.random.default_rng(83)
    x = torch.from_numpy(rng.standard_normal((64, 96)).astype(np.float32) * 3).to(torch.bfloat16)
    for s in (0.013, 1.0, 0.5, 7.3, 1 / 448):
        want = x.div(s).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        got = oracle.quantize(x.to(torch.float64).numpy(), s, "e4m3", "bf16")
        assert same(got, want), s
    g = torch.from_numpy(rng.standard_normal((64, 96)).astype(np.float32) * 1e-3).to(torch.bfloat16)
    for s in (1e-6, 3e-5):
        want = g.div(s).to(torch.float8_e5m2).to(torch.float64).numpy()
        assert same(oracle.quantize(g.to(torch.float64).numpy(), s, "e5m2", "bf16"), want), s


def test_division_rounding_matters():
    """A quotient just above an E4M3 midpoint that bfloat16 rounds onto it:
    the double rounding of the page's op and a direct cast differ."""
    # 1.0625 is the midpoint of E4M3 1.0 and 1.125; q sits 2**-12 above it,
    # which bfloat16 (8 significant bits) rounds down onto the midpoint
    q = 1.0625 + 2.0 ** -12
    assert oracle.round_to_bf16(q) == 1.0625
    assert oracle.quantize(q, 1.0, "e4m3", "fp64") == 1.125
    assert oracle.quantize(q, 1.0, "e4m3", "bf16") == 1.0


# ------------------------------------------------------------------ matmul
def representable(rng, shape, fmt, scale=1.0):
    codes = rng.integers(0, 256, shape)
    v = np.array([pins.fp8_decode(int(c), fmt) for c in codes.ravel()]).reshape(shape)
    v = np.where(np.isfinite(v), v, 0.0)
    return v * scale


def test_mm_of_representable_operands_is_the_rounded_exact_product():
    rng = np.random.default_rng(84)
    for M, N, K, xs, ws in [(5, 7, 16, 1.0, 1.0), (8, 3, 33, 2.0 ** -7, 2.0 ** 3), (1, 1, 1, 0.25, 4.0)]:
        x = representable(rng, (M, K), "e4m3", xs)
        w = representable(rng, (N, K), "e4m3", ws)
        out, x_f8, w_f8 = oracle.fp8_mm(x, w, xs, ws, in_dtype="fp64")
        assert np.array_equal(x_f8 * xs, x) and np.array_equal(w_f8 * ws, w)
        assert same(out, oracle.round_to_bf16(x @ w.T))
        out32, _, _ = oracle.fp8_mm(x, w, xs, ws, in_dtype="fp64", out_dtype="fp32")
        assert same(out32, (x @ w.T).astype(np.float32))


def test_mm_is_invariant_under_power_of_two_rescaling():
    rng = np.random.default_rng(85)
    x = oracle.round_to_bf16(rng.standard_normal((6, 40)))
    w = oracle.round_to_bf16(rng.standard_normal((9, 40)) * 0.05)
    out, x_f8, w_f8 = oracle.fp8_mm(x, w, 0.01, 0.0007)
    for k in (-5, 3, 11):
        o2, x2, w2 = oracle.fp8_mm(x * 2.0 ** k, w * 2.0 ** -k, 0.01 * 2.0 ** k, 0.0007 * 2.0 ** -k)
        assert same(o2, out) and same(x2, x_f8) and same(w2, w_f8)


def _brute_force_mm(x, w, xs, ws, fmt="e4m3"):
    """Quantise by exhaustive search, sum in rationals, round to bfloat16 by
    table search (tests/pins.py): nothing shared with the oracle."""
    M, K = x.shape
    N = w.shape[0]
    xq = [[Fraction(pins.fp8_nearest(pins.bf16_nearest(Fraction(float(x[i][k])) / Fraction(xs)), fmt))
           for k in range(K)] for i in range(M)]
    wq = [[Fraction(pins.fp8_nearest(pins.bf16_nearest(Fraction(float(w[j][k])) / Fraction(ws)), fmt))
           for k in range(K)] for j in range(N)]
    scale = Fraction(xs) * Fraction(ws)
    return np.array([[pins.bf16_nearest(scale * sum((xq[i][k] * wq[j][k] for k in range(K)), Fraction(0)))
                      for j in range(N)] for i in range(M)])


def test_mm_matches_brute_force_in_rationals():
    rng = np.random.default_rng(86)
    # scales keep |x / x_s| below E4M3's 448 (an overflow is NaN)
    for M, N, K, xs, ws in [(2, 3, 5, 0.013, 0.021), (3, 2, 9, 0.5, 1.7), (4, 4, 4, 1.1e-2, 3.1e-2)]:
        x = oracle.round_to_bf16(rng.standard_normal((M, K)))
        w = oracle.round_to_bf16(rng.standard_normal((N, K)) * 0.1)
        out, _, _ = oracle.fp8_mm(x, w, xs, ws)
        assert same(out, _brute_force_mm(x, w, xs, ws)), (M, N, K)


def test_backward_of_representable_operands():
    rng = np.random.default_rng(87)
    M, N, K = 6, 5, 12
    gs, xs, ws = 2.0 ** -10, 2.0 ** -2, 2.0 ** 4
    g = representable(rng, (M, N), "e5m2", gs)
    x_f8 = representable(rng, (M, K), "e4m3")
    w_f8 = representable(rng, (N, K), "e4m3")
    gx, gw, g_f8 = oracle.fp8_mm_backward(g, x_f8, w_f8, xs, ws, gs, in_dtype="fp64")
    assert np.array_equal(g_f8 * gs, g)
    # grad_x = g . w and grad_w = g^T . x for the dequantised operands
    assert same(gx, oracle.round_to_bf16(g @ (w_f8 * ws)))
    assert same(gw, oracle.round_to_bf16(g.T @ (x_f8 * xs)))
    assert gx.shape == (M, K) and gw.shape == (N, K)


def test_backward_matches_brute_force_in_rationals():
    """E5M2 gradient quantised by exhaustive search (after the bf16 quotient,
    itself by table search), products summed in rationals, each result
    rounded to bf16 by table search: nothing shared with the oracle."""
    rng = np.random.default_rng(89)
    M, N, K = 3, 4, 5
    gs, xs, ws = 3.7e-6, 0.013, 0.021
    g = oracle.round_to_bf16(rng.standard_normal((M, N)) * 1e-3)
    x_f8 = representable(rng, (M, K), "e4m3")
    w_f8 = representable(rng, (N, K), "e4m3")
    gx, gw, _ = oracle.fp8_mm_backward(g, x_f8, w_f8, xs, ws, gs)
    gq = [[Fraction(pins.fp8_nearest(pins.bf16_nearest(Fraction(float(g[i][j])) / Fraction(gs)), "e5m2"))
           for j in range(N)] for i in range(M)]
    X = [[Fraction(float(v)) for v in row] for row in x_f8]
    W = [[Fraction(float(v)) for v in row] for row in w_f8]
    sx, sw = Fraction(gs) * Fraction(ws), Fraction(gs) * Fraction(xs)
    want_x = np.array([[pins.bf16_nearest(sx * sum((gq[i][n] * W[n][k] for n in range(N)), Fraction(0)))
                        for k in range(K)] for i in range(M)])
    want_w = np.array([[pins.bf16_nearest(sw * sum((gq[m][n] * X[m][k] for m in range(M)), Fraction(0)))
                        for k in range(K)] for n in range(N)])
    assert same(gx, want_x) and same(gw, want_w)


def test_backward_gradients_approximate_the_unquantised_ones():
    """With scales that fill the formats, the FP8 gradients of out = x w^T
    stay within a few per cent of the exact ones (E5M2 keeps 3 significant
    bits, E4M3 4)."""
    rng = np.random.default_rng(88)
    x = rng.standard_normal((32, 64))
    w = rng.standard_normal((48, 64)) * 0.05
    g = rng.standard_normal((32, 48)) * 1e-3
    xs, ws, gs = np.abs(x).max() / 448, np.abs(w).max() / 448, np.abs(g).max() / 57344
    _, x_f8, w_f8 = oracle.fp8_mm(x, w, xs, ws, in_dtype="fp64", out_dtype="fp64")
    gx, gw, _ = oracle.fp8_mm_backward(g, x_f8, w_f8, xs, ws, gs, in_dtype="fp64", out_dtype="fp64")
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(gx, g @ w) < 0.08 and rel(gw, g.T @ x) < 0.08


# ------------------------------------------------------------ planted mistakes
def _run_pins():
    checks = [
        lambda: test_cast_matches_exhaustive_search("e4m3") is None,
        lambda: test_cast_matches_exhaustive_search("e5m2") is None,
        lambda: test_mm_of_representable_operands_is_the_rounded_exact_product() is None,
        lambda: test_mm_matches_brute_force_in_rationals() is None,
        lambda: test_backward_of_representable_operands() is None,
        lambda: test_backward_matches_brute_force_in_rationals() is None,
        lambda: test_quantize_follows_the_page_cast_of_a_bfloat16_tensor() is None,
    ]
    failures = 0
    for check in checks:
        try:
            ok = bool(check())
        except Exception:
            ok = False
        failures += not ok
    return failures


def _ties_away(x, fmt):
    F = of.FP8_FORMATS[fmt]
    x = np.asarray(x, np.float64)
    ax = np.abs(x)
    _, ex = np.frexp(np.where(np.isfinite(ax), ax, 0.0))
    e = np.maximum(ex.astype(np.int64) - 1, F["min_exp"])
    sp = np.ldexp(1.0, (e - F["frac"]).astype(np.int32))
    r = np.floor(ax / sp + 0.5) * sp
    r = np.where(r > F["max"], F["overflow"], r)
    return np.copysign(np.where(np.isfinite(ax), r, np.nan), x)


@pytest.mark.parametrize("mistake", ["no_scale", "e5m2_forward", "no_transpose", "ties_away",
                                     "saturate", "direct_division", "backward_swapped_scales"])
def test_planted_mistakes_are_caught(monkeypatch, mistake):
    assert _run_pins() == 0
    if mistake == "no_scale":
        orig = of._round_out
        monkeypatch.setattr(of, "fp8_mm", lambda x, w, x_s, w_s, in_dtype="bf16", out_dtype="bf16": (
            orig(of.quantize(x, x_s, "e4m3", in_dtype) @ of.quantize(w, w_s, "e4m3", in_dtype).T, out_dtype),
            of.quantize(x, x_s, "e4m3", in_dtype), of.quantize(w, w_s, "e4m3", in_dtype)))
    elif mistake == "e5m2_forward":
        orig_q = of.quantize
        monkeypatch.setattr(of, "quantize", lambda x, s, fmt, in_dtype="bf16": orig_q(x, s, "e5m2", in_dtype))
    elif mistake == "no_transpose":
        orig = of.fp8_mm
        monkeypatch.setattr(of, "fp8_mm", lambda *a, **k: (lambda r: (r[0].T if r[0].shape[0] == r[0].shape[1]
                                                                      else r[0][:, ::-1], r[1], r[2]))(orig(*a, **k)))
    elif mistake == "ties_away":
        monkeypatch.setattr(of, "round_to_fp8", _ties_away)
    elif mistake == "saturate":
        orig_r = of.round_to_fp8
        monkeypatch.setattr(of, "round_to_fp8", lambda x, fmt: np.clip(
            orig_r(np.clip(np.asarray(x, np.float64), -of.FP8_FORMATS[fmt]["max"], of.FP8_FORMATS[fmt]["max"]), fmt),
            -of.FP8_FORMATS[fmt]["max"], of.FP8_FORMATS[fmt]["max"]))
    elif mistake == "direct_division":
        orig_q = of.quantize
        monkeypatch.setattr(of, "quantize", lambda x, s, fmt, in_dtype="bf16": orig_q(x, s, fmt, "fp64"))
    elif mistake == "backward_swapped_scales":
        orig_b = of.fp8_mm_backward
        monkeypatch.setattr(of, "fp8_mm_backward", lambda g, x_f8, w_f8, x_s, w_s, grad_s, **k: orig_b(
            g, x_f8, w_f8, w_s, x_s, grad_s, **k))
    for name in ("round_to_fp8", "quantize", "fp8_mm", "fp8_mm_backward"):
        monkeypatch.setattr(oracle, name, getattr(of, name))
    assert _run_pins() >= 1
