"""FP8 scaled matrix multiplication, written out plainly on the CPU --
TEST INFRASTRUCTURE ONLY.

The page "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术"
(reposource.net), section "自定义FP8矩阵乘法实现", describes modded-nanogpt's
custom op ``nanogpt::mm``:

  forward   the input x and the weight w are divided by their scales x_s and
            w_s and cast to FP8 E4M3; the product x_f8 · w_f8^T is formed
            and returned in BF16 ("计算结果保持为BF16精度"), together with
            x_f8 and w_f8;
  backward  (subsection "反向传播优化") the output gradient g is divided by
            grad_s and cast to FP8 E5M2 ("更大的动态范围"); the input gradient
            is g_f8 · w_f8 and the weight gradient g_f8^T · x_f8.

Readings taken where the page is silent or abridged (also listed in the
design notes):

1. Scales.  The page's listing passes no scales to the matmul (the snippets
   are abridged).  The product is read as carrying them back: out =
   (x_s * w_s) * (x_f8 · w_f8^T), grad_x = (grad_s * w_s) * (g_f8 · w_f8),
   grad_w = (grad_s * x_s) * (g_f8^T · x_f8), so that each result
   approximates the unquantised product.
2. The division before the cast happens in the input's precision: a bf16
   input's quotient is rounded to bf16, then cast to FP8 (two roundings, as
   dividing a bf16 tensor by a Python float does); an fp32 input's quotient
   is rounded to fp32.
3. The FP8 casts are the formats' own definitions (OCP 8-bit floating point,
   E4M3 "fn" without infinities and E5M2): round to nearest, ties to even,
   with subnormals; a result beyond the largest finite value becomes NaN in
   E4M3 (it has no infinity) and an infinity in E5M2.  NaN stays NaN; an
   infinite input becomes NaN in E4M3 and stays infinite in E5M2.
4. Products are summed in float64 by the library matmul and the scaled sum
   is rounded once to the output type; the backward results are read as
   BF16 like the forward's.  E4M3 products are multiples of 2**-18 below
   2**17.6, so the forward's float64 sums are exact up to K = 2**17; the
   backward's E5M2 x E4M3 sums can round only below 2**-53 relative, far
   under the output's rounding.

Formats (bias b, f fraction bits, largest finite M, smallest subnormal):
  E4M3 (fn)  b = 7,  f = 3,  M = 448   = 1.75 * 2**8,   2**-9
  E5M2       b = 15, f = 2,  M = 57344 = 1.75 * 2**15,  2**-16
"""

import numpy as np

from .bf16 import round_to_bf16

#: per format: fraction bits, smallest normal exponent, largest finite value,
#: value a positive overflow becomes
FP8_FORMATS = {
    "e4m3": {"frac": 3, "min_exp": -6, "max": 448.0, "overflow": np.nan},
    "e5m2": {"frac": 2, "min_exp": -14, "max": 57344.0, "overflow": np.inf},
}


def round_to_fp8(x, fmt):
    """Round every element of ``x`` to the nearest value of FP8 format
    ``fmt`` ("e4m3" or "e5m2").  Returns float64 values of that format.

    The grid spacing at |x| is 2**(e - f), e = floor(log2 |x|) clamped to the
    smallest normal exponent (subnormals share the spacing of the smallest
    binade); |x| / spacing is rounded half to even, which is exact in float64
    for any float64 input because the division is by a power of two."""
    F = FP8_FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    finite = np.isfinite(ax)
    safe = np.where(finite, ax, 0.0)
    _, ex = np.frexp(safe)  # safe = m * 2**ex, m in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, F["min_exp"])
    spacing = np.ldexp(1.0, (e - F["frac"]).astype(np.int32))
    r = np.rint(safe / spacing) * spacing
    r = np.where(r > F["max"], F["overflow"], r)
    # infinities: E5M2 keeps them, E4M3 has none (NaN); NaN stays NaN
    r = np.where(finite, r, np.where(np.isinf(ax), F["overflow"], np.nan))
    return np.copysign(r, x)


def _round_to_fp32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _round_out(v, out_dtype):
    if out_dtype == "bf16":
        return round_to_bf16(v)
    if out_dtype == "fp32":
        return _round_to_fp32(v)
    if out_dtype == "fp64":
        return np.asarray(v, dtype=np.float64)
    raise ValueError(out_dtype)


def quantize(x, scale, fmt, in_dtype="bf16"):
    """FP8 value of x / scale (reading 2: the quotient rounded to the input's
    precision first).  x holds values of ``in_dtype`` ("bf16", "fp32" or
    "fp64")."""
    q = np.asarray(x, dtype=np.float64) / np.float64(scale)
    if in_dtype == "bf16":
        q = round_to_bf16(q)
    elif in_dtype == "fp32":
        q = _round_to_fp32(q)
    elif in_dtype != "fp64":
        raise ValueError(in_dtype)
    return round_to_fp8(q, fmt)


def fp8_mm(x, w, x_s, w_s, in_dtype="bf16", out_dtype="bf16"):
    """Forward of the page's FP8 matmul: x (M x K), w (N x K) ->
    (out (M x N), x_f8, w_f8), out = round((x_s * w_s) * (x_f8 . w_f8^T))."""
    x_f8 = quantize(x, x_s, "e4m3", in_dtype)
    w_f8 = quantize(w, w_s, "e4m3", in_dtype)
    acc = x_f8 @ w_f8.T
    out = _round_out(acc * (np.float64(x_s) * np.float64(w_s)), out_dtype)
    return out, x_f8, w_f8


def fp8_mm_backward(g, x_f8, w_f8, x_s, w_s, grad_s, in_dtype="bf16", out_dtype="bf16"):
    """Backward of the page's FP8 matmul: g (M x N) is cast to E5M2 with
    scale grad_s; grad_x (M x K) = (grad_s * w_s) * (g_f8 . w_f8) and
    grad_w (N x K) = (grad_s * x_s) * (g_f8^T . x_f8), each rounded once."""
    g_f8 = quantize(g, grad_s, "e5m2", in_dtype)
    grad_x = _round_out((g_f8 @ w_f8) * (np.float64(grad_s) * np.float64(w_s)), out_dtype)
    grad_w = _round_out((g_f8.T @ x_f8) * (np.float64(grad_s) * np.float64(x_s)), out_dtype)
    return grad_x, grad_w, g_f8
