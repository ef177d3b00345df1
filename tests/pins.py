"""Independent references used to pin the CPU oracle (test helpers).

Nothing here calls the oracle: each routine restates a fact about the
Newton-Schulz iteration in a different way, so that a mistake in the oracle
shows up as a disagreement.

* ``closed_form_ns``: every iterate of X' = a X + b (X X^T) X + c (X X^T)^2 X
  keeps the singular vectors of X and maps each singular value s to
  p(s) = a s + b s^3 + c s^5.  So for G = U diag(sigma) V^T,
  NS(G) = U diag(p^steps(sigma / (||G||_F + eps))) V^T, computed here from an
  SVD.  The Frobenius norm is taken from the singular values.
* ``bf16_nearest``: rounding to bfloat16 by search over the table of all
  65,536 bfloat16 bit patterns (nearest value, ties to the even pattern),
  compared in exact rational arithmetic.
* ``ns_bf16_exact``: the bf16-mode iteration in exact rational arithmetic
  (Python ``fractions``) for tiny matrices, rounding with ``bf16_nearest``.
* ``fp8_decode`` / ``fp8_nearest``: the 256 codes of the FP8 formats decoded
  from their bit fields (sign, exponent, fraction), and rounding by search
  over the finite codes in rational arithmetic (nearest value, ties to the
  code with an even fraction, overflow past the midpoint above the largest
  finite value to NaN in E4M3 and to infinity in E5M2).
"""

from decimal import Decimal, getcontext
from fractions import Fraction
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def page_constants():
    with open(os.path.join(GOLDEN, "muon_page_constants.json")) as f:
        return json.load(f)


def scalar_poly(s, steps, coeffs):
    a, b, c = coeffs
    s = np.asarray(s, dtype=np.float64)
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def closed_form_ns(G, steps, coeffs, eps=1e-7):
    G = np.asarray(G, dtype=np.float64)
    U, sig, Vt = np.linalg.svd(G, full_matrices=False)
    fro = np.sqrt(np.sum(sig ** 2))
    return (U * scalar_poly(sig / (fro + eps), steps, coeffs)) @ Vt


# ---------------------------------------------------------------- bf16 table
def _bf16_table():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch.bfloat16).to(torch.float64).numpy()
    pos = np.arange(0, 0x7F80)  # +0 .. largest finite (0x7F7F)
    return vals[pos], pos


_TABLE_VALS, _TABLE_BITS = _bf16_table()
_MAX_FIN = Fraction(float(_TABLE_VALS[-1]))
_OVERFLOW = Fraction(2) ** 128  # where the next pattern (inf) would sit


def bf16_nearest(v):
    """Nearest bfloat16 to the rational (or float) ``v``, ties to even bits."""
    v = Fraction(v)
    sign = -1 if v < 0 else 1
    a = -v if v < 0 else v
    if a > _MAX_FIN:
        mid = (_MAX_FIN + _OVERFLOW) / 2
        # the largest finite pattern 0x7F7F is odd, so the tie goes to inf
        if a >= mid:
            return sign * float("inf")
        return sign * float(_MAX_FIN)
    i = int(np.searchsorted(_TABLE_VALS, float(a), side="right")) - 1
    # float(a) may have rounded; adjust with exact comparisons
    while i + 1 < len(_TABLE_VALS) and Fraction(float(_TABLE_VALS[i + 1])) <= a:
        i += 1
    while i > 0 and Fraction(float(_TABLE_VALS[i])) > a:
        i -= 1
    lo = Fraction(float(_TABLE_VALS[i]))
    if lo == a:
        return sign * float(lo)
    hi = Fraction(float(_TABLE_VALS[i + 1])) if i + 1 < len(_TABLE_VALS) else _OVERFLOW
    dlo, dhi = a - lo, hi - a
    if dlo < dhi:
        r = lo
    elif dhi < dlo:
        r = hi
    else:
        r = lo if _TABLE_BITS[i] % 2 == 0 else hi
    if r == _OVERFLOW:
        return sign * float("inf")
    return sign * float(r)


# ------------------------------------------------- exact bf16-mode iteration
def _matmul(X, Y):
    n, k, m = len(X), len(Y), len(Y[0])
    return [[sum((X[i][t] * Y[t][j] for t in range(k)), Fraction(0)) for j in range(m)]
            for i in range(n)]


def _transpose(X):
    return [list(r) for r in zip(*X)]


def _round(M):
    return [[Fraction(bf16_nearest(v)) for v in row] for row in M]


def ns_bf16_exact(G, steps, coeffs32, eps=1e-7):
    """bf16-mode Newton-Schulz on a tiny matrix in exact arithmetic.

    ``coeffs32`` are the float32 values of (a, b, c).  The normalisation's
    square root is evaluated with 60 significant digits.
    """
    getcontext().prec = 60
    G = [[Fraction(float(v)) for v in row] for row in np.asarray(G, dtype=np.float64)]
    tall = len(G) > len(G[0])
    X = _transpose(G) if tall else G
    Xb = _round(X)
    ss = sum((v * v for row in Xb for v in row), Fraction(0))
    nu = Decimal(ss.numerator).sqrt() / Decimal(ss.denominator).sqrt()
    d = Fraction(nu) + Fraction(eps)
    X = _round([[v / d for v in row] for row in Xb])
    a, b, c = (Fraction(float(x)) for x in coeffs32)
    for _ in range(steps):
        A = _round(_matmul(X, _transpose(X)))
        AA = _matmul(A, A)
        B = _round([[b * A[i][j] + c * AA[i][j] for j in range(len(A))] for i in range(len(A))])
        BX = _matmul(B, X)
        X = _round([[a * X[i][j] + BX[i][j] for j in range(len(X[0]))] for i in range(len(X))])
    if tall:
        X = _transpose(X)
    return np.array([[float(v) for v in row] for row in X], dtype=np.float64)


# ---------------------------------------------------------------- FP8 codes
FP8_FIELDS = {"e4m3": (4, 3, 7), "e5m2": (5, 2, 15)}  # exponent bits, fraction bits, bias


def fp8_decode(code, fmt):
    """Value of the 8-bit code in format ``fmt``, from its bit fields: NaN
    for E4M3's all-ones exponent-and-fraction and E5M2's all-ones exponent
    with a non-zero fraction, infinity for E5M2's all-ones exponent with a
    zero fraction."""
    ebits, fbits, bias = FP8_FIELDS[fmt]
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> fbits) & ((1 << ebits) - 1)
    f = code & ((1 << fbits) - 1)
    if fmt == "e4m3" and e == 15 and f == 7:
        return float("nan")
    if fmt == "e5m2" and e == 31:
        return sign * float("inf") if f == 0 else float("nan")
    if e == 0:
        return sign * f * 2.0 ** (1 - bias - fbits)
    return sign * (1 + f / 2.0 ** fbits) * 2.0 ** (e - bias)


def _fp8_table(fmt):
    vals = [(fp8_decode(c, fmt), c) for c in range(0x80)]
    return sorted((Fraction(v), c) for v, c in vals if np.isfinite(v))


_FP8_TABLES = {f: _fp8_table(f) for f in FP8_FIELDS}
_FP8_NEXT = {"e4m3": Fraction(480), "e5m2": Fraction(65536)}  # where the code above the largest would sit


def fp8_nearest(v, fmt):
    """Nearest value of ``fmt`` to the rational (or float) ``v``."""
    if isinstance(v, float) and not np.isfinite(v):
        if np.isnan(v) or fmt == "e4m3":
            return float("nan")
        return v
    v = Fraction(v)
    sign = -1 if v < 0 else 1
    a = -v if v < 0 else v
    table = _FP8_TABLES[fmt]
    top, top_code = table[-1]
    if a > top:
        # a tie goes to the even code: E4M3's largest finite code 0x7E is
        # even (the tie stays), E5M2's 0x7B is odd (the tie goes to the
        # infinity code 0x7C)
        mid = (top + _FP8_NEXT[fmt]) / 2
        goes_up = a > mid or (a == mid and top_code % 2 == 1)
        if not goes_up:
            return sign * float(top)
        return float("nan") if fmt == "e4m3" else sign * float("inf")
    lo = max((t for t in table if t[0] <= a), key=lambda t: t[0])
    hi = min((t for t in table if t[0] >= a), key=lambda t: t[0])
    if lo[0] == a:
        return sign * float(lo[0])
    dlo, dhi = a - lo[0], hi[0] - a
    if dlo != dhi:
        r = lo if dlo < dhi else hi
    else:
        r = lo if lo[1] % 2 == 0 else hi
    return sign * float(r[0])
