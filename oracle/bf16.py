"""bfloat16 rounding for the CPU oracle -- TEST INFRASTRUCTURE ONLY.

The Newton-Schulz section of the modded-nanogpt walk-through page casts the
input with ``G.bfloat16()`` and then iterates on bfloat16 tensors.  bfloat16 is
an IEEE-754-style binary format with 1 sign bit, 8 exponent bits (the same
range as float32) and 7 stored fraction bits (8 significant bits).

``round_to_bf16`` restates round-to-nearest, ties-to-even directly from that
definition: the grid spacing at |x| is 2**(e-7) with e = floor(log2|x|),
clamped to the smallest normal exponent -126 so that subnormals share the
spacing 2**-133.  Scaling by a power of two is exact in float64, so
``rint(|x| / spacing) * spacing`` is the correctly rounded value.  Results
beyond the largest finite bfloat16 become infinities; NaN stays NaN.

The routine works on float64 input directly (one rounding), so it never
suffers the double rounding of a float64 -> float32 -> bfloat16 chain.
"""

import numpy as np

#: largest finite bfloat16: (2 - 2**-7) * 2**127
BF16_MAX = float((2.0 - 2.0 ** -7) * 2.0 ** 127)

_MIN_NORMAL_EXP = -126
_FRACTION_BITS = 7


def round_to_bf16(x):
    """Round every element of ``x`` to the nearest bfloat16 value.

    Returns a float64 array holding bfloat16-representable values (so later
    float64 arithmetic on them is exact for products of two such values).
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    finite = np.isfinite(ax)
    safe = np.where(finite, ax, 0.0)
    # frexp: safe = m * 2**ex with m in [0.5, 1), so floor(log2(safe)) = ex - 1.
    _, ex = np.frexp(safe)
    e = np.maximum(ex.astype(np.int64) - 1, _MIN_NORMAL_EXP)
    spacing = np.ldexp(1.0, (e - _FRACTION_BITS).astype(np.int32))
    q = np.rint(safe / spacing)  # numpy rint rounds halves to even
    r = q * spacing
    r = np.where(r > BF16_MAX, np.inf, r)
    r = np.where(finite, r, ax)  # +inf stays inf, NaN stays NaN
    return np.copysign(r, x)
