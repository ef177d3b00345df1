"""Muon step, written out plainly on the CPU -- TEST INFRASTRUCTURE ONLY.

Follows the modded-nanogpt walk-through page ("深入解析KellerJordan/
modded-nanogpt中的训练架构与优化技术", reposource.net):

* section "Muon优化器：动量正交化技术": the Muon class, defaults lr=0.02,
  momentum=0.95, nesterov=True, ns_steps=5; ``step()`` does (1) the standard
  momentum update, (2) Newton-Schulz orthogonalisation, (3) the parameter
  update.
* section "Newton-Schulz正交化": ``zeropower_via_newtonschulz5`` with
  (a, b, c) = (3.4445, -4.7750, 2.0315); cast to bfloat16, then ``steps``
  times: A = X X^T, B = b A + c A A, X = a X + B X.

Readings taken where the page is silent (each is also listed in the design
notes of the repository):

1. Momentum (the page shows only the step comment): buf <- mu*buf + g, and
   with Nesterov u <- g + mu*buf using the *updated* buf; without Nesterov
   u <- buf.
2. Orientation: a matrix with more rows than columns (strictly) is
   transposed before iterating so that the Gram matrix is the smaller one,
   and transposed back afterwards.  Square matrices are not transposed.
3. Normalisation: before iterating, X is divided by (||X||_F + 1e-7); the
   epsilon is added to the norm, not to its square.
4. Rounding (bf16 mode): the page iterates on bfloat16 tensors.  Here each of
   the three statements rounds its result once to bfloat16 (round to nearest
   even); the products inside a statement are formed exactly (float64
   accumulation of bfloat16-valued operands).  ``c*A@A`` is the same matrix as
   ``c*(A@A)``; it is not rounded separately.  The normalisation rounds the
   bfloat16 cast of the input first, takes the norm of that bfloat16 tensor in
   float64, and rounds the quotient to bfloat16.
5. Update: p <- p - lr*O, O in the original orientation; no weight decay and
   no shape-dependent scaling of lr (the page names only "parameter update").

Modes:
  "fp64": every step in float64 (the mathematical iteration).
  "bf16": momentum and update in float32 (the precision of the optimizer
          state), Newton-Schulz with the bfloat16 rounding of reading 4 and the
          float32 values of the coefficients.
"""

import numpy as np

from .bf16 import round_to_bf16

#: (a, b, c) of the quintic iteration, as printed in the Newton-Schulz section
NS_COEFFS = (3.4445, -4.7750, 2.0315)
#: epsilon added to the Frobenius norm before dividing (reading 3)
NORM_EPS = 1e-7
#: defaults of the Muon class constructor, as printed in the Muon section
MUON_DEFAULTS = {"lr": 0.02, "momentum": 0.95, "nesterov": True, "ns_steps": 5}

MODES = ("fp64", "bf16")


def _coeffs(mode):
    if mode == "fp64":
        return NS_COEFFS
    # float32 literals widened exactly to float64
    return tuple(float(np.float32(v)) for v in NS_COEFFS)


def momentum_update(g, buf, mu, nesterov, mode="fp64"):
    """Reading 1.  Returns (new_buf, u).  Float64 or float32 arithmetic."""
    dt = np.float64 if mode == "fp64" else np.float32
    g = np.asarray(g).astype(dt)
    buf = np.asarray(buf).astype(dt)
    mu = dt(mu)
    new_buf = (mu * buf + g).astype(dt)
    u = (g + mu * new_buf).astype(dt) if nesterov else new_buf.copy()
    return new_buf, u


def orient(M):
    """Reading 2: (view, transposed?) -- tall matrices are transposed."""
    if M.shape[0] > M.shape[1]:
        return M.T, True
    return M, False


def normalise(G, mode="fp64"):
    """Reading 3 (and 4 for bf16): X0 = G / (||G||_F + 1e-7)."""
    if mode == "fp64":
        X = np.asarray(G, dtype=np.float64)
        return X / (np.sqrt(np.sum(X * X)) + NORM_EPS)
    Xb = round_to_bf16(G)
    nu = np.sqrt(np.sum(Xb * Xb))
    return round_to_bf16(Xb / (nu + NORM_EPS))


def ns_gram(X, mode="fp64"):
    """A = X X^T (rounded to bfloat16 in bf16 mode)."""
    A = X @ X.T
    return A if mode == "fp64" else round_to_bf16(A)


def ns_poly(A, mode="fp64"):
    """B = b A + c A A (one rounding in bf16 mode)."""
    _, b, c = _coeffs(mode)
    B = b * A + c * (A @ A)
    return B if mode == "fp64" else round_to_bf16(B)


def ns_update(B, X, mode="fp64"):
    """X' = a X + B X (one rounding in bf16 mode)."""
    a = _coeffs(mode)[0]
    Xn = a * X + B @ X
    return Xn if mode == "fp64" else round_to_bf16(Xn)


def ns_iteration_parts(X, mode="fp64"):
    """One quintic step: A = X X^T; B = b A + c A A; X' = a X + B X.

    Returns (A, B, X') so that tests can look at the intermediate matrices.
    """
    A = ns_gram(X, mode)
    B = ns_poly(A, mode)
    return A, B, ns_update(B, X, mode)


def ns_iteration(X, mode="fp64"):
    """One quintic step; returns X'."""
    return ns_iteration_parts(X, mode)[2]


def newton_schulz5(G, steps=5, mode="fp64"):
    """zeropower_via_newtonschulz5(G, steps) for one 2-D matrix.

    Returns a float64 array in G's orientation (bfloat16 values in bf16 mode).
    """
    if mode not in MODES:
        raise ValueError(f"mode must be one of {MODES}")
    G = np.asarray(G, dtype=np.float64)
    if G.ndim != 2:
        raise ValueError("G must be 2-D")
    Gv, transposed = orient(G)
    X = normalise(Gv, mode)
    for _ in range(steps):
        X = ns_iteration(X, mode)
    return X.T if transposed else X


def muon_step(p, g, buf, lr, mu, nesterov, ns_steps, mode="fp64"):
    """One Muon step on one matrix.  Returns (new_p, new_buf, O).

    new_p and new_buf are float64 (fp64 mode) or float32 (bf16 mode); O is the
    orthogonalised update in p's orientation.
    """
    dt = np.float64 if mode == "fp64" else np.float32
    new_buf, u = momentum_update(g, buf, mu, nesterov, mode)
    O = newton_schulz5(u, ns_steps, mode)
    p = np.asarray(p).astype(dt)
    new_p = (p - dt(lr) * O.astype(dt)).astype(dt)
    return new_p, new_buf, O
