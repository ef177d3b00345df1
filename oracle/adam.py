"""Adam step with cautious weight decay, written out plainly on the CPU --
TEST INFRASTRUCTURE ONLY.

The page on the modded-nanogpt record "2026-06-11_RecursiveFromBest"
(lqnn.cn, news/184262), section "3.3 bigram 与 value-embedding 银行上的
C-Optim / 谨慎 Adam", describes the optimizer of the embedding-type banks
(bigram table, value embeddings): Adam, with weight decay applied
"cautiously" -- only where the update and the parameter have the same sign.
It quotes the rule as a mask that is true where update * p is positive, the
decay term being added to the update under that mask.

Readings taken where the page is silent (also listed in the design notes):

1. Adam itself is the textbook algorithm (Kingma & Ba, "Adam: A Method for
   Stochastic Optimization", Algorithm 1): first and second moment EMAs with
   bias correction, update m_hat / (sqrt(v_hat) + eps), t counted from 1.
2. Weight decay is decoupled (the decay term is added to the update, not to
   the gradient), with the caller's coefficient ``wd`` as given; the step
   subtracts lr times the (update + masked decay).
3. "update * p > 0" is read exactly: update and p both non-zero and of the
   same sign (so an update or parameter of 0 gets no decay).
4. ``cautious=False`` applies the decay everywhere (plain decoupled weight
   decay), ``wd = 0`` gives plain Adam.
5. Dense: every element is updated every step (the page's row-sparse
   variant, which skips rows without gradient, is not restated).

Per element, with bc1 = 1 - beta1^t and bc2 = 1 - beta2^t:
    m   <- beta1 * m + (1 - beta1) * g
    v   <- beta2 * v + (1 - beta2) * g^2
    u    = (m / bc1) / (sqrt(v / bc2) + eps)
    mask = (u > 0 and p > 0) or (u < 0 and p < 0)       (cautious)
    p   <- p - lr * (u + wd * p * mask)

Modes:
  "fp64": every operation in float64 (the definition).
  "fp32": every operation one IEEE float32 operation in the order written
          above (no fused multiply-add); the hyper-parameters are rounded to
          float32 first, and the constants (1 - beta1), (1 - beta2), bc1 and
          bc2 are formed in float64 from the rounded betas and rounded once
          to float32 -- the arithmetic the GPU kernel performs.
"""

import numpy as np

#: hyper-parameter defaults of the textbook algorithm (lr, beta1, beta2, eps)
ADAM_DEFAULTS = {"lr": 1e-3, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8}


def adam_constants(beta1, beta2, step):
    """(1 - beta1, 1 - beta2, 1 - beta1^t, 1 - beta2^t) in float64."""
    if step < 1:
        raise ValueError("step counts from 1")
    return 1.0 - beta1, 1.0 - beta2, 1.0 - beta1 ** step, 1.0 - beta2 ** step


def cautious_mask(u, p):
    """Reading 3: u and p non-zero with the same sign."""
    return ((u > 0) & (p > 0)) | ((u < 0) & (p < 0))


def adam_step(p, g, m, v, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, cautious=True,
              mode="fp64"):
    """One step for one tensor; returns (new_p, new_m, new_v).  Inputs are
    not modified.  ``g`` may be any float dtype (its values are used exactly)."""
    if mode == "fp64":
        f = np.float64
    elif mode == "fp32":
        f = np.float32
    else:
        raise ValueError(mode)
    if mode == "fp32":
        beta1, beta2 = float(np.float32(beta1)), float(np.float32(beta2))
    omb1, omb2, bc1, bc2 = (f(c) for c in adam_constants(beta1, beta2, step))
    b1, b2, lr_, eps_, wd_ = f(beta1), f(beta2), f(lr), f(eps), f(wd)
    p = np.asarray(p, dtype=f)
    g = np.asarray(g, dtype=f)
    m = np.asarray(m, dtype=f)
    v = np.asarray(v, dtype=f)
    m1 = b1 * m + omb1 * g
    v1 = b2 * v + omb2 * (g * g)
    u = (m1 / bc1) / (np.sqrt(v1 / bc2) + eps_)
    decay = wd_ * p
    if cautious:
        decay = np.where(cautious_mask(u, p), decay, f(0))
    p1 = p - lr_ * (u + decay)
    return p1, m1, v1
