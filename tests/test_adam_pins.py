"""Pins of the cautious-Adam oracle (oracle.adam) against facts outside it.

Source: the page on the modded-nanogpt record "2026-06-11_RecursiveFromBest"
(lqnn.cn, news/184262), section "3.3 bigram 与 value-embedding 银行上的
C-Optim / 谨慎 Adam" (cautious weight decay: decay only where update and
parameter agree in sign); Adam itself is the textbook algorithm.

Pins:
  * closed forms: first step from zero state (u = g / (|g| + eps)); a
    constant gradient for t steps (bias correction makes m_hat = g and
    v_hat = g^2 exactly, so every step moves p by lr * g / (|g| + eps));
  * library routines for the special cases: torch.optim.AdamW (float64) for
    plain decoupled decay (cautious=False), torch.optim.Adam for wd = 0;
  * hand-worked values of the cautious mask on a small table;
  * the float32 mode against the float64 mode within float32 rounding;
  * planted mistakes in copies of the oracle (dropped bias correction,
    swapped betas, eps under the square root, inverted mask, decay on the
    gradient) each fail at least one pin.
"""

import numpy as np
import pytest
import torch

from oracle.adam import ADAM_DEFAULTS, adam_constants, adam_step, cautious_mask

RNG = np.random.default_rng(31)


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ------------------------------------------------------------ closed forms
def pin_first_step(step_fn):
    p = RNG.standard_normal(500)
    g = RNG.standard_normal(500) * 10.0 ** RNG.uniform(-6, 0, 500)
    z = np.zeros(500)
    lr, eps = 0.01, 1e-8
    p1, m1, v1 = step_fn(p, g, z, z, 1, lr=lr, beta1=0.9, beta2=0.999, eps=eps, wd=0.0)
    ok = rel(p1, p - lr * g / (np.abs(g) + eps)) < 1e-12
    ok &= rel(m1, 0.1 * g) < 1e-12 and rel(v1, 0.001 * g * g) < 1e-12
    return ok


def pin_constant_gradient(step_fn):
    p0 = RNG.standard_normal(300)
    g = RNG.standard_normal(300) * 1e-3
    p, m, v = p0.copy(), np.zeros(300), np.zeros(300)
    lr, eps, b1, b2 = 0.003, 1e-10, 0.8, 0.99
    for t in range(1, 21):
        p, m, v = step_fn(p, g, m, v, t, lr=lr, beta1=b1, beta2=b2, eps=eps, wd=0.0)
    ok = rel(p, p0 - 20 * lr * g / (np.abs(g) + eps)) < 1e-10
    ok &= rel(m, (1 - b1 ** 20) * g) < 1e-12 and rel(v, (1 - b2 ** 20) * g * g) < 1e-12
    return ok


def test_first_step_closed_form():
    assert pin_first_step(adam_step)


def test_constant_gradient_closed_form():
    assert pin_constant_gradient(adam_step)


# ------------------------------------------------------- library routines
def torch_reference(opt_cls, p0, grads, **kw):
    t = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = opt_cls([t], **kw)
    for g in grads:
        t.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
    return t.detach().numpy()


def pin_adamw(step_fn, steps=6):
    p0 = RNG.standard_normal(400) * 0.02
    grads = [RNG.standard_normal(400) * 1e-3 for _ in range(steps)]
    lr, b1, b2, eps, wd = 0.004, 0.9, 0.95, 1e-8, 0.1
    ref = torch_reference(torch.optim.AdamW, p0, grads, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(400), np.zeros(400)
    for t, g in enumerate(grads, start=1):
        p, m, v = step_fn(p, g, m, v, t, lr=lr, beta1=b1, beta2=b2, eps=eps, wd=wd, cautious=False)
    return rel(p, ref) < 1e-12


def pin_adam(step_fn, steps=6):
    p0 = RNG.standard_normal(400)
    grads = [RNG.standard_normal(400) for _ in range(steps)]
    ref = torch_reference(torch.optim.Adam, p0, grads, lr=0.01, betas=(0.9, 0.999), eps=1e-8)
    p, m, v = p0.copy(), np.zeros(400), np.zeros(400)
    for t, g in enumerate(grads, start=1):
        p, m, v = step_fn(p, g, m, v, t, lr=0.01, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, cautious=True)
    return rel(p, ref) < 1e-12


def test_plain_decoupled_decay_is_torch_adamw():
    assert pin_adamw(adam_step)


def test_no_decay_is_torch_adam():
    assert pin_adam(adam_step)


# ------------------------------------------------------- the cautious mask
# p, g with t = 1 and zero state: u = g / (|g| + eps) ~ sign(g)
MASK_P = np.array([1.0, 1.0, -1.0, -1.0, 0.0, 2.0])
MASK_G = np.array([1.0, -1.0, 1.0, -1.0, 1.0, 0.0])
# lr = 0.1, wd = 0.5:   p - 0.1 * (u + 0.5 * p * mask)
MASK_CAUTIOUS = np.array([0.85, 1.1, -1.1, -0.85, -0.1, 2.0])
MASK_PLAIN = np.array([0.85, 1.05, -1.05, -0.85, -0.1, 1.9])


def pin_mask(step_fn):
    z = np.zeros(6)
    c, _, _ = step_fn(MASK_P, MASK_G, z, z, 1, lr=0.1, beta1=0.9, beta2=0.999, eps=1e-12, wd=0.5,
                      cautious=True)
    n, _, _ = step_fn(MASK_P, MASK_G, z, z, 1, lr=0.1, beta1=0.9, beta2=0.999, eps=1e-12, wd=0.5,
                      cautious=False)
    return np.abs(c - MASK_CAUTIOUS).max() < 1e-9 and np.abs(n - MASK_PLAIN).max() < 1e-9


def test_cautious_mask_hand_values():
    assert pin_mask(adam_step)


def test_mask_is_sign_agreement():
    u = np.array([1.0, -1.0, 1.0, -1.0, 0.0, 2.0, -0.0, np.nan, 1e-45])
    p = np.array([2.0, -3.0, -1.0, 1.0, 5.0, 0.0, -1.0, 1.0, 1e-45])
    np.testing.assert_array_equal(cautious_mask(u, p), [True, True, False, False, False, False, False, False, True])


# ------------------------------------------------------ float32 arithmetic
def test_fp32_mode_is_float32_rounding_of_the_definition():
    n = 20000
    p = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    g = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
    m = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
    v = ((RNG.standard_normal(n) * 1e-3) ** 2).astype(np.float32)
    kw = dict(lr=0.008, beta1=0.9, beta2=0.95, eps=1e-10, wd=0.05, cautious=True)
    p32, m32, v32 = adam_step(p, g, m, v, 7, mode="fp32", **kw)
    p64, m64, v64 = adam_step(p, g, m, v, 7, mode="fp64", **kw)
    assert p32.dtype == m32.dtype == v32.dtype == np.float32
    # a few float32 roundings per element
    u32 = np.finfo(np.float32).eps
    assert np.all(np.abs(m32 - m64) <= 4 * u32 * (0.9 * np.abs(m) + 0.1 * np.abs(g)))
    assert np.all(np.abs(v32 - v64) <= 4 * u32 * (0.95 * v + 0.05 * g.astype(np.float64) ** 2))
    # p moves by lr*u ~ lr; p itself carries the float32 rounding of p
    assert np.all(np.abs(p32 - p64) <= 2 * u32 * np.abs(p64) + 16 * u32 * 0.008 * (1 + 0.05 * np.abs(p)))


def test_constants_and_step_count():
    omb1, omb2, bc1, bc2 = adam_constants(0.9, 0.999, 3)
    assert omb1 == pytest.approx(0.1) and omb2 == pytest.approx(0.001)
    assert bc1 == pytest.approx(1 - 0.729) and bc2 == pytest.approx(1 - 0.999 ** 3)
    with pytest.raises(ValueError):
        adam_constants(0.9, 0.999, 0)
    assert ADAM_DEFAULTS["beta1"] == 0.9 and ADAM_DEFAULTS["beta2"] == 0.999


# ------------------------------------------------------ planted mistakes
def _mutant(kind):
    def step(p, g, m, v, t, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, cautious=True, mode="fp64"):
        p, g, m, v = (np.asarray(x, np.float64) for x in (p, g, m, v))
        b1, b2 = (beta2, beta1) if kind == "swapped_betas" else (beta1, beta2)
        gg = g + wd * p if kind == "decay_on_gradient" else g
        m1 = b1 * m + (1 - b1) * gg
        v1 = b2 * v + (1 - b2) * gg * gg
        bc1, bc2 = (1.0, 1.0) if kind == "no_bias_correction" else (1 - b1 ** t, 1 - b2 ** t)
        if kind == "eps_in_sqrt":
            u = (m1 / bc1) / np.sqrt(v1 / bc2 + eps)
        else:
            u = (m1 / bc1) / (np.sqrt(v1 / bc2) + eps)
        mask = cautious_mask(u, p)
        if kind == "inverted_mask":
            mask = ~mask
        decay = 0.0 if kind == "decay_on_gradient" else wd * p
        if cautious:
            decay = np.where(mask, decay, 0.0)
        return p - lr * (u + decay), m1, v1
    return step


@pytest.mark.parametrize("kind", ["no_bias_correction", "swapped_betas", "eps_in_sqrt", "inverted_mask",
                                  "decay_on_gradient"])
def test_planted_mistakes_are_caught(kind):
    step = _mutant(kind)
    pins = [pin_first_step, pin_constant_gradient, pin_adamw, pin_adam, pin_mask]
    failed = 0
    for pin in pins:
        try:
            failed += not pin(step)
        except Exception:
            failed += 1
    assert failed >= 1, kind


def test_unmutated_copy_passes_every_pin():
    step = _mutant("none")
    assert all(pin(step) for pin in [pin_first_step, pin_constant_gradient, pin_adamw, pin_adam, pin_mask])
