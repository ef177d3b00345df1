"""Pins of the CPU oracle against facts fixed outside it (CPU only).

Each test checks the oracle against something it does not compute itself:
the constants printed on the page (golden fixture), the SVD closed form of
the iteration, exact invariants, exact rational brute force, and an
independent bfloat16 rounding routine.  ``test_planted_mistakes`` shows that
plausible mistakes in the oracle fail at least one of these pins.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import oracle.muon as om
from tests import pins

CONST = pins.page_constants()
COEFFS = tuple(CONST["ns_coeffs"])
COEFFS32 = tuple(float(np.float32(v)) for v in COEFFS)


def rel(x, y):
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


# ------------------------------------------------------------- constants
def test_constants_match_page():
    assert oracle.NS_COEFFS == COEFFS
    assert oracle.MUON_DEFAULTS == CONST["defaults"]
    assert oracle.NORM_EPS == 1e-7


# ------------------------------------------------------------- bf16 rounding
def _edge_f32():
    f = np.finfo(np.float32)
    vals = [0.0, -0.0, 1.0, -1.0, f.max, -f.max, f.tiny, -f.tiny, 1e-45, -1e-45,
            np.inf, -np.inf, 3.3895313892515355e38, 3.3961e38, 1.00390625, 1.01171875,
            1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 2 ** -126 * 1.5, 2 ** -133, 2 ** -134, 3 * 2 ** -135]
    return np.array(vals, dtype=np.float32)


def test_bf16_rounding_matches_torch_on_float32():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    # ties: low 16 bits exactly 0x8000
    ties = ((rng.integers(0, 2 ** 16, size=20000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties[~np.isnan(ties)], _edge_f32()])
    ours = oracle.round_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all(), x[~same][:10]
    assert np.array_equal(np.signbit(ours), np.signbit(ref))
    assert np.isnan(oracle.round_to_bf16(np.array([np.nan])))[0]


def test_bf16_rounding_float64_against_table_search():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000),
        # exact float64 midpoints between neighbouring bf16 values
        (1 + (2 * rng.integers(0, 128, 500) + 1) / 256.0) * 2.0 ** rng.integers(-120, 120, 500),
        # just above / below the midpoints
        np.nextafter(1 + 1 / 256.0, 2.0) * np.ones(1), np.nextafter(1 + 1 / 256.0, 0.0) * np.ones(1),
        np.array([3.3961e38, 3.39e38, 3.4e38, 2.0 ** -134, 2.0 ** -133 * 1.5, 2.0 ** -140]),
    ])
    ours = oracle.round_to_bf16(x)
    ref = np.array([pins.bf16_nearest(float(v)) for v in x])
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------- fp64 closed form
SHAPES = [(1, 1), (1, 7), (7, 1), (2, 2), (5, 5), (8, 13), (13, 8), (16, 64), (64, 16), (40, 40), (33, 70)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("steps", [0, 1, 2, 5, 7])
def test_fp64_matches_svd_closed_form(shape, steps):
    rng = np.random.default_rng(hash((shape, steps)) % 2 ** 32)
    G = rng.standard_normal(shape) * 3.0
    got = oracle.newton_schulz5(G, steps, "fp64")
    want = pins.closed_form_ns(G, steps, COEFFS)
    assert got.shape == G.shape
    assert rel(got, want) <= 1e-10


@pytest.mark.parametrize("shape,r", [((24, 40), 3), ((40, 24), 5), ((32, 32), 1)])
def test_fp64_closed_form_rank_deficient(shape, r):
    rng = np.random.default_rng(7)
    G = rng.standard_normal((shape[0], r)) @ rng.standard_normal((r, shape[1]))
    got = oracle.newton_schulz5(G, 5, "fp64")
    assert rel(got, pins.closed_form_ns(G, 5, COEFFS)) <= 1e-10


# ------------------------------------------------------------- invariants
def test_transpose_invariant():
    rng = np.random.default_rng(2)
    for shape in [(12, 30), (30, 12), (17, 17)]:
        G = rng.standard_normal(shape)
        assert np.abs(oracle.newton_schulz5(G.T, 5) - oracle.newton_schulz5(G, 5).T).max() <= 1e-12


def test_scale_invariant():
    rng = np.random.default_rng(3)
    G = rng.standard_normal((20, 36))
    fro = np.linalg.norm(G)
    # exact invariance once the epsilon is negligible against the norm
    big = oracle.newton_schulz5(1e6 * G, 5)
    assert rel(oracle.newton_schulz5(1e9 * G, 5), big) <= 1e-12
    # otherwise the epsilon changes the scale of X0 by about
    # (eps/||G||) * |1/alpha - 1|; the output moves by at most a small multiple
    base = oracle.newton_schulz5(G, 5)
    for alpha in [1e-3, 0.5, 7.0, 1e3]:
        bound = 3.0 * (1e-7 / fro) * abs(1.0 / alpha - 1.0) + 1e-13
        assert rel(oracle.newton_schulz5(alpha * G, 5), base) <= bound


def test_rank_r_output_keeps_subspaces():
    rng = np.random.default_rng(4)
    r = 4
    G = rng.standard_normal((30, r)) @ rng.standard_normal((r, 50))
    O = oracle.newton_schulz5(G, 5)
    U, s, Vt = np.linalg.svd(G)
    so = np.linalg.svd(O, compute_uv=False)
    assert so[r:].max() <= 1e-12 * so[0]
    Ur, Vr = U[:, :r], Vt[:r].T
    # O lives in span(U_r) x span(V_r)
    assert np.linalg.norm(O - Ur @ (Ur.T @ O) @ Vr @ Vr.T) <= 1e-10 * np.linalg.norm(O)


@pytest.mark.parametrize("n", [8, 64, 128])
def test_orthogonal_input_gives_flat_spectrum(n):
    rng = np.random.default_rng(n)
    Q, R = np.linalg.qr(rng.standard_normal((n, n)))
    O = oracle.newton_schulz5(Q, 5)
    want = float(pins.scalar_poly(1.0 / (math.sqrt(n) + 1e-7), 5, COEFFS))
    s = np.linalg.svd(O, compute_uv=False)
    assert np.abs(s - want).max() <= 1e-12


def test_orthogonal_values_reported_in_design():
    # p^5(1/(sqrt(n)+1e-7)) for the square sizes the workloads use
    table = {128: 0.722762174, 512: 0.808606867, 768: 1.083594575,
             1024: 1.132923611, 1600: 0.933209462, 4096: 0.902525754}
    for n, v in table.items():
        assert abs(float(pins.scalar_poly(1.0 / (math.sqrt(n) + 1e-7), 5, COEFFS)) - v) <= 1e-9


# ------------------------------------------------------------- tiny brute force
def test_one_by_one_and_zero():
    for g in [2.5, -0.75, 1e-3]:
        O = oracle.newton_schulz5(np.array([[g]]), 5)
        s = abs(g) / (abs(g) + 1e-7)
        want = math.copysign(float(pins.scalar_poly(s, 5, COEFFS)), g)
        assert abs(O[0, 0] - want) <= 1e-12
    for shape in [(3, 5), (5, 3), (1, 1)]:
        for mode in ("fp64", "bf16"):
            assert not oracle.newton_schulz5(np.zeros(shape), 5, mode).any()


def test_row_vector():
    g = np.array([[3.0, -4.0, 12.0]])  # norm 13
    O = oracle.newton_schulz5(g, 5)
    want = float(pins.scalar_poly(13.0 / (13.0 + 1e-7), 5, COEFFS)) * g / 13.0
    assert np.abs(O - want).max() <= 1e-12


@pytest.mark.parametrize("shape", [(1, 1), (2, 3), (3, 2), (4, 4), (3, 5)])
@pytest.mark.parametrize("steps", [0, 1, 5])
def test_bf16_mode_matches_exact_rational_brute_force(shape, steps):
    rng = np.random.default_rng(hash((shape, steps, "b")) % 2 ** 32)
    G = rng.standard_normal(shape).astype(np.float32).astype(np.float64)
    got = oracle.newton_schulz5(G, steps, "bf16")
    want = pins.ns_bf16_exact(G, steps, COEFFS32)
    assert np.array_equal(got, want), (got, want)


def test_bf16_mode_values_are_bf16():
    rng = np.random.default_rng(9)
    O = oracle.newton_schulz5(rng.standard_normal((16, 48)), 5, "bf16")
    assert np.array_equal(O, oracle.round_to_bf16(O))


def test_bf16_mode_close_to_fp64():
    rng = np.random.default_rng(10)
    G = rng.standard_normal((64, 256))
    assert rel(oracle.newton_schulz5(G, 5, "bf16"), oracle.newton_schulz5(G, 5, "fp64")) <= 3e-2


# ------------------------------------------------------------- momentum / step
def test_momentum_by_hand():
    # g = 1, buf = 4, mu = 1/2: buf' = 2 + 1 = 3; Nesterov u = 1 + 3/2
    nb, u = oracle.momentum_update(np.array([1.0]), np.array([4.0]), 0.5, True)
    assert nb[0] == 3.0 and u[0] == 2.5
    nb, u = oracle.momentum_update(np.array([1.0]), np.array([4.0]), 0.5, False)
    assert nb[0] == 3.0 and u[0] == 3.0
    nb, u = oracle.momentum_update(np.array([1.0], np.float32), np.array([4.0], np.float32), 0.5, True, "bf16")
    assert nb.dtype == np.float32 and nb[0] == 3.0 and u[0] == 2.5
    # zero buffer: u = (1 + mu) g
    g = np.array([0.3, -1.2])
    nb, u = oracle.momentum_update(g, np.zeros(2), 0.95, True)
    assert np.allclose(u, 1.95 * g, rtol=0, atol=1e-15) and np.array_equal(nb, g)


def test_muon_step_one_by_one():
    p, g, buf = np.array([[1.0]]), np.array([[2.0]]), np.zeros((1, 1))
    new_p, new_buf, O = oracle.muon_step(p, g, buf, 0.02, 0.95, True, 5, "fp64")
    u = 2.0 + 0.95 * 2.0
    o = float(pins.scalar_poly(u / (u + 1e-7), 5, COEFFS))
    assert abs(O[0, 0] - o) <= 1e-12
    assert abs(new_p[0, 0] - (1.0 - 0.02 * o)) <= 1e-12
    assert new_buf[0, 0] == 2.0


def test_muon_step_tall_orientation():
    rng = np.random.default_rng(11)
    p = rng.standard_normal((9, 4)) * 0.02
    g = rng.standard_normal((9, 4))
    buf = rng.standard_normal((9, 4)) * 0.1
    new_p, new_buf, O = oracle.muon_step(p, g, buf, 0.02, 0.95, True, 5, "fp64")
    u = g + 0.95 * (0.95 * buf + g)
    assert rel(O, pins.closed_form_ns(u, 5, COEFFS)) <= 1e-10
    assert np.allclose(new_p, p - 0.02 * O, rtol=0, atol=1e-15)


# ------------------------------------------------------------- planted mistakes
def _coeffs_a(mode):
    return om._coeffs(mode)[0]


def _double_round_poly(A):
    _, b, c = om._coeffs("bf16")
    AA = oracle.round_to_bf16(A @ A)  # extra rounding of A A
    return oracle.round_to_bf16(b * A + c * AA)


def _eps_on_square(G, mode="fp64"):
    X = np.asarray(G, dtype=np.float64)
    return X / np.sqrt(np.sum(X * X) + 1e-7)


def _run_pins():
    """The subset of pins that must catch each planted mistake.

    Returns how many pins failed (an exception counts as a failure).
    """
    checks = []
    rng = np.random.default_rng(123)
    for shape in [(6, 6), (5, 9), (9, 5)]:
        G = rng.standard_normal(shape)
        checks.append(lambda G=G: rel(oracle.newton_schulz5(G, 5), pins.closed_form_ns(G, 5, COEFFS)) <= 1e-10)
    for shape in [(3, 3), (2, 4)]:
        G = rng.standard_normal(shape).astype(np.float32).astype(np.float64)
        checks.append(lambda G=G: np.array_equal(oracle.newton_schulz5(G, 2, "bf16"),
                                                 pins.ns_bf16_exact(G, 2, COEFFS32)))
    checks.append(lambda: oracle.momentum_update(np.array([1.0]), np.array([4.0]), 0.5, True)[1][0] == 2.5)
    failures = 0
    for check in checks:
        try:
            ok = bool(check())
        except Exception:
            ok = False
        failures += not ok
    return failures


@pytest.mark.parametrize("mistake", ["b_sign", "drop_c", "update_order", "eps_on_square",
                                     "extra_rounding", "no_nesterov"])
def test_planted_mistakes_are_caught(monkeypatch, mistake):
    assert _run_pins() == 0
    if mistake == "b_sign":
        monkeypatch.setattr(om, "NS_COEFFS", (COEFFS[0], -COEFFS[1], COEFFS[2]))
    elif mistake == "drop_c":
        monkeypatch.setattr(om, "NS_COEFFS", (COEFFS[0], COEFFS[1], 0.0))
    elif mistake == "update_order":
        monkeypatch.setattr(om, "ns_update", lambda B, X, mode="fp64": _coeffs_a(mode) * X + X @ B)
    elif mistake == "eps_on_square":
        monkeypatch.setattr(om, "normalise", _eps_on_square)
    elif mistake == "extra_rounding":
        orig = om.ns_poly
        monkeypatch.setattr(om, "ns_poly", lambda A, mode="fp64": orig(A, mode) if mode == "fp64"
                            else _double_round_poly(A))
    elif mistake == "no_nesterov":
        orig_m = om.momentum_update
        monkeypatch.setattr(om, "momentum_update", lambda g, b, mu, nest, mode="fp64": orig_m(g, b, mu, False, mode))
        monkeypatch.setattr(oracle, "momentum_update", om.momentum_update)
    assert _run_pins() >= 1
