"""GPU parity of adam_step (Adam with cautious weight decay) against the
oracle, through the C ABI.

The kernel performs one IEEE float32 operation per step of the formula, in
the oracle's order and without fused multiply-adds, so it must equal the
oracle's "fp32" mode bit for bit; the "fp64" mode (the definition) bounds
the float32 rounding.  Cases: ragged sizes around the vector width and the
block size, bf16 and fp32 gradients, cautious and plain decay, no decay,
several chained steps, the sign cases of the mask, non-finite values, and
the full embedding-type bank (4 x 50304 x 768) compared in full.
"""

import numpy as np
import pytest
import torch

from newton_schulz_08_gb300 import inputs, muon
from oracle import adam_step as oracle_adam
from oracle import round_to_bf16

pytestmark = pytest.mark.gpu

HP = dict(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-10)


def upload(state, g_bf16):
    p, m, v, g = state
    dev = torch.device("cuda")
    gt = torch.from_numpy(g).to(dev)
    return (torch.from_numpy(p).to(dev), gt.to(torch.bfloat16) if g_bf16 else gt,
            torch.from_numpy(m).to(dev), torch.from_numpy(v).to(dev))


def run_gpu(states, step, g_bf16=True, wd=0.05, cautious=True, **hp):
    kw = dict(HP, **hp)
    T = [upload(s, g_bf16) for s in states]
    muon.adam_step([t[0] for t in T], [t[1] for t in T], [t[2] for t in T], [t[3] for t in T], step,
                   lr=kw["lr"], beta1=kw["beta1"], beta2=kw["beta2"], eps=kw["eps"], weight_decay=wd,
                   cautious=cautious)
    torch.cuda.synchronize()
    return [tuple(x.cpu().numpy() for x in (t[0], t[2], t[3])) for t in T]


def run_oracle(state, step, g_bf16=True, wd=0.05, cautious=True, mode="fp32", **hp):
    kw = dict(HP, **hp)
    p, m, v, g = state
    gq = round_to_bf16(g) if g_bf16 else g
    return oracle_adam(p, gq, m, v, step, lr=kw["lr"], beta1=kw["beta1"], beta2=kw["beta2"], eps=kw["eps"],
                       wd=wd, cautious=cautious, mode=mode)


def states_of(sizes, seed_offset=0):
    return [inputs.adam_state((n,), seed_offset + i) for i, n in enumerate(sizes)]


RAGGED = [1, 3, 4, 5, 1023, 1024, 1025, 8191, 8192, 8193, 2 * 8192 + 7, 100_003]


def assert_bit_exact(got, want):
    for name, a, b in zip(("p", "m", "v"), got, want):
        b = np.asarray(b, np.float32)
        assert a.dtype == np.float32 and a.shape == b.shape
        same = (a.view(np.uint32) == b.view(np.uint32))
        assert same.all(), f"{name}: {int((~same).sum())} of {a.size} differ, first at {np.argmax(~same)}"


@pytest.mark.parametrize("g_bf16", [True, False])
@pytest.mark.parametrize("cautious,wd", [(True, 0.05), (False, 0.05), (True, 0.0)])
def test_bit_exact_against_float32_oracle(g_bf16, cautious, wd):
    states = states_of(RAGGED)
    got = run_gpu(states, inputs.ADAM_STEP, g_bf16, wd, cautious)
    for s, gpu in zip(states, got):
        assert_bit_exact(gpu, run_oracle(s, inputs.ADAM_STEP, g_bf16, wd, cautious))


def test_three_chained_steps_from_zero_state():
    sizes = [777, 8192 * 3 + 1, 40_000]
    base = states_of(sizes, 50)
    dev_states = [(p, np.zeros_like(p), np.zeros_like(p), g) for p, _, _, g in base]
    ref = [(p.copy(), np.zeros_like(p), np.zeros_like(p)) for p, _, _, _ in base]
    dev = torch.device("cuda")
    P = [torch.from_numpy(s[0]).to(dev) for s in dev_states]
    M = [torch.zeros_like(x) for x in P]
    V = [torch.zeros_like(x) for x in P]
    for step in (1, 2, 3):
        grads = [inputs.adam_state((n,), 50 + i, step=step)[3] for i, n in enumerate(sizes)]
        G = [torch.from_numpy(g).to(dev).to(torch.bfloat16) for g in grads]
        muon.adam_step(P, G, M, V, step, weight_decay=0.1, cautious=True, **{k: HP[k] for k in HP})
        ref = [oracle_adam(r[0], round_to_bf16(g), r[1], r[2], step, wd=0.1, cautious=True, mode="fp32", **HP)
               for r, g in zip(ref, grads)]
    torch.cuda.synchronize()
    for i in range(len(sizes)):
        assert_bit_exact((P[i].cpu().numpy(), M[i].cpu().numpy(), V[i].cpu().numpy()), ref[i])


def test_float64_definition_within_float32_rounding():
    states = states_of([50_000, 8193])
    got = run_gpu(states, 7)
    for s, (p, m, v) in zip(states, got):
        P, Mm, Vv = run_oracle(s, 7, mode="fp64")
        dp_gpu, dp_ref = p.astype(np.float64) - s[0], P - s[0]
        assert np.linalg.norm(dp_gpu - dp_ref) <= 1e-5 * np.linalg.norm(dp_ref)
        assert np.abs(m - Mm).max() <= 1e-6 * np.abs(Mm).max()
        assert np.abs(v - Vv).max() <= 1e-6 * np.abs(Vv).max()


def test_mask_sign_cases():
    # t = 1 from zero state: u = g / (|g| + eps) has the sign of g
    p = np.array([1.0, 1.0, -1.0, -1.0, 0.0, 2.0, -0.0, 0.5], np.float32)
    g = np.array([1.0, -1.0, 1.0, -1.0, 1.0, 0.0, -1.0, 0.0], np.float32)
    z = np.zeros_like(p)
    for cautious in (True, False):
        got = run_gpu([(p, z, z, g)], 1, g_bf16=False, wd=0.5, cautious=cautious, lr=0.1, eps=1e-12)[0]
        assert_bit_exact(got, run_oracle((p, z, z, g), 1, False, 0.5, cautious, lr=0.1, eps=1e-12))
    want = np.array([0.85, 1.1, -1.1, -0.85, -0.1, 2.0, 0.1, 0.5], np.float32)
    got = run_gpu([(p, z, z, g)], 1, g_bf16=False, wd=0.5, cautious=True, lr=0.1, eps=1e-12)[0][0]
    np.testing.assert_allclose(got, want, atol=1e-6)


def test_non_finite_values_stay_local():
    p, m, v, g = inputs.adam_state((4096,), 90)
    g = g.copy()
    g[17] = np.nan
    g[4000] = np.inf
    got = run_gpu([(p, m, v, g)], 3, g_bf16=False)[0]
    assert np.isnan(got[0][17]) and not np.isfinite(got[0][4000])
    finite = np.ones(4096, bool)
    finite[[17, 4000]] = False
    assert np.isfinite(got[0][finite]).all()
    with np.errstate(invalid="ignore"):
        want = run_oracle((p, m, v, g), 3, False)
    np.testing.assert_array_equal(got[0][finite].view(np.uint32), want[0][finite].view(np.uint32))


def test_full_embedding_bank_bit_exact():
    shapes = inputs.adam_bank_shapes()
    states = [inputs.adam_state(s, i) for i, s in enumerate(shapes)]
    got = run_gpu(states, inputs.ADAM_STEP, True, 0.05, True)
    for s, gpu in zip(states, got):
        assert_bit_exact(gpu, run_oracle(s, inputs.ADAM_STEP, True, 0.05, True))
