"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark uses (one muon_step / ns5_bank call over the whole bank).

The GPU processes every matrix of a bank; the CPU oracle checks sampled
matrices one by one.  Properties that hold at any size cover the largest
shapes.

Tolerances on O = (p_before - p_after) / lr, the orthogonalised update:
  vs the bf16-emulating oracle: relative Frobenius <= 1e-2, max-abs <= 3e-2;
  vs the fp64 oracle: relative Frobenius <= 5e-2;
  momentum buffers: relative <= 1e-5 (fp32, elementwise closed form).
Rank-32-plus-noise inputs: the bf16 iteration amplifies its own rounding
noise in the ~1000 tiny singular directions by up to a^5 ~ 485, so no bf16
implementation reaches the relative-Frobenius bounds there (the bf16 oracle
itself is ~0.22 from fp64, and two bf16 orderings differ by ~1.5e-2).  For
those matrices the test checks what is determined: the projection of O on
the top-32 singular subspace of G against fp64 (<= 1e-2), the norm of the
remainder against the bf16 oracle's (within 5 %), and max-abs <= 3e-2.
"""

import functools

import numpy as np
import pytest
import torch

import oracle
from newton_schulz_08_gb300 import inputs, muon
from tests.gpu_helpers import (TOL_BUF_REL, TOL_MAXABS_BF16, TOL_REL_BF16, TOL_REL_FP64,
                               bf16_np, check_status, rel, to_dev)

pytestmark = pytest.mark.gpu
LR, MU = 0.02, 0.95


def check_O(O_gpu, u, what, rank32=False):
    ob = oracle.newton_schulz5(u, 5, "bf16")
    of = oracle.newton_schulz5(u, 5, "fp64")
    assert np.abs(O_gpu - ob).max() <= TOL_MAXABS_BF16, what
    if not rank32:
        assert rel(O_gpu, ob) <= TOL_REL_BF16, (what, rel(O_gpu, ob))
        assert rel(O_gpu, of) <= TOL_REL_FP64, (what, rel(O_gpu, of))
        return
    U, _, Vt = np.linalg.svd(np.asarray(u, np.float64), full_matrices=False)
    Ur, Vr = U[:, :32], Vt[:32].T

    def sig(O):
        return Ur.T @ O @ Vr

    def rest(O):
        return np.linalg.norm(O - Ur @ sig(O) @ Vr.T)

    assert rel(sig(O_gpu), sig(of)) <= 1e-2, what
    r_gpu, r_b = rest(O_gpu), rest(ob)
    assert abs(r_gpu - r_b) <= 0.05 * r_b, (what, r_gpu, r_b)


# ---------------------------------------------------------------- single
def test_single_128x512():
    cfg = inputs.SINGLE
    p, g, b = inputs.single()
    R, C = cfg["shape"]
    P, Bd, Gd = to_dev(p), to_dev(b), to_dev(g)
    ws = muon.new_workspace(muon.muon_workspace_size([(R, C)]))
    muon.muon_step([P], [Gd], [Bd], lr=cfg["lr"], momentum=cfg["momentum"], nesterov=True,
                   ns_steps=cfg["ns_steps"], workspace=ws)
    check_status(ws)
    new_p, new_buf, O = oracle.muon_step(p, g, b, LR, MU, True, 5, "bf16")
    # (i) momentum buffer
    assert rel(Bd.cpu().numpy(), new_buf) <= TOL_BUF_REL
    # (ii) O, recovered from the parameter change, against the oracles (the
    # update itself is checked bit for bit in test_gpu_kernels)
    O_from_p = (p.astype(np.float64) - P.cpu().numpy()) / LR
    _, u = oracle.momentum_update(g, b, MU, True, "bf16")
    check_O(O_from_p, u, "single")
    assert rel(O_from_p, O) <= TOL_REL_BF16


# ---------------------------------------------------------------- gpt2 bank
def test_gpt2_bank_three_steps():
    """All 72 matrices at every step: buffers (1e-5) and O against the fp64
    oracle (5e-2); O against the bf16 oracle (1e-2 / 3e-2) for all 72 at
    step 0 and for one matrix of each kind at the later steps."""
    shapes = inputs.gpt2_shapes()
    ps = [inputs.param(s, i) for i, s in enumerate(shapes)]
    bs = [inputs.buffer(s, i) for i, s in enumerate(shapes)]
    P = [to_dev(p) for p in ps]
    B = [to_dev(b) for b in bs]
    ws = muon.new_workspace(muon.muon_workspace_size(shapes))
    bufs_oracle = [b.copy() for b in bs]
    sampled = [0, 34, 71]  # q of layer 0, c_fc (tall) of layer 5, c_proj (wide) of layer 11
    for step in range(3):
        g32 = [inputs.grad(s, i, step=step) for i, s in enumerate(shapes)]
        G = [to_dev(g, torch.bfloat16) for g in g32]
        gseen = [oracle.round_to_bf16(g).astype(np.float32) for g in g32]
        p_before = [x.cpu().numpy() for x in P]
        muon.muon_step(P, G, B, lr=LR, momentum=MU, nesterov=True, ns_steps=5, workspace=ws)
        check_status(ws)
        for i in range(len(shapes)):
            nb, u = oracle.momentum_update(gseen[i], bufs_oracle[i], MU, True, "bf16")
            bufs_oracle[i] = nb
            assert rel(B[i].cpu().numpy(), nb) <= TOL_BUF_REL, (step, i)
            O_gpu = (p_before[i].astype(np.float64) - P[i].cpu().numpy()) / LR
            if step == 0 or i in sampled:
                check_O(O_gpu, u, f"gpt2 step {step} matrix {i}")
            else:
                of = oracle.newton_schulz5(u, 5, "fp64")
                assert rel(O_gpu, of) <= TOL_REL_FP64, (step, i, rel(O_gpu, of))


# ---------------------------------------------------------------- spectra
@functools.lru_cache(maxsize=None)
def spectra_bank():
    shapes = inputs.spectra_shapes()
    return shapes, [oracle.round_to_bf16(inputs.spectra_matrix(s[0], i)).astype(np.float32)
                    for i, s in enumerate(shapes)]


def test_spectra_sweep_ns5():
    shapes, Gs = spectra_bank()
    Gd = [to_dev(g, torch.bfloat16) for g in Gs]
    ws = muon.new_workspace(muon.ns5_bank_workspace_size(shapes))
    outs = muon.ns5_bank(Gd, 5, workspace=ws)
    check_status(ws)
    for i in [0, 63, 64]:
        check_O(bf16_np(outs[i]), Gs[i].astype(np.float64), f"spectra {i}")


# ---------------------------------------------------------------- rect
def test_rect_bank():
    shapes = inputs.rect_shapes()
    ps = [inputs.param(s, i) for i, s in enumerate(shapes)]
    bs = [np.zeros(s, np.float32) for s in shapes]
    g32 = [inputs.rect_grad(s, i) for i, s in enumerate(shapes)]
    P = [to_dev(p) for p in ps]
    B = [to_dev(b) for b in bs]
    G = [to_dev(g, torch.bfloat16) for g in g32]
    ws = muon.new_workspace(muon.muon_workspace_size(shapes))
    muon.muon_step(P, G, B, lr=LR, momentum=MU, ns_steps=5, workspace=ws)
    check_status(ws)
    for i in [0, 5, 8, 13, 16, 21, 24, 29]:  # a dense and a rank-32 matrix of each shape
        gseen = oracle.round_to_bf16(g32[i]).astype(np.float32)
        nb, u = oracle.momentum_update(gseen, bs[i], MU, True, "bf16")
        assert rel(B[i].cpu().numpy(), nb) <= TOL_BUF_REL
        O_gpu = (ps[i].astype(np.float64) - P[i].cpu().numpy()) / LR
        check_O(O_gpu, u, f"rect {i}", rank32=(i % 8) >= 4)


# ---------------------------------------------------------------- 1.5B bank
def test_gpt1p5b_bank():
    shapes = inputs.gpt1p5b_shapes()
    P, B, G = [], [], []
    for i, s in enumerate(shapes):
        P.append(to_dev(inputs.param(s, i)))
        B.append(to_dev(inputs.buffer(s, i)))
        G.append(to_dev(inputs.grad(s, i), torch.bfloat16))
    sampled = [0, 4, 5, 287]
    p_before = {i: P[i].cpu().numpy() for i in sampled}
    ws = muon.new_workspace(muon.muon_workspace_size(shapes))
    muon.muon_step(P, G, B, lr=LR, momentum=MU, ns_steps=5, workspace=ws)
    check_status(ws)
    for i in sampled:
        s = shapes[i]
        gseen = oracle.round_to_bf16(inputs.grad(s, i)).astype(np.float32)
        nb, u = oracle.momentum_update(gseen, inputs.buffer(s, i), MU, True, "bf16")
        assert rel(B[i].cpu().numpy(), nb) <= TOL_BUF_REL
        O_gpu = (p_before[i].astype(np.float64) - P[i].cpu().numpy()) / LR
        check_O(O_gpu, u, f"1.5B matrix {i}")


# ---------------------------------------------------------------- any size
def test_transpose_path_is_exact_at_large_size():
    """A tall matrix is transposed in the first pass, so NS(G^T) and NS(G)^T
    are computed from the same X and must agree bit for bit."""
    g = torch.Generator(device="cuda").manual_seed(99)
    G = torch.randn((2048, 8192), generator=g, device="cuda", dtype=torch.float32)
    O_wide = muon.ns5(G, 5)
    O_tall = muon.ns5(G.t().contiguous(), 5)
    assert torch.equal(O_tall, O_wide.t())


def test_orthogonal_input_flat_spectrum_at_8192():
    """For an orthogonal n x n input, every singular value of O is
    p^5(1/(sqrt(n) + 1e-7)) up to the bf16 error of the iteration."""
    n = 8192
    g = torch.Generator(device="cuda").manual_seed(7)
    Q, _ = torch.linalg.qr(torch.randn((n, n), generator=g, device="cuda", dtype=torch.float32))
    O = muon.ns5(Q.contiguous(), 5).float()
    s = torch.linalg.svdvals(O).double().cpu().numpy()
    a, b, c = oracle.NS_COEFFS
    x = 1.0 / (np.sqrt(n) + 1e-7)
    for _ in range(5):
        x = a * x + b * x ** 3 + c * x ** 5
    assert np.abs(s - x).max() <= 3e-2 * x, (s.min(), s.max(), x)
