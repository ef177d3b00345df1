"""GPU parity of each kernel and of small end-to-end calls, through the C ABI.

Every comparison is against the CPU oracle on the same seeded inputs.  The
single-step test isolates each tensor-core kernel: the oracle's step function
is fed the GPU's own input to that kernel (X0 for the Gram, A for the
polynomial, B and X0 for the update), so a mismatch points at one kernel.
"""

import numpy as np
import pytest
import torch

import oracle
from newton_schulz_08_gb300 import inputs, muon
from tests.gpu_helpers import (TOL_BUF_REL, TOL_MAXABS_BF16, TOL_REL_BF16, TOL_REL_FP64,
                               assert_bf16_close, bf16_np, check_status, diagonal_blocks_symmetric, rel,
                               sym_from_upper_blocks, to_dev, ws_view)

pytestmark = pytest.mark.gpu

A_, B_, C_ = (float(np.float32(v)) for v in oracle.NS_COEFFS)

# spans one tile, several tiles, ragged tails in both dimensions, tall and
# wide, columns that are not a multiple of 8, and degenerate 1-wide shapes
SHAPES = [(128, 512), (256, 256), (200, 328), (300, 100), (129, 257), (100, 37), (37, 100),
          (1, 1), (1, 37), (37, 1), (384, 1536), (1536, 384), (520, 520)]


def gauss(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def as_seen(G, dtype):
    """The values the GPU reads: bf16 inputs are rounded on upload."""
    return oracle.round_to_bf16(G) if dtype == torch.bfloat16 else G.astype(np.float64)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_normalise_x0(shape, dtype):
    G = gauss(shape, 1)
    out = muon.ns5(to_dev(G, dtype), ns_steps=0)
    torch.cuda.synchronize()
    want = oracle.newton_schulz5(as_seen(G, dtype), 0, "bf16")
    check_x0(bf16_np(out), want)


def check_x0(got, want):
    """X0 = bf16(Xb / (||Xb|| + 1e-7)): the GPU forms the norm and the quotient
    in fp32, the oracle in fp64.  Xb has at most 256 significands per binade,
    so when one significand's quotient lies within fp32 error of a bf16
    midpoint every entry with that significand rounds the other way: entries
    may differ by one bf16 spacing, a few percent of them at most."""
    assert_bf16_close(got, want, 0.0, "X0", slack=0.0, max_frac=0.05)
    assert rel(got, want) <= 2e-3


@pytest.mark.parametrize("shape", SHAPES)
def test_one_step_each_kernel(shape):
    R, C = shape
    G = gauss(shape, 2)
    lay = muon.ns5_workspace_layout(1, R, C)
    ws = muon.new_workspace(muon.ns5_workspace_size(1, R, C))
    out = muon.ns5(to_dev(G), ns_steps=1, workspace=ws)
    check_status(ws)
    m, n, ldx, lda = lay["m"], lay["n"], lay["ldx"], lay["lda"]
    X0 = ws_view(ws, lay["x_offset"][0], m, n, ldx)
    A_st = ws_view(ws, lay["a_offset"], m, m, lda)
    B_st = ws_view(ws, lay["b_offset"], m, m, lda)
    # A and B are stored as their 256 x 256 blocks on and above the diagonal
    # (diagonal blocks computed whole, exactly symmetric)
    assert diagonal_blocks_symmetric(A_st) and diagonal_blocks_symmetric(B_st)
    A = sym_from_upper_blocks(A_st)
    B = sym_from_upper_blocks(B_st)
    X1 = ws_view(ws, lay["x_offset"][1], m, n, ldx)
    # X0 is the oracle's normalised input (orientation: tall inputs transposed)
    Gv, tall = oracle.orient(G.astype(np.float64))
    check_x0(X0, oracle.normalise(Gv, "bf16"))
    # Gram kernel: A = bf16(X0 X0^T)
    absX = np.abs(X0)
    assert_bf16_close(A, oracle.ns_gram(X0, "bf16"), absX @ absX.T, "A")
    # polynomial kernel: B = bf16(b A + c A A)
    absA = np.abs(A)
    assert_bf16_close(B, oracle.ns_poly(A, "bf16"), abs(B_) * absA + abs(C_) * absA @ absA, "B")
    # update kernel: X1 = bf16(a X0 + B X0), and O is X1 in G's orientation
    assert_bf16_close(X1, oracle.ns_update(B, X0, "bf16"), abs(A_) * absX + np.abs(B) @ absX, "X1")
    O = bf16_np(out)
    assert np.array_equal(O, X1.T if tall else X1)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("steps", [2, 5])
def test_ns5_matches_oracle(shape, steps):
    G = gauss(shape, 3)
    out = bf16_np(muon.ns5(to_dev(G), ns_steps=steps))
    ob = oracle.newton_schulz5(G, steps, "bf16")
    of = oracle.newton_schulz5(G, steps, "fp64")
    if min(shape) == 1:
        # a single row or column: O = p^steps(~1) g/||g||, exact up to rounding
        assert np.abs(out - ob).max() <= 2 * bf16_ulp_max(ob)
        return
    assert rel(out, ob) <= TOL_REL_BF16
    assert np.abs(out - ob).max() <= TOL_MAXABS_BF16
    assert rel(out, of) <= TOL_REL_FP64


def bf16_ulp_max(v):
    from tests.gpu_helpers import bf16_ulp
    return float(bf16_ulp(np.abs(v).max()))


def test_ns5_batched_equals_single():
    G = gauss((5, 200, 328), 4)
    Gt = to_dev(G)
    batched = muon.ns5(Gt, 5)
    for i in range(5):
        single = muon.ns5(Gt[i].contiguous(), 5)
        assert torch.equal(batched[i], single)


def test_ns5_bank_equals_per_shape_calls():
    shapes = [(200, 328), (328, 200), (64, 64), (128, 512), (37, 100)]
    Gs = [to_dev(gauss(s, 10 + i)) for i, s in enumerate(shapes)]
    outs = muon.ns5_bank(Gs, 5)
    for g, o in zip(Gs, outs):
        assert torch.equal(o, muon.ns5(g, 5))


def run_step(shapes, nesterov=True, steps=5, gdtype=torch.bfloat16, seed=0, lr=0.02, mu=0.95):
    rng = np.random.default_rng(seed)
    ps = [rng.standard_normal(s).astype(np.float32) * np.float32(0.02) for s in shapes]
    gs = [rng.standard_normal(s).astype(np.float32) * np.float32(1e-3) for s in shapes]
    bs = [rng.standard_normal(s).astype(np.float32) * np.float32(1e-3) for s in shapes]
    P = [to_dev(p) for p in ps]
    Gd = [to_dev(g, gdtype) for g in gs]
    Bd = [to_dev(b) for b in bs]
    ws = muon.muon_step(P, Gd, Bd, lr=lr, momentum=mu, nesterov=nesterov, ns_steps=steps)
    check_status(ws)
    gseen = [as_seen(g, gdtype).astype(np.float32) for g in gs]
    return ps, gseen, bs, [t.cpu().numpy() for t in P], [t.cpu().numpy() for t in Bd]


@pytest.mark.parametrize("nesterov", [True, False])
@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32])
def test_muon_step_mixed_bank(nesterov, gdtype):
    shapes = [(256, 256), (300, 100), (100, 300), (129, 257), (64, 64), (37, 100), (256, 256)]
    lr, mu = 0.02, 0.95
    ps, gs, bs, P, Bn = run_step(shapes, nesterov, 5, gdtype, seed=5, lr=lr, mu=mu)
    for i in range(len(shapes)):
        new_p, new_buf, O = oracle.muon_step(ps[i], gs[i], bs[i], lr, mu, nesterov, 5, "bf16")
        assert rel(Bn[i], new_buf) <= TOL_BUF_REL
        O_gpu = (ps[i].astype(np.float64) - P[i].astype(np.float64)) / lr
        assert rel(O_gpu, O) <= TOL_REL_BF16, i
        assert np.abs(O_gpu - O).max() <= TOL_MAXABS_BF16
        _, _, O64 = oracle.muon_step(ps[i], gs[i], bs[i], lr, mu, nesterov, 5, "fp64")
        assert rel(O_gpu, O64) <= TOL_REL_FP64


def check_bank_against_oracle(shapes, ps, gs, bs, P, Bn, lr=0.02, mu=0.95):
    for i in range(len(shapes)):
        new_p, new_buf, O = oracle.muon_step(ps[i], gs[i], bs[i], lr, mu, True, 5, "bf16")
        assert rel(Bn[i], new_buf) <= TOL_BUF_REL, i
        O_gpu = (ps[i].astype(np.float64) - P[i].astype(np.float64)) / lr
        assert rel(O_gpu, O) <= TOL_REL_BF16, (i, shapes[i])
        assert np.abs(O_gpu - O).max() <= TOL_MAXABS_BF16, (i, shapes[i])


def test_bank_beyond_one_launch_per_phase():
    """12 shape classes (each phase takes two launches of at most 8 classes)
    and 108 matrices (the momentum pass takes two launches of at most 96).
    Every matrix: momentum buffer, and O against the fp64 oracle; one matrix
    per class: O against the bf16 oracle.  (The bf16 bound is checked on a
    subset: two bf16 evaluations that differ only in fp32 accumulation order
    already differ by up to ~8e-3 on Gaussian matrices of these sizes, so
    over a hundred draws the 1e-2 bound has no margin.)"""
    base = [(128, 384), (384, 128), (256, 256), (192, 320), (320, 192), (256, 512), (512, 256),
            (160, 480), (480, 160), (300, 300), (224, 448), (448, 224)]
    shapes = [base[i % len(base)] for i in range(108)]
    lr, mu = 0.02, 0.95
    ps, gs, bs, P, Bn = run_step(shapes, True, 5, torch.bfloat16, seed=11, lr=lr, mu=mu)
    for i in range(len(shapes)):
        nb, u = oracle.momentum_update(gs[i], bs[i], mu, True, "bf16")
        assert rel(Bn[i], nb) <= TOL_BUF_REL, i
        O_gpu = (ps[i].astype(np.float64) - P[i].astype(np.float64)) / lr
        O64 = oracle.newton_schulz5(u, 5, "fp64")
        assert rel(O_gpu, O64) <= TOL_REL_FP64, (i, shapes[i])
    picks = list(range(len(base)))
    check_bank_against_oracle([shapes[i] for i in picks], [ps[i] for i in picks], [gs[i] for i in picks],
                              [bs[i] for i in picks], [P[i] for i in picks], [Bn[i] for i in picks], lr, mu)


@pytest.mark.parametrize("shape", [(2, 65536), (65536, 3), (256, 40000)])
def test_extreme_aspect_ratios(shape):
    """Long contractions (up to 1024 K blocks per tile), 2- and 3-row Gram
    matrices padded inside one tile, and a tall matrix whose width is not a
    multiple of 4 (the scalar path of the transposing momentum pass)."""
    ps, gs, bs, P, Bn = run_step([shape], True, 5, torch.bfloat16, seed=12)
    check_bank_against_oracle([shape], ps, gs, bs, P, Bn)


def test_zero_matrix_leaves_param():
    p = np.random.default_rng(7).standard_normal((128, 256)).astype(np.float32)
    P = to_dev(p)
    z = torch.zeros((128, 256), device="cuda", dtype=torch.bfloat16)
    b = torch.zeros((128, 256), device="cuda")
    ws = muon.muon_step([P], [z], [b])
    check_status(ws)
    assert np.array_equal(P.cpu().numpy(), p)


def test_nonfinite_is_reported():
    G = gauss((64, 128), 8)
    G[3, 5] = np.inf
    ws = muon.new_workspace(muon.ns5_workspace_size(1, 64, 128))
    muon.ns5(to_dev(G), 5, workspace=ws)
    assert muon.muon_device_status(ws) == muon.MUON_WARN_NONFINITE
    # a finite call on the same workspace clears the status
    muon.ns5(to_dev(gauss((64, 128), 9)), 5, workspace=ws)
    assert muon.muon_device_status(ws) == muon.MUON_OK


def test_bounded_wait_expires_and_context_survives():
    G = to_dev(gauss((256, 512), 11))
    ws = muon.new_workspace(muon.ns5_workspace_size(1, 256, 512))
    muon.muon_set_debug("inject_stall", 1)
    muon.muon_set_debug("wait_budget_cycles", 20_000_000)  # ~10 ms
    try:
        muon.ns5(G, 1, workspace=ws)
        st = muon.muon_device_status(ws)
    finally:
        muon.muon_set_debug("inject_stall", 0)
        muon.muon_set_debug("wait_budget_cycles", 4_000_000_000)
    assert st == muon.MUON_ERR_DEVICE_TIMEOUT
    out = muon.ns5(G, 5, workspace=ws)
    check_status(ws)
    ob = oracle.newton_schulz5(G.cpu().numpy(), 5, "bf16")
    assert rel(bf16_np(out), ob) <= TOL_REL_BF16


def test_deterministic():
    shapes = [(256, 256), (300, 100)]
    r1 = run_step(shapes, seed=12)
    r2 = run_step(shapes, seed=12)
    for a, b in zip(r1[3] + r1[4], r2[3] + r2[4]):
        assert np.array_equal(a, b)


def test_resume_matches_straight_run():
    """3 steps in a row == 2 steps, state copied to the host and back, 1 step."""
    shapes = [(200, 328), (328, 200)]
    rng = np.random.default_rng(13)
    p0 = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    grads = [[to_dev(rng.standard_normal(s).astype(np.float32) * 1e-3, torch.bfloat16) for s in shapes]
             for _ in range(3)]

    def fresh():
        return [to_dev(p) for p in p0], [torch.zeros(s, device="cuda") for s in shapes]

    P1, B1 = fresh()
    for k in range(3):
        muon.muon_step(P1, grads[k], B1)
    P2, B2 = fresh()
    for k in range(2):
        muon.muon_step(P2, grads[k], B2)
    host = [t.cpu() for t in P2 + B2]
    P3 = [h.cuda() for h in host[:2]]
    B3 = [h.cuda() for h in host[2:]]
    muon.muon_step(P3, grads[2], B3)
    for a, b in zip(P1 + B1, P3 + B3):
        assert torch.equal(a, b)


def test_empty_calls():
    assert muon.ns5(torch.empty((0, 8, 8), device="cuda"), 5).shape == (0, 8, 8)
    assert muon.ns5_bank([], 5) == []


def test_cuda_graph_capture_replays_the_step():
    """muon_step under stream capture (cluster launches, programmatic
    dependent launch, the status memset): replaying the captured step three
    times gives the eager result bit for bit."""
    shapes = [(256, 256), (300, 100), (100, 300), (129, 257)]
    rng = np.random.default_rng(21)
    P0 = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(0.02)) for s in shapes]
    G = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(1e-3), torch.bfloat16) for s in shapes]
    B0 = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(1e-3)) for s in shapes]
    P, B = [p.clone() for p in P0], [b.clone() for b in B0]
    ws = muon.muon_step(P, G, B)  # plan, attributes and workspace set up outside the capture
    for x, x0 in zip(P + B, P0 + B0):
        x.copy_(x0)
    for _ in range(3):
        muon.muon_step(P, G, B, workspace=ws)
    want = [x.clone() for x in P + B]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        muon.muon_step(P, G, B, workspace=ws)
    for x, x0 in zip(P + B, P0 + B0):
        x.copy_(x0)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    check_status(ws)
    for a, b in zip(P + B, want):
        assert torch.equal(a, b)


# The bf16 bound holds for up to five steps.  Two bf16 evaluations that differ
# only in fp32 accumulation order drift apart with every further step: an
# emulation of fp32 accumulation on these inputs is 6.7e-3 from the bf16
# oracle after 5 steps and 1.18e-2 after 7 (256 x 256), so 7 steps get twice
# the bound, and the fp64 bound, which the bf16 oracle itself meets with room
# (1.6-1.8e-2 after 7 steps), as well.
STEP_COUNT_TOL_BF16 = {0: TOL_REL_BF16, 1: TOL_REL_BF16, 2: TOL_REL_BF16, 7: 2 * TOL_REL_BF16}


@pytest.mark.parametrize("steps", [0, 1, 2, 7])
def test_muon_step_any_step_count(steps):
    """The final X sits in ping-pong buffer (steps % 2); 0 steps applies X0."""
    shapes = [(256, 256), (300, 100), (100, 300)]
    lr, mu = 0.02, 0.95
    ps, gs, bs, P, Bn = run_step(shapes, True, steps, torch.bfloat16, seed=31, lr=lr, mu=mu)
    for i in range(len(shapes)):
        _, new_buf, O = oracle.muon_step(ps[i], gs[i], bs[i], lr, mu, True, steps, "bf16")
        _, _, O64 = oracle.muon_step(ps[i], gs[i], bs[i], lr, mu, True, steps, "fp64")
        assert rel(Bn[i], new_buf) <= TOL_BUF_REL
        O_gpu = (ps[i].astype(np.float64) - P[i].astype(np.float64)) / lr
        assert rel(O_gpu, O) <= STEP_COUNT_TOL_BF16[steps], (steps, i, rel(O_gpu, O))
        assert rel(O_gpu, O64) <= TOL_REL_FP64, (steps, i, rel(O_gpu, O64))
        assert np.abs(O_gpu - O).max() <= TOL_MAXABS_BF16


@pytest.mark.parametrize("shape", [(256, 256), (300, 100), (100, 300), (520, 1030), (1030, 520), (130, 258),
                                   (77, 45), (45, 77), (768, 3072), (3072, 768)])
def test_parameter_update_is_one_fma_per_entry(shape):
    """The last update applies p <- p - lr O in its epilogue, O the
    bf16-rounded final X.  With momentum 0 the step's X is the gradient
    itself, so ns5 of the same gradient (given as float32, which takes the
    same cast-and-norm loop) yields the step's O bit for bit, and every
    parameter must equal fl32(p - lr O): one fused multiply-add (lr O is
    exact in float64, and so is the difference here).  Wide, tall and ragged
    shapes: the tall path writes p's rows straight from registers, the wide
    path sweeps the staged rows, and n % 4 != 0 takes the scalar path."""
    lr = np.float32(0.02)
    p = inputs.param(shape, 40)
    g = oracle.round_to_bf16(inputs.grad(shape, 40)).astype(np.float32)
    dev = torch.device("cuda")
    P = torch.from_numpy(p).to(dev)
    G = torch.from_numpy(g).to(dev).to(torch.bfloat16)
    B = torch.zeros_like(P)
    ws = muon.muon_step([P], [G], [B], lr=float(lr), momentum=0.0, nesterov=True, ns_steps=5)
    O = muon.ns5(G.float(), 5)
    torch.cuda.synchronize()
    check_status(ws)
    O = O.float().cpu().numpy().astype(np.float64)
    want = (p.astype(np.float64) - np.float64(lr) * O).astype(np.float32)
    got = P.cpu().numpy()
    same = got.view(np.uint32) == want.view(np.uint32)
    assert same.all(), (int((~same).sum()), got.size)


def test_last_update_of_a_bank_beyond_the_streamed_maps():
    """A bank of more matrices than one launch carries parameter maps for
    (230, against 190): the last update takes the register path over three
    shape classes.  With momentum 0 the step's O is ns5_bank's O of the same
    gradients bit for bit, and every parameter must equal fl32(p - lr O)."""
    shapes = [(64, 128)] * 100 + [(128, 64)] * 100 + [(96, 200)] * 30
    lr = np.float32(0.02)
    dev = torch.device("cuda")
    ps = [inputs.param(s, 500 + i) for i, s in enumerate(shapes)]
    gs = [oracle.round_to_bf16(inputs.grad(s, 500 + i)).astype(np.float32) for i, s in enumerate(shapes)]
    P = [torch.from_numpy(p).to(dev) for p in ps]
    G = [torch.from_numpy(g).to(dev).to(torch.bfloat16) for g in gs]
    B = [torch.zeros_like(x) for x in P]
    ws = muon.muon_step(P, G, B, lr=float(lr), momentum=0.0, nesterov=True, ns_steps=5)
    O = muon.ns5_bank([g.float() for g in G], 5)
    torch.cuda.synchronize()
    check_status(ws)
    bad = 0
    for i in range(len(shapes)):
        o = O[i].float().cpu().numpy().astype(np.float64)
        want = (ps[i].astype(np.float64) - np.float64(lr) * o).astype(np.float32)
        got = P[i].cpu().numpy()
        bad += int((got.view(np.uint32) != want.view(np.uint32)).sum())
    assert bad == 0, bad


def test_step_graph_replay_equals_eager():
    """A step recorded in a CUDA graph changes nothing while it is recorded,
    and two replays give the parameters and buffers of two eager steps bit
    for bit (wide, tall and square matrices)."""
    shapes = [(256, 256), (300, 100), (128, 512), (768, 3072)]
    dev = torch.device("cuda")
    P0 = [torch.from_numpy(inputs.param(s, 600 + i)).to(dev) for i, s in enumerate(shapes)]
    B0 = [torch.from_numpy(inputs.buffer(s, 600 + i)).to(dev) for i, s in enumerate(shapes)]
    G = [torch.from_numpy(inputs.grad(s, 600 + i)).to(dev).to(torch.bfloat16) for i, s in enumerate(shapes)]
    Pg, Bg = [p.clone() for p in P0], [b.clone() for b in B0]
    Pe, Be = [p.clone() for p in P0], [b.clone() for b in B0]
    sg = muon.StepGraph(Pg, G, Bg, lr=0.02, momentum=0.95, nesterov=True, ns_steps=5)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(Pg, P0)) and all(torch.equal(a, b) for a, b in zip(Bg, B0))
    ws = None
    for _ in range(2):
        sg.replay()
        ws = muon.muon_step(Pe, G, Be, lr=0.02, momentum=0.95, nesterov=True, ns_steps=5, workspace=ws)
    torch.cuda.synchronize()
    check_status(sg.workspace)
    check_status(ws)
    for a, b in zip(Pg + Bg, Pe + Be):
        assert torch.equal(a, b)


def test_zero_lr_and_zero_momentum():
    """lr = 0 leaves the parameters bit for bit; momentum 0 makes the buffer
    the gradient (fp32 value of the bf16 gradient)."""
    shapes = [(256, 256), (300, 100)]
    ps, gs, bs, P, Bn = run_step(shapes, True, 5, torch.bfloat16, seed=32, lr=0.0, mu=0.0)
    for i in range(len(shapes)):
        assert np.array_equal(P[i], ps[i])
        assert np.array_equal(Bn[i], gs[i])
