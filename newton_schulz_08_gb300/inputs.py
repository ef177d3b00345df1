"""Seeded synthetic inputs for the Muon step workloads.

This module only draws random tensors; it holds none of the step's arithmetic.
Both the CUDA path (through the tests and the benchmark) and the CPU oracle
take their inputs from here, as NumPy arrays on the host.

Every matrix has its own seed, so a single matrix of a large bank can be
regenerated on its own (the parity tests check sampled matrices of a bank
against the oracle).  Draws use NumPy's PCG64 generator.

Workloads (matrix shapes are rows x cols as stored, row-major):

* ``single``   one 128x512 matrix; g ~ N(0,1) fp32, p ~ N(0, 0.02^2) fp32,
               momentum buffer zeros.
* ``gpt2``     GPT-2-124M hidden-matrix bank, d = 768, 12 layers, each with
               q, k, v, o (768x768), c_fc (3072x768), c_proj (768x3072):
               72 matrices, 84.93 M parameters; p ~ N(0, 0.02^2) fp32,
               buffers ~ N(0, 1e-3^2) fp32, grads ~ N(0, 1e-3^2) bf16 drawn
               afresh for every step.
* ``spectra``  square bf16 G = U diag(s) V^T with U, V Haar-orthogonal (QR of a
               Gaussian with the signs of R's diagonal folded in) and s
               log-uniform in [1e-4, 1]; 64 of 1024x1024 and 16 of 4096x4096.
* ``rect``     8 each of 1024x4096, 4096x1024, 768x3072, 2048x8192 bf16
               grads: the first 4 of each shape dense N(0,1), the last 4
               rank-32 (Gaussian factors) plus 1e-3 N(0,1) noise; p ~
               N(0, 0.02^2), buffers zero.
* ``gpt1p5b``  1.5B-shaped bank, d = 1600, 48 layers of 4 x (1600x1600),
               6400x1600, 1600x6400 (288 matrices, 1.4746 B parameters);
               as ``gpt2`` otherwise, one step.
* ``adam``     embedding-type bank for the Adam step: 4 tables of
               50304 x 768 (GPT-2-124M's padded vocabulary x width; the page
               names the bigram and value-embedding banks but not their
               sizes), 154.53 M fp32 parameters; p ~ N(0, 0.02^2), first
               moment ~ N(0, 1e-3^2), second moment = (N(0, 1e-3^2))^2
               (non-negative), grads ~ N(0, 1e-3^2) bf16; the state is that
               of a step in mid-training (step count 10).
"""

import numpy as np

# seed bases per tensor kind; matrix i of a bank uses base + i
SEED_P = 1_000_000
SEED_BUF = 2_000_000
SEED_G = 3_000_000  # + 10_000 * step
SEED_U = 4_000_000
SEED_V = 5_000_000
SEED_S = 6_000_000
SEED_RECT = 7_000_000
SEED_ADAM = 8_000_000  # + 4 * tensor + {0: p, 1: m, 2: v, 3: g} + 1_000 * step


def gpt2_shapes(d=768, layers=12):
    shapes = []
    for _ in range(layers):
        shapes += [(d, d)] * 4 + [(4 * d, d), (d, 4 * d)]
    return shapes


def gpt1p5b_shapes():
    return gpt2_shapes(d=1600, layers=48)


def rect_shapes():
    shapes = []
    for s in [(1024, 4096), (4096, 1024), (768, 3072), (2048, 8192)]:
        shapes += [s] * 8
    return shapes


def spectra_shapes():
    return [(1024, 1024)] * 64 + [(4096, 4096)] * 16


def normal(shape, std, seed, dtype=np.float32):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x.astype(dtype, copy=False)


def param(shape, i, std=0.02):
    return normal(shape, std, SEED_P + i)


def buffer(shape, i, std=1e-3):
    if std == 0.0:
        return np.zeros(shape, np.float32)
    return normal(shape, std, SEED_BUF + i)


def grad(shape, i, step=0, std=1e-3):
    """float32 draw; bf16 banks round it to bfloat16 when uploading."""
    return normal(shape, std, SEED_G + 10_000 * step + i)


ADAM_TABLE = (50304, 768)
ADAM_STEP = 10


def adam_bank_shapes(tables=4):
    return [ADAM_TABLE] * tables


def adam_state(shape, i, step=0):
    """Tensor i of an Adam bank: (p, m, v, g) float32 (g is rounded to
    bfloat16 when a bank uploads bf16 gradients).  Gradients differ per step."""
    rng = [np.random.default_rng(SEED_ADAM + 4 * i + k) for k in range(3)]
    p = rng[0].standard_normal(shape, dtype=np.float32) * np.float32(0.02)
    m = rng[1].standard_normal(shape, dtype=np.float32) * np.float32(1e-3)
    v = np.square(rng[2].standard_normal(shape, dtype=np.float32) * np.float32(1e-3))
    g = np.random.default_rng(SEED_ADAM + 4 * i + 3 + 1_000 * step).standard_normal(shape, dtype=np.float32)
    return p, m, v, g * np.float32(1e-3)


def haar(n, seed):
    rng = np.random.default_rng(seed)
    Z = rng.standard_normal((n, n))
    Q, R = np.linalg.qr(Z)
    return Q * np.sign(np.diag(R))


def spectra_matrix(n, i):
    """float64 U diag(s) V^T; rounded to bfloat16 when uploading."""
    U = haar(n, SEED_U + i)
    V = haar(n, SEED_V + i)
    s = np.exp(np.random.default_rng(SEED_S + i).uniform(np.log(1e-4), 0.0, n))
    return (U * s) @ V.T


def rect_grad(shape, i):
    """Matrix i of the rect bank: dense when i % 8 < 4, else rank 32 + noise."""
    rng = np.random.default_rng(SEED_RECT + i)
    R, C = shape
    if i % 8 < 4:
        return rng.standard_normal((R, C), dtype=np.float32)
    L = rng.standard_normal((R, 32), dtype=np.float32)
    Rt = rng.standard_normal((C, 32), dtype=np.float32)
    noise = rng.standard_normal((R, C), dtype=np.float32)
    return L @ Rt.T + np.float32(1e-3) * noise


SINGLE = {"shape": (128, 512), "lr": 0.02, "momentum": 0.95, "nesterov": True, "ns_steps": 5}


def single():
    """The 128x512 single-matrix case: (p, g, buf) float32."""
    shape = SINGLE["shape"]
    g = normal(shape, 1.0, 0)
    p = normal(shape, 0.02, 1)
    return p, g, np.zeros(shape, np.float32)


def spectra_matrix_device(n, i, device, dtype=None):
    """The spectra recipe drawn with torch on `device` (seeded per matrix):
    U, V from QR of Gaussians with R's diagonal signs folded in, s
    log-uniform in [1e-4, 1], G = U diag(s) V^T in float32.  Used where
    host generation of large banks would be too slow (timing runs); the
    parity tests use spectra_matrix."""
    import torch
    g = torch.Generator(device=device).manual_seed(SEED_U + i)
    Z = torch.randn((2, n, n), generator=g, device=device, dtype=torch.float32)
    Q, R = torch.linalg.qr(Z)
    Q = Q * torch.sign(torch.diagonal(R, dim1=-2, dim2=-1)).unsqueeze(-2)
    s = torch.exp(torch.empty(n, device=device).uniform_(float(np.log(1e-4)), 0.0, generator=g))
    G = (Q[0] * s) @ Q[1].T
    return G if dtype is None else G.to(dtype)
