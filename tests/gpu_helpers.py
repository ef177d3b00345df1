"""Shared helpers for the GPU parity tests (comparisons and buffer views)."""

import numpy as np
import torch

from newton_schulz_08_gb300 import muon

# tolerances on O (bf16 iteration): GPU vs the bf16-emulating oracle and vs
# the fp64 oracle, relative Frobenius / elementwise max-abs
TOL_REL_BF16 = 1e-2
TOL_MAXABS_BF16 = 3e-2
TOL_REL_FP64 = 5e-2
TOL_BUF_REL = 1e-5


def rel(x, y):
    return float(np.linalg.norm(np.asarray(x, np.float64) - np.asarray(y, np.float64))
                 / max(np.linalg.norm(np.asarray(y, np.float64)), 1e-300))


def bf16_ulp(v):
    """Spacing of bfloat16 numbers at |v| (normal range; subnormal spacing below)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    _, ex = np.frexp(a)
    return np.ldexp(1.0, ex - 8)


def assert_bf16_close(got, want, absmag, what, slack=1e-5, max_frac=0.05):
    """Elementwise: within one bf16 spacing of `want`, plus `slack` times the
    magnitude `absmag` of the sum that produced it (fp32 accumulation order);
    and at most `max_frac` of the elements may differ at all."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    bound = bf16_ulp(want) * 1.0001 + slack * np.asarray(absmag, np.float64)
    bad = np.abs(got - want) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond bound; worst {np.abs(got - want)[bad].max():.3e}"
    frac = float(np.mean(got != want)) if got.size else 0.0
    assert frac <= max_frac, f"{what}: {frac:.3%} of elements differ"


def ws_view(ws, offset, rows, cols, ld, batch=1, index=0):
    """bf16 matrix view into a workspace tensor (torch uint8) -> float64 numpy."""
    start = offset + 2 * index * rows * ld
    t = ws[start:start + 2 * rows * ld].view(torch.bfloat16).view(rows, ld)[:, :cols]
    return t.float().cpu().numpy().astype(np.float64)


def sym_from_upper_blocks(M, block=256):
    """The full symmetric matrix from its stored blocks on and above the
    diagonal (blocks below the diagonal are not written by the kernels)."""
    F = M.copy()
    m = M.shape[0]
    for i0 in range(0, m, block):
        for j0 in range(0, i0, block):
            F[i0:i0 + block, j0:j0 + block] = M[j0:j0 + block, i0:i0 + block].T
    return F


def diagonal_blocks_symmetric(M, block=256):
    m = M.shape[0]
    return all(np.array_equal(M[i:i + block, i:i + block], M[i:i + block, i:i + block].T)
               for i in range(0, m, block))


def to_dev(a, dtype=torch.float32, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device).to(dtype)


def bf16_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_status(ws):
    st = muon.muon_device_status(ws)
    assert st == muon.MUON_OK, muon.muon_status_str(st)
