"""The debug build (libmuon_debug.so, compiled with MUON_DEBUG): its
kernels check the ranges of their raw-pointer accesses and the alignment of
their TMA coordinates, counting failures instead of trapping.  Every entry
point runs through it on shapes that reach the ragged, tall, wide, streamed
and register paths; no check may fail and every result must equal the
release library's bit for bit (the checks only guard accesses)."""

import numpy as np
import pytest
import torch

from newton_schulz_08_gb300 import muon
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(256, 256), (300, 100), (100, 300), (129, 257), (768, 768), (64, 3072), (37, 1)]


@pytest.fixture
def debug_lib(monkeypatch):
    L = muon.load(muon.DEBUG_LIB_PATH)
    failures = __import__("ctypes").c_longlong(-1)
    assert L.muon_debug_check_failures(failures) == 0  # a debug build; clears the counters
    return L


def failures(L):
    import ctypes
    n = ctypes.c_longlong(-1)
    assert L.muon_debug_check_failures(n) == 0
    return n.value


def run_all(seed):
    rng = np.random.default_rng(seed)
    out = []
    P = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(0.02)) for s in SHAPES]
    G = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(1e-3), torch.bfloat16) for s in SHAPES]
    B = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(1e-3)) for s in SHAPES]
    muon.muon_step(P, G, B)
    out += P + B
    out.append(muon.ns5(to_dev(rng.standard_normal((3, 200, 72)).astype(np.float32)), 5))
    out += muon.ns5_bank([to_dev(rng.standard_normal(s).astype(np.float32)) for s in SHAPES[:4]], 5)
    x = to_dev(rng.standard_normal((272, 384)).astype(np.float32), torch.bfloat16)
    w = to_dev(rng.standard_normal((528, 384)).astype(np.float32) * np.float32(0.05), torch.bfloat16)
    # scales that fill the formats without overflow (largest quotient 448 / 1.05, 57344 / 1.05)
    x_s, w_s = (float(t.abs().max().float()) / 448.0 * 1.05 for t in (x, w))
    o, xq, wq = muon.fp8_mm(x, w, x_s, w_s)
    g = to_dev(rng.standard_normal((272, 528)).astype(np.float32) * np.float32(1e-3), torch.bfloat16)
    gx, gw, gq = muon.fp8_mm_backward(g, xq, wq, x_s, w_s, float(g.abs().max().float()) / 57344.0 * 1.05)
    out += [o, xq.view(torch.uint8), wq.view(torch.uint8), gx, gw, gq.view(torch.uint8)]
    pa = [to_dev(rng.standard_normal(n).astype(np.float32)) for n in (10_007, 64)]
    ma = [torch.zeros_like(t) for t in pa]
    va = [torch.zeros_like(t) for t in pa]
    ga = [to_dev(rng.standard_normal(t.numel()).astype(np.float32), torch.bfloat16) for t in pa]
    muon.adam_step(pa, ga, ma, va, 1, lr=1e-3, weight_decay=0.1)
    out += pa + ma + va
    torch.cuda.synchronize()
    return out


def test_debug_build_passes_its_checks_and_matches_release(debug_lib, monkeypatch):
    want = run_all(5)
    monkeypatch.setattr(muon, "_lib", debug_lib)
    got = run_all(5)
    assert failures(debug_lib) == 0
    for a, b in zip(got, want):
        assert not a.float().isnan().any()
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))  # bit for bit
