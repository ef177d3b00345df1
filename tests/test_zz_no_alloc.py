"""ns5_noalloc: the Newton-Schulz call for callers that may not allocate
device memory (for example code hosted by a framework whose allocator owns
the GPU, or latency-critical code where cudaMalloc could synchronise the
device).  It runs the same kernels as ns5 but takes its scratch from a static
64 MiB device array inside the library instead of a caller workspace.

The GPU tests call it through the C ABI twice in a row, on different shapes
and dtypes, and compare each result with ns5 given a normal workspace; and
check that, once the first call has loaded the library's device code, calls
change neither the memory PyTorch's allocator holds nor the device's free
memory.  The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from newton_schulz_08_gb300 import muon
from tests.gpu_helpers import TOL_MAXABS_BF16, TOL_REL_BF16, bf16_np, rel


def call_noalloc(G, out, ns_steps=5):
    batch, rows, cols = G.shape
    return muon.lib().ns5_noalloc(ctypes.c_void_p(G.data_ptr()), muon._dtype_code(G),
                                  ctypes.c_void_p(out.data_ptr()), batch, rows, cols, ns_steps,
                                  muon._stream(None))


def test_rejects_problems_beyond_the_static_scratch():
    # one 4096 x 4096 matrix needs ~128 MiB of scratch: refused before any
    # device work (fake addresses are never touched)
    L = muon.lib()
    assert muon.ns5_workspace_size(1, 4096, 4096) > muon.NOALLOC_SCRATCH_BYTES
    st = L.ns5_noalloc(ctypes.c_void_p(0x100000), muon.MUON_BF16, ctypes.c_void_p(0x40000000),
                       1, 4096, 4096, 5, None)
    assert st == muon.MUON_ERR_SCRATCH_LIMIT
    assert "static scratch" in muon.muon_status_str(st)
    assert L.ns5_noalloc(None, muon.MUON_BF16, None, 0, 8, 8, 5, None) == muon.MUON_OK


@pytest.mark.gpu
def test_noalloc_matches_ns5_on_two_calls_in_a_row():
    rng = np.random.default_rng(2024)
    cases = [
        torch.from_numpy(rng.standard_normal((3, 300, 100)).astype(np.float32)).cuda(),
        torch.from_numpy(rng.standard_normal((2, 256, 512)).astype(np.float32)).cuda().to(torch.bfloat16),
    ]
    for G in cases:
        assert muon.ns5_workspace_size(*G.shape) <= muon.NOALLOC_SCRATCH_BYTES
        out = torch.empty(G.shape, dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(G, out) == muon.MUON_OK
        ref = muon.ns5(G, 5)
        torch.cuda.synchronize()
        got, want = bf16_np(out), bf16_np(ref)
        assert rel(got, want) <= TOL_REL_BF16
        assert np.abs(got - want).max() <= TOL_MAXABS_BF16
        # same kernels, same arithmetic: the results are in fact identical
        assert torch.equal(out, ref)


@pytest.mark.gpu
def test_noalloc_calls_allocate_no_device_memory():
    rng = np.random.default_rng(7)
    G = torch.from_numpy(rng.standard_normal((2, 384, 640)).astype(np.float32)).cuda()
    out = torch.empty(G.shape, dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(G, out) == muon.MUON_OK  # loads the module, reserves the array
    torch.cuda.synchronize()
    held, (free, _) = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()
    for _ in range(2):
        assert call_noalloc(G, out) == muon.MUON_OK
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == held
    assert torch.cuda.mem_get_info()[0] == free


@pytest.mark.gpu
def test_noalloc_status_reports_ok_nonfinite_and_timeout():
    """ns5_noalloc_status reads the status word inside the static array: OK
    after a finite call, the non-finite warning after a NaN input, the
    timeout after a call whose MMA warp issues nothing (bounded waits, ~10 ms),
    and OK again after a finite call."""
    rng = np.random.default_rng(11)
    G = torch.from_numpy(rng.standard_normal((1, 256, 512)).astype(np.float32)).cuda()
    out = torch.empty(G.shape, dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(G, out) == muon.MUON_OK
    assert muon.ns5_noalloc_status() == muon.MUON_OK
    Gn = G.clone()
    Gn[0, 3, 5] = float("nan")
    assert call_noalloc(Gn, out) == muon.MUON_OK
    assert muon.ns5_noalloc_status() == muon.MUON_WARN_NONFINITE
    muon.muon_set_debug("inject_stall", 1)
    muon.muon_set_debug("wait_budget_cycles", 20_000_000)
    try:
        st = call_noalloc(G, out, ns_steps=1)
        status = muon.ns5_noalloc_status()
    finally:
        muon.muon_set_debug("inject_stall", 0)
        muon.muon_set_debug("wait_budget_cycles", 4_000_000_000)
    assert st == muon.MUON_OK
    assert status == muon.MUON_ERR_DEVICE_TIMEOUT
    assert call_noalloc(G, out) == muon.MUON_OK
    assert muon.ns5_noalloc_status() == muon.MUON_OK
    assert torch.equal(out, muon.ns5(G, 5))
