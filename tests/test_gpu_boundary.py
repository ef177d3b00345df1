"""GPU checks of the C ABI's promises around preparation (include/muon.h):

* a call whose preparation fails (every tensor-map encode made to fail
  through the "fail_tensor_map_encode" debug knob) returns an error and has
  enqueued nothing: the workspace's status word and every buffer keep the
  bytes they held before the call;
* a prepared call reused from the cache gives the same result, bit for bit,
  as a freshly prepared one, and still checks the workspace size;
* lr, momentum and nesterov are not part of the cache key: changing them
  between calls on the same buffers takes effect.
"""

import ctypes

import numpy as np
import pytest
import torch

from newton_schulz_08_gb300 import muon
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(256, 256), (300, 100), (100, 300)]


def bank(seed):
    rng = np.random.default_rng(seed)
    P = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(0.02)) for s in SHAPES]
    G = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(1e-3), torch.bfloat16) for s in SHAPES]
    B = [to_dev(rng.standard_normal(s).astype(np.float32) * np.float32(1e-3)) for s in SHAPES]
    return P, G, B


def test_failed_preparation_enqueues_nothing():
    P, G, B = bank(1)
    ws = muon.new_workspace(muon.muon_workspace_size(SHAPES))
    ws.fill_(0xAB)
    before = [x.clone() for x in P + B]
    torch.cuda.synchronize()
    muon.muon_plan_cache_clear()
    muon.muon_set_debug("fail_tensor_map_encode", 1)
    try:
        with pytest.raises(muon.MuonError) as e:
            muon.muon_step(P, G, B, workspace=ws)
        assert e.value.status == muon.MUON_ERR_CUDA
        Gn = torch.randn((2, 128, 192), device="cuda")
        wn = muon.new_workspace(muon.ns5_workspace_size(2, 128, 192))
        wn.fill_(0xAB)
        with pytest.raises(muon.MuonError):
            muon.ns5(Gn, 5, workspace=wn)
    finally:
        muon.muon_set_debug("fail_tensor_map_encode", 0)
    torch.cuda.synchronize()
    # the status word is cleared first thing when a call is enqueued: it is
    # untouched, and so is every buffer
    assert bool((ws == 0xAB).all())
    assert bool((wn == 0xAB).all())
    for x, x0 in zip(P + B, before):
        assert torch.equal(x, x0)
    # the same call now prepares normally
    muon.muon_step(P, G, B, workspace=ws)
    assert muon.muon_device_status(ws) == muon.MUON_OK


def test_cached_call_equals_fresh_call():
    P1, G, B1 = bank(2)
    P2, B2 = [p.clone() for p in P1], [b.clone() for b in B1]
    ws = muon.new_workspace(muon.muon_workspace_size(SHAPES))
    muon.muon_plan_cache_clear()
    for _ in range(3):  # first call prepares, the others reuse
        muon.muon_step(P1, G, B1, workspace=ws)
    for _ in range(3):  # prepared afresh every time
        muon.muon_plan_cache_clear()
        muon.muon_step(P2, G, B2, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(P1 + B1, P2 + B2):
        assert torch.equal(a, b)


def test_cached_call_still_checks_workspace_size():
    P, G, B = bank(3)
    need = muon.muon_workspace_size(SHAPES)
    ws = muon.new_workspace(need)
    muon.muon_step(P, G, B, workspace=ws)  # prepared and cached
    arr, n = muon._descs(P, G, B)
    st = muon.lib().muon_step(arr, n, 0.02, 0.95, 1, 5, ctypes.c_void_p(ws.data_ptr()), need - 1,
                              muon._stream(None))
    assert st == muon.MUON_ERR_WORKSPACE_TOO_SMALL


def test_scalars_are_not_part_of_the_key():
    """Same buffers, different lr / momentum / nesterov: each call must use
    its own scalars (compared with a call prepared afresh)."""
    P1, G, B1 = bank(4)
    P2, B2 = [p.clone() for p in P1], [b.clone() for b in B1]
    ws = muon.new_workspace(muon.muon_workspace_size(SHAPES))
    settings = [(0.02, 0.95, True), (0.05, 0.9, False), (0.0, 0.0, True)]
    muon.muon_plan_cache_clear()
    for lr, mu, nest in settings:
        muon.muon_step(P1, G, B1, lr=lr, momentum=mu, nesterov=nest, workspace=ws)
    for lr, mu, nest in settings:
        muon.muon_plan_cache_clear()
        muon.muon_step(P2, G, B2, lr=lr, momentum=mu, nesterov=nest, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(P1 + B1, P2 + B2):
        assert torch.equal(a, b)
