"""The wait-profile diagnostic (python -m newton_schulz_08_gb300.wait_profile)
over the library's wait_profile_buffer hook: every tile of every phase is
counted once per CTA of its pair, and the role timers run."""

import pytest

from newton_schulz_08_gb300 import wait_profile

pytestmark = pytest.mark.gpu


def test_wait_profile_counts_every_tile():
    # 512x512: 2x2 output tiles, 3 on or above the diagonal; 256x1024 (m = 256,
    # n = 1024): 1 Gram tile, 1x4 update tiles
    shapes = [(512, 512)] * 4 + [(256, 1024)] * 2
    tiles = {"gram": 4 * 3 + 2 * 1, "poly": 4 * 3 + 2 * 1, "update": 4 * 4 + 2 * 4}
    out = wait_profile.profile(shapes, steps=2)
    for phase, d in out.items():
        # per launch, summed over CTAs: both CTAs of a pair count the tile
        assert round(d["tiles"] * d["ctas"]) == 2 * tiles[phase], (phase, d)
        assert d["kernel"] > 0 and d["mma_loop"] > 0 and d["epi_busy"] > 0
        assert d["ctas"] % 2 == 0


def test_kernel_kinds_of_a_step():
    """Launches per kernel kind (the library's kernel-event hook).  A Muon step
    ends with the update that applies p -= lr O itself (update_apply) and
    launches no apply pass; ns5_bank writes O with the apply pass; a step
    with no Newton-Schulz iteration applies X0 with it.  Both classes here are
    at most 768 wide, so each phase is one launch."""
    import torch

    from newton_schulz_08_gb300 import inputs, muon
    shapes = [(512, 512), (256, 1024), (1024, 256)]
    dev = torch.device("cuda")
    P = [torch.from_numpy(inputs.param(s, i)).to(dev) for i, s in enumerate(shapes)]
    B = [torch.from_numpy(inputs.buffer(s, i)).to(dev) for i, s in enumerate(shapes)]
    G = [torch.from_numpy(inputs.grad(s, i)).to(dev).to(torch.bfloat16) for i, s in enumerate(shapes)]

    def launches(fn):
        muon.muon_set_debug("record_kernel_events", 1)
        try:
            muon.muon_kernel_times()  # drops earlier records
            fn()
            torch.cuda.synchronize()
            return {kind: n for kind, (_, n) in muon.muon_kernel_times().items()}
        finally:
            muon.muon_set_debug("record_kernel_events", 0)

    k = launches(lambda: muon.muon_step(P, G, B, ns_steps=5))
    assert (k["momentum_cast"], k["normalise"], k["gram"], k["poly"], k["update"], k["update_apply"],
            k["apply"]) == (1, 1, 5, 5, 4, 1, 0), k
    k = launches(lambda: muon.ns5_bank(G, 5))
    assert (k["gram"], k["update"], k["update_apply"], k["apply"]) == (5, 5, 0, 1), k
    k = launches(lambda: muon.muon_step(P, G, B, ns_steps=0))
    assert (k["gram"], k["update"], k["update_apply"], k["apply"]) == (0, 0, 0, 1), k
