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
