"""The benchmark's work accounting (CPU): algorithmic and dense-equivalent
Newton-Schulz FLOPs and elementwise bytes per step, against the figures the
closed forms give for the benchmark banks, and the issued-MMA count against
a direct tile enumeration."""

import pytest

import bench

# per Muon step, 5 Newton-Schulz steps: algorithmic m(m+1)n + m^2(m+1) + 2m^2n
# and dense-equivalent 4m^2n + 2m^3 per matrix and step, summed over the bank
CASES = {
    "gpt2": (1.142e12, 1.631e12),
    "spectra": (1.375e12 + 2.199e13, 2.062e12 + 3.299e13),
    "rect": (5.820e12, 8.057e12),
    "gpt1p5b": (4.130e13, 5.898e13),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_flop_accounting(name):
    shapes = bench.workload_shapes(name)
    alg, dense = CASES[name]
    assert sum(bench.ns_flops(shapes).values()) == pytest.approx(alg, rel=1e-3)
    assert bench.ns_flops_dense(shapes) == pytest.approx(dense, rel=1e-3)


def test_issued_flops_enumerate_tiles():
    # 300 x 100: m = 100, one 256-tile, K padded to 128 (Gram: n = 300 -> 320)
    shapes = [(300, 100)]
    f = bench.ns_flops_issued(shapes, steps=1)
    assert f["gram"] == 2.0 * 256 * 256 * 320
    assert f["poly"] == 2.0 * 256 * 256 * 128
    assert f["update"] == 2.0 * 2 * 256 * 256 * 128  # 1 x 2 output tiles of the 100 x 300 X
    # 768 x 768: 3 x 3 tiles, 6 on or above the diagonal
    f = bench.ns_flops_issued([(768, 768)], steps=1)
    assert f["gram"] == f["poly"] == 2.0 * 6 * 256 * 256 * 768
    assert f["update"] == 2.0 * 9 * 256 * 256 * 768
    # issued work never falls below the algorithmic work
    for name in CASES:
        shapes = bench.workload_shapes(name)
        alg, iss = bench.ns_flops(shapes), bench.ns_flops_issued(shapes)
        assert all(iss[k] >= alg[k] for k in alg)


def test_elementwise_bytes():
    shapes = bench.workload_shapes("gpt2")
    e = sum(r * c for r, c in shapes)
    b = bench.hbm_bytes(shapes, 2)
    assert b["momentum_cast"] == 12 * e == pytest.approx(1.019e9, rel=1e-3)
    assert b["normalise"] == 4 * e
    assert b["apply"] == 10 * e
    # the last update with the parameter update: X and B read, p read and
    # written (GPT-2 bank: every matrix has m = 768)
    assert b["update_apply"] == 10 * e + len(shapes) * 2 * 768 ** 2
    b = bench.hbm_bytes(shapes, 2, ns5_only=True)
    assert b["momentum_cast"] == 4 * e and b["apply"] == 4 * e
