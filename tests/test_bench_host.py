"""The benchmark's work accounting (CPU): algorithmic and dense-equivalent
Newton-Schulz FLOPs and elementwise bytes per step, against the figures the
closed forms give for the benchmark banks, and the issued-MMA count against
a direct tile enumeration."""

import numpy as np
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


def test_kernel_report_work_per_launch():
    """Each launch of a Newton-Schulz phase does one iteration's work over
    the bank; with the last update timed as update_apply, the update kind
    holds the other NS_STEPS - 1 iterations.  Shares sum to one and each
    fraction is the achieved rate over its peak."""
    shapes = bench.workload_shapes("gpt2")
    flops, issued = bench.ns_flops(shapes), bench.ns_flops_issued(shapes)
    gbytes = bench.hbm_bytes(shapes, 2)
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 7000.0}
    steps, ns = 3, bench.NS_STEPS
    fused = {"momentum_cast": (0.5, steps), "normalise": (0.2, steps), "gram": (1.0, ns * steps),
             "poly": (0.8, ns * steps), "update": (1.6, (ns - 1) * steps), "update_apply": (0.6, steps),
             "apply": (0.0, 0)}
    k = bench.kernel_report(fused, steps, flops, issued, gbytes, peaks)
    assert "apply" not in k
    per_iter = flops["update"] / ns
    assert k["update"]["work_per_launch"] == pytest.approx(per_iter)
    assert k["update"]["launches_per_step"] == ns - 1
    assert k["gram"]["work_per_launch"] == pytest.approx(flops["gram"] / ns)
    assert k["update_apply"]["unit"] == "GB/s" and k["update_apply"]["work_per_launch"] == gbytes["update_apply"]
    assert sum(v["share"] for v in k.values()) == pytest.approx(1.0)
    for v in k.values():
        assert v["frac"] == pytest.approx(v["achieved"] / v["peak"])
    # the Newton-Schulz-only path: all NS_STEPS updates under one kind
    plain = dict(fused, update=(2.0, ns * steps), update_apply=(0.0, 0), apply=(0.3, steps))
    k = bench.kernel_report(plain, steps, flops, issued, gbytes, peaks)
    assert "update_apply" not in k
    assert k["update"]["work_per_launch"] == pytest.approx(per_iter)
    assert k["update"]["issued_tflops"] == pytest.approx(issued["update"] / ns / (2.0 / (ns * steps) * 1e-3) / 1e12)
    # flops is not modified
    assert flops == bench.ns_flops(shapes)


def test_fp8_workload_operands_and_oracle_sample():
    """The FP8 workload's operands fill E4M3 without overflow, x and its
    output exceed the 129 MB L2, and the oracle sample counts 2 N K FLOPs
    per row."""
    M, N, K = bench.FP8_SHAPE
    assert M * K * 2 > 129e6 / 2 and M * N * 2 > 129e6
    assert K % 16 == 0 and N % 8 == 0
    x, w, x_s, w_s = bench.fp8_operands(0)
    assert x.shape == (M, K) and w.shape == (N, K)
    assert np.abs(x).max() / x_s < 448 and np.abs(w).max() / w_s < 448
    f, t = bench.fp8_oracle_sample(0.0)
    assert f == 2.0 * 16 * N * K and t > 0
