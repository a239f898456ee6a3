"""The benchmark's host-side arithmetic on CPU: the roofline traffic read back from the
committed ncu summaries, the choice between the HBM and the tensor bound, and the
algorithmic byte and flop counts per kernel."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _metric(path, key):
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    for line in open(path):
        if line.startswith("| " + key + " |"):
            val, unit = line.split("|")[2].split()
            return float(val) * scale[unit]
    raise KeyError(key)


@pytest.mark.parametrize("name", sorted(bench.PROFILE_OF))
def test_profiled_traffic_is_read_plus_write_of_the_summary(name):
    path = os.path.join(ROOT, "profiles", bench.PROFILE_OF[name])
    traffic, state = bench.profiled_traffic(name)
    expect = _metric(path, "dram__bytes_read.sum") + _metric(path, "dram__bytes_write.sum")
    assert traffic == pytest.approx(expect, rel=1e-12)
    assert re.fullmatch(r"commit [0-9a-f]{7,40}", state), state


def test_unknown_kernel_has_no_traffic():
    assert bench.profiled_traffic("no_such_kernel") == (None, None)


def test_roofline_takes_the_closer_bound():
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
    # an HBM-bound kernel (no flops): the HBM bound
    r = bench.roofline_of("k", {"achieved_gbs": 3400.0}, peaks, split3=True)
    assert (r["bound"], r["frac"]) == ("hbm", 0.5)
    # a contraction far from its tensor peak but near the bandwidth: still HBM
    r = bench.roofline_of("g", {"achieved_gbs": 5100.0, "achieved_tflops": 60.0}, peaks, split3=True)
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(0.75)
    # the three-term split runs three bf16 products: its tensor peak is a third of bf16's
    r = bench.roofline_of("g", {"achieved_gbs": 100.0, "achieved_tflops": 570.0}, peaks, split3=True)
    assert r["bound"] == "tensor" and r["peak"] == pytest.approx(1900.0 / 3) and r["frac"] == pytest.approx(0.9)
    r = bench.roofline_of("g", {"achieved_gbs": 100.0, "achieved_tflops": 570.0}, peaks, split3=False)
    assert r["peak"] == pytest.approx(1900.0) and r["frac"] == pytest.approx(0.3)
    # GEMMs are timed inside the step: the sustained bf16 figure when there is one
    r = bench.roofline_of("g", {"achieved_gbs": 100.0, "achieved_tflops": 510.0},
                          dict(peaks, bf16_tflops_sustained=1700.0), split3=False)
    assert r["peak"] == pytest.approx(1700.0) and r["frac"] == pytest.approx(0.3)


def test_kernel_table_counts_the_path_bytes():
    P, N = 128, 256
    t = bench.kernel_table(P, N, 4, 4, False)
    # the reverse scan reads g, c, a, h and writes the four seeds, fp32
    assert t["bwd_scan"]["bytes"] == 8 * N * 4
    # with a window it also reads R
    assert bench.kernel_table(P, N, 4, 4, True)["bwd_scan"]["bytes"] == 9 * N * 4
    # the forward scan reads a, u and writes h; the input projection reads xhat, writes a, u, c
    assert t["fwd_scan"]["bytes"] == 3 * N * 4
    assert t["proj_in"]["bytes"] == P * 4 + 3 * N * 4 and t["proj_in"]["flops"] == 2 * P * 3 * N
    # bf16 seeds halve the seed bytes of the reverse scan's writes
    assert bench.kernel_table(P, N, 2, 2, False)["bwd_scan"]["bytes"] == 4 * N * 4 + 4 * N * 2
