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


@pytest.mark.parametrize("key", sorted(k for k in bench.PROFILE_OF
                                        if os.path.exists(os.path.join(ROOT, "profiles", bench.PROFILE_OF[k]))))
def test_profiled_traffic_is_read_plus_write_of_the_summary(key):
    path = os.path.join(ROOT, "profiles", bench.PROFILE_OF[key])
    traffic, state, fresh = bench.profiled_traffic(key[1], key[0])
    scale = 1.0
    for line in open(path):
        if line.startswith("Traffic scale:"):
            scale = float(line.split(":", 1)[1].split()[0])
    expect = (_metric(path, "dram__bytes_read.sum") + _metric(path, "dram__bytes_write.sum")) * scale
    assert traffic == pytest.approx(expect, rel=1e-12)
    # a summary names the library sources it was captured from; only a capture of the
    # current sources is fresh
    assert state is None or re.fullmatch(r"[0-9a-f]{16}", state), state
    assert fresh == (state == bench.source_hash(bench.KERNEL_TU.get(key[1])))


def test_unknown_kernel_has_no_traffic():
    assert bench.profiled_traffic("no_such_kernel") == (None, None, False)


def test_source_hash_is_stable():
    assert bench.source_hash() == bench.source_hash()
    assert re.fullmatch(r"[0-9a-f]{16}", bench.source_hash())
    # a kernel's hash covers its own translation unit and the headers only
    assert bench.source_hash("adj_scan.cu") != bench.source_hash("adj_gemm_tc.cu")
    for name, tu in bench.KERNEL_TU.items():
        assert os.path.exists(os.path.join(ROOT, "adjoint_gradients_long_gb300", "csrc", tu)), name


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
    # the tensor fraction is taken against the burst peak, the sustained one given beside it
    r = bench.roofline_of("g", {"achieved_gbs": 100.0, "achieved_tflops": 510.0},
                          dict(peaks, bf16_tflops_sustained=1700.0), split3=False)
    assert r["peak"] == pytest.approx(1900.0) and r["frac"] == pytest.approx(510.0 / 1900.0)
    assert r["peak_sustained"] == pytest.approx(1700.0) and r["frac_sustained"] == pytest.approx(0.3)


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


def test_kernel_table_stack_entries():
    P, N, K = 2048, 256, 4
    t = bench.kernel_table(P, N, 2, 2, True, K)
    # the normalisation's backward reads y, dxhat, gy and writes gy_prev (fp32) plus r
    assert t["rms_norm_bwd"]["bytes"] == 16 * P + 4
    # in a stack the input gradient reads D, gy, xhat, r and the row dots, and writes gy_prev
    # and its bf16 copy
    assert t["input_grad"]["bytes"] == 3 * N * 2 + 8 * P + 2 * P + 4 + 4 * 2 + 2 * P
    # the backward GEMMs read the cotangent's bf16 copy
    assert t["cot_proj"]["bytes"] == 2 * P + 4 * N and t["param_dW_o"]["bytes"] == 2 * N + 2 * P
    # proj_out: c . h read in bf16, y written, the residual read (bf16 input once, fp32
    # stream K-1 times); the forward scan reads a, u, c and writes h and c . h
    assert t["proj_out"]["bytes"] == 2 * N + 4 * P + (2 * P + 3 * 4 * P) / 4
    assert t["fwd_scan"]["bytes"] == 16 * N + 2 * N


def test_clock_summary_reads_reasons():
    lines = ["0, 1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active",
             "0, 2000, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage"]
    c = bench.summarize_clocks(lines)
    assert c["sm_mhz"] == 1950 and c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    assert c["samples"] == 2 and c["power_w_max"] == 1000.0


def test_selective_kernel_table():
    """The general selective layer: the forward scan reads z and xhat and writes h (P N
    states a token) and y; the reverse scan reads z, xhat, gy and h and writes dz."""
    P, N = 1024, 16
    t = bench.sel_kernel_table(P, N, 2, 2)
    zw = P + 2 * N
    assert t["sel_fwd"]["bytes"] == 4 * zw + 2 * P + 4 * P * N + 4 * P
    assert t["sel_bwd"]["bytes"] == 4 * zw + 2 * P + 4 * P + 4 * P * N + 2 * zw
    assert t["sel_proj"]["flops"] == 2 * P * zw and t["sel_dW"]["flops"] == 2 * P * zw
    # the state dominates: its 4 P N bytes are over four fifths of a scan's bytes a token
    assert 4 * P * N / t["sel_bwd"]["bytes"] > 0.8


def test_selective_stack_kernel_table():
    """A stack of K selective layers: layers 2..K add the residual input to the forward
    scan, r, gadd and the row dots (slices + 1 floats) to the reverse scan, and run the input
    GEMM and the normalisation once each; the table's scan counts are means over the K."""
    P, N, K = 1024, 16, 4
    one = bench.sel_kernel_table(P, N, 2, 2)
    t = bench.sel_kernel_table(P, N, 2, 2, K)
    zw, nsl = P + 2 * N, P // 128
    assert "sel_dx" not in one and "rms_norm" not in one
    assert t["sel_fwd"]["bytes"] - one["sel_fwd"]["bytes"] == (K - 1) / K * 4 * P
    assert t["sel_bwd"]["bytes"] - one["sel_bwd"]["bytes"] == (K - 1) / K * (4 + 4 * P + 4 * (nsl + 1))
    assert t["sel_dx"]["bytes"] == 2 * zw + 4 * P + 2 * P + 4 + 4 * (nsl + 1) + 4 * P
    assert t["sel_dx"]["flops"] == 2 * zw * P
    assert t["rms_norm"]["bytes"] == 4 * P + 2 * P + 4


def test_workload_arg():
    assert bench.workload_arg("ssm1_1m") == ("ssm1_1m", None)
    assert bench.workload_arg("ssm1_1m:full") == ("ssm1_1m", None)
    assert bench.workload_arg("ssm8_p512:4096") == ("ssm8_p512", 4096)
