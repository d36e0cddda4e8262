"""The FLOP and byte counts against the numbers the pages print for their
worked example (tests/golden/roofline_worked_example.txt, with citations)."""
import math
import os

import pytest

from dense_gemm_14_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "roofline_worked_example.txt")


def golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val, tol = line.split()
            out[key] = (float(val), float(tol))
    return out


def close(x, key, g):
    val, tol = g[key]
    assert math.isclose(x, val, rel_tol=tol, abs_tol=0 if tol else 1e-12), (key, x, val)


def test_exact_integer_counts():
    assert roofline.flops(3072, 3072, 3072) == 57_982_058_496
    assert roofline.flops(256, 256, 256) == 33_554_432
    assert roofline.ideal_bytes(3072, 3072, 3072) == 113_246_208
    assert roofline.no_reuse_bytes(3072, 3072, 3072) == 231_928_233_984
    # mixed element sizes: bf16 in, fp32 out
    assert roofline.ideal_bytes(8192, 8192, 8192, 2, 4) == 536_870_912
    assert roofline.ideal_bytes(16384, 11008, 4096, 2, 4) == 945_815_552


def test_worked_example_numbers():
    g = golden()
    n = int(g["n"][0])
    peak, bw, l2 = 26.7e12, 360e9, 2500e9
    close(roofline.no_reuse_bytes(n, n, n) and 2 * n ** 3 / (8 * n ** 3), "oi_naive", g)
    close(peak / bw / 1e0, "ridge_flop_per_byte", g)
    ridge = float(f"{peak / bw:.2f}")
    assert math.ceil(ridge * 6) in (int(g["crossover_n"][0]), int(g["crossover_n"][0]) + 1)
    assert abs(ridge * 6 - g["crossover_n"][0]) < 1
    close(roofline.flops(n, n, n), "flops", g)
    close(roofline.flops(n, n, n) / peak * 1e3, "t_compute_ms", g)
    close(roofline.ideal_bytes(n, n, n) / 1e6, "ideal_bytes_mb", g)
    close(roofline.ideal_bytes(n, n, n) / bw * 1e3, "t_ideal_dram_ms", g)
    close(roofline.no_reuse_bytes(n, n, n) / 1e9, "no_reuse_bytes_gb", g)
    printed_gb = g["no_reuse_bytes_gb"][0]
    close(printed_gb * 1e9 / bw * 1e3, "t_no_reuse_dram_ms", g)
    close(printed_gb * 1e9 / l2 * 1e3, "t_no_reuse_l2_ms", g)
    assert math.isclose(roofline.intensity(n, n, n), n / 6)


def test_measured_throughput_arithmetic():
    g = golden()
    n = int(g["n"][0])
    f = roofline.flops(n, n, n)
    close(f / (g["l1_3072_ms"][0] * 1e-3) / 1e12, "l1_3072_tflops", g)
    close(f / (g["l1reg_3072_ms"][0] * 1e-3) / 1e12, "l1reg_3072_tflops", g)
    close(g["l1_3072_ms"][0] / g["l1reg_3072_ms"][0], "speedup_l1_to_l1reg", g)


def test_gb300_fp32_peak_from_unit_counts():
    assert roofline.fp32_alu_peak_tflops() == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
    assert roofline.fp32_alu_peak_tflops() == pytest.approx(80.55, rel=1e-3)


def test_measured_peaks_fallback(tmp_path):
    p = roofline.measured_peaks(str(tmp_path / "missing.json"))
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0
    f = tmp_path / "peaks.json"
    f.write_text('{"hbm_gbs": 6765.3, "bf16_tflops": 1939.3, "bf16_tflops_sustained": 1711.4}')
    p = roofline.measured_peaks(str(f))
    assert p["source"] == "measured" and p["bf16_tflops"] == 1939.3
