"""Pins for the FLOP and byte accounting against figures the pages print."""
import json
import os

from dense_gemm_10_gb300 import metrics

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def test_flops_4096_matches_pages():
    g = GOLDEN["flops_4096_cubed"]
    f = metrics.flops(g["M"], g["N"], g["K"])
    assert f == 137438953472
    for printed, half_unit in g["printed"]:
        assert abs(f - printed) <= half_unit


def test_naive_traffic_blowup_matches_page():
    """One thread per output reads a K-long row of A and column of B: M*N*K reads per operand."""
    g = GOLDEN["naive_traffic_1024_cubed"]
    naive = g["M"] * g["N"] * g["K"] * g["elem_bytes"]
    ideal = g["M"] * g["K"] * g["elem_bytes"]
    assert abs(naive - g["naive_bytes_per_operand_printed"]) / g["naive_bytes_per_operand_printed"] < 0.08
    assert abs(ideal - g["ideal_bytes_per_operand_printed"]) / g["ideal_bytes_per_operand_printed"] < 0.05
    assert naive // ideal == g["blowup_printed"]


def test_intensity_4096_16bit_matches_page():
    g = GOLDEN["intensity_4096_cubed_16bit"]
    ai = metrics.arithmetic_intensity(g["M"], g["N"], g["K"], "f16", "f16")
    assert abs(ai - g["printed"]) / g["printed"] <= g["rel_tol"]


def test_algorithmic_bytes_counts_c_read_only_with_beta():
    b0 = metrics.algorithmic_bytes(4096, 4096, 4096, "bf16", "f32", 0.0)
    b1 = metrics.algorithmic_bytes(4096, 4096, 4096, "bf16", "f32", 0.5)
    assert b0 == 2 * 4096 * 4096 * 2 + 4096 * 4096 * 4
    assert b1 - b0 == 4096 * 4096 * 4


def test_lm_head_bytes():
    # 64 x 4096 activations + 32000 x 4096 weights (bf16) + 64 x 32000 fp32 outputs
    assert metrics.algorithmic_bytes(64, 32000, 4096) == 64 * 4096 * 2 + 32000 * 4096 * 2 + 64 * 32000 * 4
