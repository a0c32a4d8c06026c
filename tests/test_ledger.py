"""The cost ledger against the numbers the pages print."""
import json
import os

import pytest

from dense_tiled_gemm_fp16_gb300 import ledger

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def g():
    with open(os.path.join(GOLDEN, "ledger.json")) as f:
        return json.load(f)


def test_square_min_traffic_and_naive_reads():
    d = g()
    n = 4096
    assert ledger.min_bytes(n, n, n) / 2 ** 20 == d["square_4096_min_traffic_MiB"]
    naive = 2 * n ** 3 * 2  # every output re-reads a row of A and a column of B
    assert naive / 1e9 == pytest.approx(d["square_4096_naive_read_GB_approx"], rel=0.01)
    # square AI = 2M/(3b)
    assert ledger.intensity(n, n, n) == pytest.approx(2 * n / (3 * 2))


def test_stage_accumulator_and_istage():
    d = g()
    assert ledger.stage_bytes(128, 128, 32) == d["stage_bytes_128x128x32"]
    assert 3 * ledger.stage_bytes(128, 128, 32) == d["stage_bytes_3_stages"]
    assert 128 * 128 == d["accumulator_elements_128x128"]
    assert 128 * 128 // 128 == d["accumulator_per_thread_128_threads"]
    assert ledger.stage_intensity(64, 64) == d["istage_64"]
    assert ledger.stage_intensity(128, 128) == d["istage_128"]
    assert ledger.accumulator_bytes(64, 64) == d["acc_bytes_64"]
    assert ledger.accumulator_bytes(128, 128) == d["acc_bytes_128"]


def test_moe_throughput_numbers_agree_with_2mnk():
    d = g()
    f = ledger.flops(d["moe_M"], d["moe_N"], d["moe_K"])
    assert f / (d["moe_tilelang_ms"] * 1e-3) / 1e12 == pytest.approx(d["moe_tilelang_tflops"], rel=1e-6)
    assert f / (d["moe_blas_ms"] * 1e-3) / 1e12 == pytest.approx(d["moe_blas_tflops"], rel=1e-6)


def test_roofline_bound_classification():
    # 4096^3 sits far above the machine balance, decode-like M=16 far below it
    assert ledger.bound(4096, 4096, 4096, 1905.4, 6782.8) == "tensor"
    assert ledger.bound(16, 16384, 8192, 1905.4, 6782.8) == "hbm"
    r = ledger.roofline_tflops(16, 16384, 8192, 1905.4, 6782.8)
    assert r == pytest.approx(ledger.intensity(16, 16384, 8192) * 6.7828)
