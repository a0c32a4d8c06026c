"""Host-side checks of the measurement plumbing in bench.py: the source hash
that ties a committed ncu summary to the kernel it was taken on, the traffic
lookup, the clock-sample parser and the peak table fallback."""
import os
import shutil

import pytest

import bench

SOURCES = ("ptx.cuh", "gemm_kernel.cuh", "gemm_f16.cu", "repack.cuh")


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of the kernel sources under a scratch root that bench.py reads."""
    src = os.path.join(bench.ROOT, "dense_tiled_gemm_fp16_gb300", "csrc")
    dst = tmp_path / "dense_tiled_gemm_fp16_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in SOURCES:
        shutil.copy(os.path.join(src, f), dst / f)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_source_hash_ignores_comments_and_spacing(tree):
    h0 = bench.kernel_source_hash()
    k = tree / "dense_tiled_gemm_fp16_gb300" / "csrc" / "gemm_kernel.cuh"
    text = k.read_text()
    k.write_text("// a new comment\n/* and a\n block */\n" + text.replace("\n", "\n\n", 3))
    assert bench.kernel_source_hash() == h0
    k.write_text(text.replace("kBK = 64", "kBK = 32", 1))
    assert bench.kernel_source_hash() != h0


def _summary(tree, workload, digest, nbytes):
    (tree / "profiles" / f"gemm_f16_persistent__{workload}.md").write_text(
        f"# summary\n\n```\nkernel: gemm_f16_persistent\nworkload: {workload}\n"
        f"kernel_source_sha256_16: {digest}\ndram_bytes_per_launch: {nbytes}\n```\n")


def test_traffic_only_from_a_summary_of_the_same_sources(tree):
    assert bench.profiled_traffic("square_4096") is None            # no summary
    _summary(tree, "square_4096", bench.kernel_source_hash(), 123456)
    assert bench.profiled_traffic("square_4096") == 123456
    _summary(tree, "square_4096", "0" * 16, 123456)                 # other sources
    assert bench.profiled_traffic("square_4096") is None


def test_committed_summaries_are_well_formed():
    # every committed summary names its kernel and workload, the sources' hash
    # and a positive byte count, and gives the ncu command that made it, with
    # the clocks left alone
    import re
    d = os.path.join(bench.ROOT, "profiles")
    names = [f for f in os.listdir(d) if f.startswith("gemm_f16_persistent__")]
    assert names
    for f in names:
        text = open(os.path.join(d, f)).read()
        workload = f[len("gemm_f16_persistent__"):-len(".md")]
        assert f"workload: {workload}" in text, f
        assert re.search(r"kernel_source_sha256_16: [0-9a-f]{16}\b", text), f
        assert int(re.search(r"dram_bytes_per_launch: (\d+)", text).group(1)) > 0, f
        cmds = [line for line in text.splitlines() if line.startswith("ncu ")]
        assert cmds and all("--clock-control none" in c for c in cmds), f


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_samples_are_parsed_per_gpu(tmp_path):
    rows = [
        "0, GPU-a, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, GPU-a, 1950, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, GPU-a, 300, 2070, 90.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # idle sample
        "1, GPU-b, 1000, 2070, 1400.0, 0x40, Active, Not Active, Not Active, Not Active",   # another GPU
        "garbage line",
    ]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler("GPU-a")
    s.proc, s.path = _Done(), str(path)
    c = s.stop()
    assert c["samples"] == 3
    assert c["sm_max_mhz"] == 2070.0
    assert c["sm_mhz"] == pytest.approx((2070 + 1950) / 2)      # median of the loaded samples
    assert c["reasons"] == ["sw_power_cap"]                        # GPU-b's hw_slowdown is not ours
    assert not path.exists()


def test_peaks_fall_back_when_no_measurement_is_present(tree):
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["tflops"] > 0 and p["hbm_gbs"] > 0
    (tree / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6782.8, "bf16_tflops": 1905.4}')
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["tflops"] == 1905.4 and p["tflops_sustained"] == 1905.4


def test_whole_job_rate_counts_every_replica():
    # 3 steps of 2e9 FLOPs on each of 4 replicas in 6 ms (the slowest rank)
    assert bench.whole_job_rate(2e9, 3, 4, 6.0) == pytest.approx(2e9 * 3 * 4 / 6e-3)


def test_cpu_baseline_runs_the_oracle_on_the_workload_itself():
    # the slab the CPU baseline times is the workload's own product: on the
    # small tail case the slab covers every row and equals the oracle's C
    import numpy as np

    import oracle
    from synth import workloads

    oracle.build()
    for name in ("tail_130x70x65_b_rowmajor", "tail_130x70x65_b_transposed"):
        w = workloads.BY_NAME[name]
        run, flops = bench.oracle_slab(w, w.M, threads=1)
        assert flops == 2.0 * w.M * w.N * w.K
        want = oracle.gemm(np.ascontiguousarray(w.A.host_view()), w.B.host_view())
        assert np.array_equal(run().view(np.uint16), want.view(np.uint16)), name
        rate, rows, dt, reps = bench.cpu_oracle_rate(w, 0.05, threads=1)
        assert rows == w.M and reps >= 1 and dt > 0 and rate > 0


def test_roofline_rates_against_burst_and_sustained_peaks():
    peaks = {"tflops": 2000.0, "tflops_sustained": 1600.0, "hbm_gbs": 8000.0, "source": "measured"}
    # 2e12 FLOPs in 1.25 ms: 1600 TFLOP/s, 0.8 of the burst peak, 1.0 of the sustained one
    r = bench.roofline("tensor", 2e12, 1e9, 1.25, peaks, "no_such_workload", busy_ms=25.0)
    assert r["unit"] == "TFLOP/s" and r["peak_kind"] == "burst" and r["peak"] == 2000.0
    assert r["achieved"] == pytest.approx(1600.0) and r["frac"] == pytest.approx(0.8)
    assert r["frac_of_sustained"] == pytest.approx(1.0) and r["traffic"] is None
    # a timed region long enough to run under the power limit: the sustained peak
    r = bench.roofline("tensor", 2e12, 1e9, 1.25, peaks, "no_such_workload", busy_ms=250.0)
    assert r["peak_kind"] == "sustained" and r["peak"] == 1600.0 and r["frac"] == pytest.approx(1.0)
    assert r["frac_of_burst"] == pytest.approx(0.8)
    # 4e8 bytes in 0.1 ms: 4000 GB/s, half of the copy bandwidth
    r = bench.roofline("hbm", 1e9, 4e8, 0.1, peaks, "no_such_workload")
    assert r["unit"] == "GB/s" and r["achieved"] == pytest.approx(4000.0) and r["frac"] == pytest.approx(0.5)


def test_cpu_baseline_labels_its_sample_and_adds_a_single_thread_run():
    import oracle
    from synth import workloads

    oracle.build()
    w = workloads.BY_NAME["tail_130x70x65_b_rowmajor"]
    cpu = bench.cpu_baseline(w, 0.05, 2)
    assert cpu["kind"] == "oracle" and cpu["cores"] == 2 and cpu["value"] > 0
    assert cpu["full_workload_s_kind"] == "measured"       # the slab is the whole product
    assert cpu["single_thread"]["cores"] == 1 and cpu["single_thread"]["value"] > 0
    big = workloads.BY_NAME["square_4096"]                   # not a single-thread workload
    cpu = bench.cpu_baseline(big, 0.05, 1)
    assert "single_thread" not in cpu and cpu["full_workload_s_kind"].startswith("extrapolated")
    assert cpu["full_workload_s"] > 0


def test_vs_baseline_only_for_the_pages_own_workload():
    # the pages measured only the MoE-flattened shape (117.25 TFLOPS on a C500)
    v, ref = bench.vs_pages("moe_131072x2048x7168", 1800.0, "TFLOP/s")
    assert v == pytest.approx(1800.0 / 117.25, abs=1e-3) and "C500" in ref
    assert bench.vs_pages("square_4096", 1500.0, "TFLOP/s") == (None, None)
    assert bench.vs_pages("moe_131072x2048x7168", 1800.0, "GB/s") == (None, None)
