"""Debug bounds checking (GEMM_F16_OPT_DEBUG_BOUNDS): with it on, every
gathered operand load and every per-thread store of C is checked against the
byte range its view spans.  Correct plans must run clean (status 0, results
bit-exact); the checker's own test shrinks every range by 16 bytes, so the
accesses to the last 8 elements, which lie inside the real views, are reported
(GEMM_F16_ERR_BOUNDS) and skipped.  No access ever leaves a view: the check
only removes accesses."""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from tests.parity import assert_bits
from tests.test_gemm_gpu import make_view

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
OPTIONS = (g.OPT_FORCE_GATHER, g.OPT_SPLITS, g.OPT_SWAP, g.OPT_PAIR, g.OPT_STREAMK, g.OPT_REPACK,
           g.OPT_DEBUG_BOUNDS, g.OPT_TILE_N)


@pytest.fixture(autouse=True)
def _defaults():
    g.gemm_f16_device_status(reset=True)
    yield
    for o in OPTIONS:
        g.gemm_f16_set_option(o, 0)
    g.gemm_f16_device_status(reset=True)


def ints(rng, shape):
    return rng.integers(-3, 4, shape).astype(np.float16)


CASES = [
    # (M, N, K, layout of A, layout of B, options)
    (300, 260, 200, "pitch", "offset", {g.OPT_REPACK: 1}),
    (257, 129, 300, "strided", "col", {g.OPT_REPACK: 1}),
    (130, 70, 65, "row", "row", {}),
    (700, 500, 320, "row", "row", {g.OPT_FORCE_GATHER: 7}),                  # A, B gathered, C masked
    (16, 1000, 700, "pitch", "offset", {g.OPT_REPACK: 1}),                    # swapped: transposed C stores
    (900, 384, 640, "offset", "pitch", {g.OPT_REPACK: 1, g.OPT_STREAMK: 2}),  # masked fixup stores
    (600, 333, 500, "row", "strided", {g.OPT_REPACK: 1, g.OPT_SPLITS: 3, g.OPT_TILE_N: 128}),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-{c[4]}-{len(c[5])}")
def test_checked_plans_run_clean(case):
    M, N, K, la, lb, opts = case
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    g.gemm_f16_set_option(g.OPT_DEBUG_BOUNDS, 1)
    rng = np.random.default_rng(M + N + K)
    Ah, Bh = ints(rng, (M, K)), ints(rng, (K, N))
    C = g.matmul(make_view(Ah, la), make_view(Bh, lb))
    torch.cuda.synchronize()
    assert g.gemm_f16_device_status() == 0
    assert_bits(C.cpu().numpy(), oracle.gemm(Ah, Bh), f"checked {case}")


def test_checked_batched_grouped_and_fused_run_clean():
    g.gemm_f16_set_option(g.OPT_DEBUG_BOUNDS, 1)
    g.gemm_f16_set_option(g.OPT_REPACK, 1)
    rng = np.random.default_rng(71)
    nb, M, N, K = 4, 140, 96, 72   # batch strides not 16-byte multiples: gathered
    Ah, Bh = ints(rng, (nb, M, K)), ints(rng, (nb, K, N))
    Abuf = torch.zeros((nb, M * K + 3), dtype=torch.float16)
    Abuf[:, :M * K] = torch.from_numpy(Ah.reshape(nb, -1))
    A = Abuf.to(DEV).as_strided((nb, M, K), (M * K + 3, K, 1))
    C = g.bmm(A, torch.from_numpy(Bh).to(DEV))
    torch.cuda.synchronize()
    assert g.gemm_f16_device_status() == 0
    ref = oracle.gemm_batched(Ah, Bh)
    for b in range(nb):
        assert_bits(C[b].cpu().numpy(), ref[b], f"checked batched {b}")
    rows = [130, 0, 77, 301]
    Ah, Bh, Uh = ints(rng, (sum(rows), 96)), ints(rng, (4, 96, 70)), ints(rng, (4, 96, 70))
    A = torch.from_numpy(np.ascontiguousarray(Ah.T)).to(DEV).t()   # column-major A, unaligned group starts
    C = g.grouped_fused_mm(A, torch.from_numpy(Bh).to(DEV), rows, act="relu", b_up=torch.from_numpy(Uh).to(DEV))
    torch.cuda.synchronize()
    assert g.gemm_f16_device_status() == 0
    assert_bits(C.cpu().numpy(), oracle.gemm_fused_grouped(Ah, Bh, rows, Uh, act="relu"), "checked grouped fused")


def test_checker_reports_accesses_past_a_shortened_range():
    rng = np.random.default_rng(72)
    M, N, K = 300, 260, 200
    Ah, Bh = ints(rng, (M, K)), ints(rng, (K, N))
    A, B = make_view(Ah, "pitch"), make_view(Bh, "offset")
    g.gemm_f16_set_option(g.OPT_REPACK, 1)
    g.gemm_f16_set_option(g.OPT_FORCE_GATHER, 4)      # C through per-thread stores as well
    g.gemm_f16_set_option(g.OPT_DEBUG_BOUNDS, 2)
    g.matmul(A, B)
    torch.cuda.synchronize()
    assert g.gemm_f16_device_status(reset=True) == g.ERR_BOUNDS
    g.gemm_f16_set_option(g.OPT_DEBUG_BOUNDS, 1)       # the true ranges: clean again
    C = g.matmul(A, B)
    torch.cuda.synchronize()
    assert g.gemm_f16_device_status() == 0
    assert_bits(C.cpu().numpy(), oracle.gemm(Ah, Bh), "after the checker's test")
