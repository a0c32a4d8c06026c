"""The padding form of boundary handling: operands TMA cannot address are
copied once into an aligned buffer (AI-infra page, section 05: mask or pad,
counting the extra storage), then read through TMA.

Every case forces or relies on the copy and compares with the oracle (bit for
bit on integer inputs); the plan must report the copy and TMA operands.
"""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from synth import workloads
from tests.parity import assert_bits, assert_close, oracle_threads, sampled_reference
from tests.test_gemm_gpu import make_view

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for o in (g.OPT_FORCE_GATHER, g.OPT_SPLITS, g.OPT_TILE_N, g.OPT_PANEL, g.OPT_SWAP,
              g.OPT_TIMEOUT_MS, g.OPT_MAX_CTAS, g.OPT_PAIR, g.OPT_STREAMK, g.OPT_TAIL_SPLIT, g.OPT_MAX_STAGES,
              g.OPT_REPACK):
        g.gemm_f16_set_option(o, 0)


CASES = [
    # (M, N, K, layout of A, layout of B, expected repack bits)
    (130, 70, 65, "row", "row", 3),          # pitches 130 B and 140 B
    (130, 70, 65, "row", "col", 3),          # B a transposed view of [70, 65]
    (300, 260, 200, "offset", "pitch", 3),   # unaligned base, unaligned pitch
    (257, 129, 300, "col", "offset", 3),     # A MN-major with an odd pitch
    (200, 190, 150, "strided", "strided", 3),  # no unit stride: element copies
    (520, 700, 384, "pitch16", "pitch", 2),  # only B needs the copy
    (1000, 512, 136, "pitch", "pitch16", 1),  # only A; pair tiles afterwards
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-{c[4]}")
def test_forced_copy_matches_oracle(case):
    M, N, K, la, lb, bits = case
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = make_view(Ah, la), make_view(Bh, lb)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    g.gemm_f16_set_option(g.OPT_REPACK, 2)
    plan = g.plan_for(A, B, out)
    assert plan["repack"] == bits and plan["a_tma"] and plan["b_tma"], plan
    g.matmul(A, B, out=out)
    torch.cuda.synchronize()
    assert_bits(out.cpu().numpy(), oracle.gemm(Ah, Bh, threads=oracle_threads()), f"copied operands {case}")
    # the source views are left as they were
    assert np.array_equal(A.cpu().numpy().view(np.uint16), Ah.view(np.uint16))
    assert g.gemm_f16_device_status() == 0


def test_copy_is_the_default_for_large_products_only():
    rng = np.random.default_rng(3)
    small = make_view(rng.integers(-3, 4, (130, 65)).astype(np.float16), "pitch")
    smallb = make_view(rng.integers(-3, 4, (65, 70)).astype(np.float16), "pitch")
    out = torch.empty((130, 70), dtype=torch.float16, device=DEV)
    assert g.plan_for(small, smallb, out)["repack"] == 0
    A = make_view(rng.integers(-3, 4, (1000, 1000)).astype(np.float16), "pitch")
    B = make_view(rng.integers(-3, 4, (1000, 1000)).astype(np.float16), "offset")
    out = torch.empty((1000, 1000), dtype=torch.float16, device=DEV)
    assert g.plan_for(A, B, out)["repack"] == 3
    g.gemm_f16_set_option(g.OPT_REPACK, 1)
    assert g.plan_for(A, B, out)["repack"] == 0
    g.gemm_f16_set_option(g.OPT_REPACK, 0)
    g.gemm_f16_set_option(g.OPT_FORCE_GATHER, 3)   # a forced gather is never replaced
    assert g.plan_for(A, B, out)["repack"] == 0


def test_copy_with_batches_groups_and_gate_up():
    rng = np.random.default_rng(5)
    g.gemm_f16_set_option(g.OPT_REPACK, 2)
    # batched, batch strides not 16-byte multiples (each problem padded by 3 elements)
    nb, M, N, K = 4, 140, 96, 72
    Ah = rng.integers(-3, 4, (nb, M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (nb, K, N)).astype(np.float16)
    Abuf = torch.zeros((nb, M * K + 3), dtype=torch.float16)
    Bbuf = torch.zeros((nb, K * N + 3), dtype=torch.float16)
    Abuf[:, :M * K] = torch.from_numpy(Ah.reshape(nb, -1))
    Bbuf[:, :K * N] = torch.from_numpy(Bh.reshape(nb, -1))
    A = Abuf.to(DEV).as_strided((nb, M, K), (M * K + 3, K, 1))
    B = Bbuf.to(DEV).as_strided((nb, K, N), (K * N + 3, N, 1))
    C = g.bmm(A, B)
    torch.cuda.synchronize()
    ref = oracle.gemm_batched(Ah, Bh)
    for b in range(nb):
        assert_bits(C[b].cpu().numpy(), ref[b], f"batched copy problem {b}")
    # grouped, B group stride odd
    rows = [130, 0, 77, 300]
    G, N, K = len(rows), 136, 90
    Ah = rng.integers(-3, 4, (sum(rows), K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (G, K, N)).astype(np.float16)
    Bbuf = torch.zeros((G, K * N + 5), dtype=torch.float16)
    Bbuf[:, :K * N] = torch.from_numpy(Bh.reshape(G, -1))
    B = Bbuf.to(DEV).as_strided((G, K, N), (K * N + 5, N, 1))
    C = g.grouped_mm(torch.from_numpy(Ah).to(DEV), B, rows)
    torch.cuda.synchronize()
    assert_bits(C.cpu().numpy(), oracle.gemm_grouped(Ah, Bh, rows), "grouped copy")
    # gate/up with unaligned projections: both are copied
    M, N, K = 130, 70, 65
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    Uh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B, U = (torch.from_numpy(x).to(DEV) for x in (Ah, Bh, Uh))
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    p = g.fused_plan_for(A, B, out, act="relu", b_up=U)
    assert p["repack"] == 3 and p["b_tma"] and p["gated"], p
    g.fused_mm(A, B, act="relu", b_up=U, out=out)
    torch.cuda.synchronize()
    assert_bits(out.cpu().numpy(), oracle.gemm_fused(Ah, Bh, Uh, act="relu"), "gate/up copy")
    assert g.gemm_f16_device_status() == 0


def test_irregular_shape_through_the_gather_at_full_size():
    """The 3001x1999x4097 configuration (A a transposed view) with the copy
    switched off: the masked gather path at full size, on sampled outputs."""
    w = workloads.IRREGULAR_3001x1999x4097
    g.gemm_f16_set_option(g.OPT_REPACK, 1)
    A, B = w.A.device_view(DEV), w.B.device_view(DEV)
    out = torch.empty((w.M, w.N), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["repack"] == 0 and not plan["a_tma"] and not plan["b_tma"], plan
    g.matmul(A, B, out=out)
    torch.cuda.synchronize()
    rng = np.random.default_rng(77)
    ms = np.concatenate([rng.integers(0, w.M, 2048), [w.M - 1] * 4, [0, 0]])
    ns = np.concatenate([rng.integers(0, w.N, 2048), [w.N - 1, 0, 1, 2], [w.N - 1, 0]])
    got = out[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)].cpu().numpy()
    assert_close(got, sampled_reference(w, ms, ns), w.K, "irregular, gathered")
    assert g.gemm_f16_device_status() == 0
