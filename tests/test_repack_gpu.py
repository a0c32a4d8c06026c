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
    # (M, N, K, layout of A, layout of B, expected repack bits; 4: C, whose width
    # N is not a multiple of 8 here, goes out through the aligned buffer)
    (130, 70, 65, "row", "row", 7),          # pitches 130 B and 140 B
    (130, 70, 65, "row", "col", 7),          # B a transposed view of [70, 65]
    (300, 260, 200, "offset", "pitch", 7),   # unaligned base, unaligned pitch
    (257, 129, 300, "col", "offset", 7),     # A MN-major with an odd pitch
    (200, 190, 150, "strided", "strided", 7),  # no unit stride: element copies
    (520, 700, 384, "pitch16", "pitch", 6),  # only B needs the copy
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
    assert p["repack"] == 7 and p["b_tma"] and p["gated"], p
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


def _padded_out(M, N, ldc, offset=0):
    """C as an M x N view of a NaN-filled device buffer: row pitch ldc, base
    `offset` elements past the buffer's start."""
    buf = torch.full((M * ldc + offset + 8,), float("nan"), dtype=torch.float16, device=DEV)
    return buf, buf[offset:offset + M * ldc].view(M, ldc)[:, :N]


def _check_view_and_padding(buf, view, ref, what):
    got = view.cpu().numpy()
    assert_bits(got, ref, what)
    # every element of the buffer outside the view is still NaN
    mask = torch.ones_like(buf, dtype=torch.bool)
    M, N = view.shape
    ldc = view.stride(0)
    start = view.storage_offset()
    idx = start + torch.arange(M, device=DEV)[:, None] * ldc + torch.arange(N, device=DEV)[None, :]
    mask[idx.reshape(-1)] = False
    assert torch.isnan(buf[mask].float()).all(), f"{what}: an element outside the view was written"


OUT_CASES = [
    # (M, N, K, ldc, base offset in elements, options)
    (600, 1999, 512, 2001, 0, {}),                  # 1.2e9 FLOPs: the default plan takes the buffer
    (300, 1003, 200, 1008, 0, {g.OPT_REPACK: 2}),   # N not a multiple of 8, aligned pitch
    (300, 256, 200, 256, 1, {g.OPT_REPACK: 2}),     # base 2 bytes past a 16-byte boundary
    (1190, 1216, 2984, 1219, 0, {g.OPT_STREAMK: 2}),  # stream-K fix-up stores into the buffer
    (777, 333, 96, 333, 3, {g.OPT_REPACK: 2, g.OPT_PAIR: 1}),   # single-CTA tiles
]


@pytest.mark.parametrize("case", OUT_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-ldc{c[3]}-off{c[4]}")
def test_c_through_the_aligned_buffer(case):
    """A C that TMA cannot store in place goes out by TMA into an aligned
    buffer and is copied into the view by the unpack kernel: bit-exact, and no
    element of C's buffer outside the M x N view is written."""
    M, N, K, ldc, off, opts = case
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    rng = np.random.default_rng(M + N + K + ldc)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = torch.from_numpy(Ah).to(DEV), torch.from_numpy(Bh).to(DEV)
    buf, C = _padded_out(M, N, ldc, off)
    plan = g.plan_for(A, B, C)
    assert plan["repack"] & 4 and plan["c_tma"], plan
    g.matmul(A, B, out=C)
    torch.cuda.synchronize()
    _check_view_and_padding(buf, C, oracle.gemm(Ah, Bh, threads=oracle_threads()), f"C via buffer {case}")
    assert g.gemm_f16_device_status() == 0


def test_c_through_the_aligned_buffer_batched_grouped_fused():
    g.gemm_f16_set_option(g.OPT_REPACK, 2)
    rng = np.random.default_rng(9)
    # batched: each problem's C padded by 3 elements (batch stride not a 16-byte multiple)
    nb, M, N, K = 3, 300, 256, 128
    Ah = rng.integers(-3, 4, (nb, M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (nb, K, N)).astype(np.float16)
    cbuf = torch.full((nb * (M * N + 3),), float("nan"), dtype=torch.float16, device=DEV)
    C3 = cbuf.as_strided((nb, M, N), (M * N + 3, N, 1))
    g.bmm(torch.from_numpy(Ah).to(DEV), torch.from_numpy(Bh).to(DEV), out=C3)
    torch.cuda.synchronize()
    ref = oracle.gemm_batched(Ah, Bh)
    for b in range(nb):
        assert_bits(C3[b].cpu().numpy(), ref[b], f"batched via buffer, problem {b}")
        assert torch.isnan(cbuf[b * (M * N + 3) + M * N:(b + 1) * (M * N + 3)].float()).all()
    # grouped, odd ldc; groups end inside tiles (per-thread stores into the buffer there)
    rows = [130, 77, 301]
    G, N, K = len(rows), 256, 96
    Ah = rng.integers(-3, 4, (sum(rows), K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (G, K, N)).astype(np.float16)
    buf, C = _padded_out(sum(rows), N, N + 1)
    g.grouped_mm(torch.from_numpy(Ah).to(DEV), torch.from_numpy(Bh).to(DEV), rows, out=C)
    torch.cuda.synchronize()
    _check_view_and_padding(buf, C, oracle.gemm_grouped(Ah, Bh, rows), "grouped via buffer")
    # fused bias + ReLU, odd ldc
    M, N, K = 400, 300, 200
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    bias = rng.integers(-3, 4, (N,)).astype(np.float16)
    buf, C = _padded_out(M, N, N + 5)
    g.fused_mm(torch.from_numpy(Ah).to(DEV), torch.from_numpy(Bh).to(DEV), act="relu",
               bias=torch.from_numpy(bias).to(DEV), out=C)
    torch.cuda.synchronize()
    _check_view_and_padding(buf, C, oracle.gemm_fused(Ah, Bh, act="relu", bias=bias), "fused via buffer")
    assert g.gemm_f16_device_status() == 0


@pytest.mark.parametrize("N", [1, 9, 255, 256, 257, 511, 513, 1000])
def test_c_copy_every_alignment_offset(N):
    """The C copy for every 2-byte offset of the view's base inside a 16-byte
    word (offsets 0..7 elements) and ragged segment ends: the view bit for bit,
    nothing outside it written."""
    g.gemm_f16_set_option(g.OPT_REPACK, 2)
    rng = np.random.default_rng(N)
    M, K = 200, 64   # (M > 64: no swapped plan)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = torch.from_numpy(Ah).to(DEV), torch.from_numpy(Bh).to(DEV)
    ref = oracle.gemm(Ah, Bh)
    for off in range(8):
        ldc = N + 3 + off   # a pitch that is not a multiple of 8 for most offsets
        buf, C = _padded_out(M, N, ldc, off)
        plan = g.plan_for(A, B, C)
        assert plan["repack"] & 4 and not plan["swap_ab"], plan
        g.matmul(A, B, out=C)
        torch.cuda.synchronize()
        _check_view_and_padding(buf, C, ref, f"N={N} offset={off}")
    assert g.gemm_f16_device_status() == 0
