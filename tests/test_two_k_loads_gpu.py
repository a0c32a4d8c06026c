"""Two K blocks per copy: each pipeline phase of a full-width tile can load both
of its 64-wide K blocks with one TMA copy per operand (a map with the K block
as an outer dimension) instead of one copy per block.  Every plan shape that
takes it, and every one that must fall back (a ragged last K block, a phase
of one block, narrow tail pieces, K below two blocks), gives the oracle's
result bit for bit on integer inputs, and the same bits as one copy per block.
"""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from tests.parity import assert_bits, oracle_threads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for o in (g.OPT_SPLITS, g.OPT_PAIR, g.OPT_STREAMK, g.OPT_TAIL_SPLIT, g.OPT_SWAP, g.OPT_TWO_K_LOADS):
        g.gemm_f16_set_option(o, 0)


def ints(rng, shape):
    return rng.integers(-3, 4, shape).astype(np.float16)


def view(x: np.ndarray, layout: str):
    """A device fp16 view of `x` [r, c]: row-major, or the transpose of a
    row-major [c, r] (column-major)."""
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(DEV) if layout == "row" else t.t().contiguous().to(DEV).t()


def run_both(call):
    """`call()` with two-block copies (default) and with one copy per block."""
    g.gemm_f16_set_option(g.OPT_TWO_K_LOADS, 0)
    c2 = call()
    torch.cuda.synchronize()
    g.gemm_f16_set_option(g.OPT_TWO_K_LOADS, 1)
    c1 = call()
    torch.cuda.synchronize()
    g.gemm_f16_set_option(g.OPT_TWO_K_LOADS, 0)
    return c2.cpu().numpy(), c1.cpu().numpy()


# (M, N, K, A layout, B layout, options, does the plan take two-block copies?)
CASES = [
    (1100, 1280, 896, "row", "row", {}, 1),                       # pair, K-major A, MN-major B (3-D boxes)
    (1100, 1288, 896, "row", "col", {}, 1),                       # pair, K-major B
    (704, 576, 296, "col", "col", {}, 1),                         # MN-major A, ragged last K block (296 = 4 * 64 + 40)
    (640, 512, 200, "row", "row", {}, 1),                         # K = 200: the second phase holds the ragged block
    (512, 640, 128, "row", "col", {}, 1),                         # exactly one two-block phase
    (512, 640, 64, "row", "col", {}, 0),                          # one K block: nothing to pair
    (704, 520, 296, "row", "row", {}, 0),                         # MN-major B of 520 columns: 2-D boxes per atom column
    (1024, 640, 1024, "row", "row", {g.OPT_PAIR: 1}, 1),          # single-CTA tiles
    (1190, 1216, 2984, "row", "col", {g.OPT_STREAMK: 2}, 1),      # stream-K units starting at odd K blocks
    (512, 512, 4096, "row", "row", {g.OPT_SPLITS: 3}, 1),         # split-K: segments of 21 and 22 blocks
    (4096, 4096, 512, "row", "row", {}, 1),                       # tail split: narrow pieces read one block per copy
    (16, 4096, 1024, "row", "row", {}, 1),                        # swapped small M on pairs (MN-major kernel A)
    (48, 2048, 520, "row", "col", {}, 1),                         # swapped, stream-K, ragged K
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}{c[4]}-{c[5]}")
def test_two_k_block_copies_match_the_oracle(case):
    M, N, K, la, lb, opts, expect = case
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    Ah, Bh = ints(rng, (M, K)), ints(rng, (K, N))
    A, B = view(Ah, la), view(Bh, lb)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["two_k_loads"] == expect, plan
    assert plan["a_tma"] and plan["b_tma"] and not plan["repack"], plan
    if case[:3] == (4096, 4096, 512):
        assert plan["tail_split"] > 1, plan
    c2, c1 = run_both(lambda: g.matmul(A, B, out=out))
    assert_bits(c2, oracle.gemm(Ah, Bh, threads=oracle_threads()), f"two-block copies {case[:6]}")
    assert_bits(c2, c1, "one copy per block")
    g.gemm_f16_set_option(g.OPT_TWO_K_LOADS, 1)
    assert g.plan_for(A, B, out)["two_k_loads"] == 0
    assert g.gemm_f16_device_status() == 0


@pytest.mark.parametrize("nb,M,N,K,la,lb", [
    (3, 1000, 512, 448, "row", "row"),    # batch dimension on 4-D / 5-D maps, MN-major B
    (4, 300, 260, 200, "row", "col"),     # ragged K, K-major B
    (2, 768, 768, 1024, "col", "row"),    # MN-major A with a batch dimension (5-D box)
])
def test_batched_two_k_block_copies(nb, M, N, K, la, lb):
    rng = np.random.default_rng(nb * 100 + M + N + K)
    Ah, Bh = ints(rng, (nb, M, K)), ints(rng, (nb, K, N))

    def dev3(x, layout):
        t = torch.from_numpy(np.ascontiguousarray(x))
        return t.to(DEV) if layout == "row" else t.transpose(1, 2).contiguous().to(DEV).transpose(1, 2)

    A, B = dev3(Ah, la), dev3(Bh, lb)
    c2, c1 = run_both(lambda: g.bmm(A, B))
    ref = oracle.gemm_batched(Ah, Bh, threads=oracle_threads())
    for b in range(nb):
        assert_bits(c2[b], ref[b], f"batched two-block copies, problem {b}")
    assert_bits(c2, c1, "one copy per block")
    assert g.gemm_f16_device_status() == 0


@pytest.mark.parametrize("rows,N,K", [([512, 384, 640], 512, 448), ([130, 0, 256, 1, 700], 320, 200)])
def test_grouped_two_k_block_copies(rows, N, K):
    rng = np.random.default_rng(sum(rows) + N + K)
    Ah, Bh = ints(rng, (sum(rows), K)), ints(rng, (len(rows), K, N))
    A, B = torch.from_numpy(Ah).to(DEV), torch.from_numpy(Bh).to(DEV)
    c2, c1 = run_both(lambda: g.grouped_mm(A, B, rows))
    assert_bits(c2, oracle.gemm_grouped(Ah, Bh, rows, threads=oracle_threads()), "grouped two-block copies")
    assert_bits(c2, c1, "one copy per block")
    assert g.gemm_f16_device_status() == 0


# (M, N, K, B layout, options, does the plan take two-block copies?)
GATED = [
    (1000, 512, 448, "row", {}, 1),                 # pair form: rank 0 the gate box, rank 1 the up box
    (600, 384, 200, "col", {}, 1),                  # K-major B and B_up, ragged K
    (1000, 512, 448, "row", {g.OPT_PAIR: 1}, 0),    # single CTA: gate and up boxes interleave in each slot
]


@pytest.mark.parametrize("case", GATED, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-{c[4]}")
def test_gate_up_two_k_block_copies(case):
    M, N, K, lb, opts, expect = case
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    rng = np.random.default_rng(M + 5 * N + 3 * K)
    Ah, Bh, Uh = ints(rng, (M, K)), ints(rng, (K, N)), ints(rng, (K, N))
    bh, buh = ints(rng, (N,)), ints(rng, (N,))
    A, B, U = view(Ah, "row"), view(Bh, lb), view(Uh, lb)
    bias, bias_up = torch.from_numpy(bh).to(DEV), torch.from_numpy(buh).to(DEV)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    plan = g.fused_plan_for(A, B, out, bias=bias, act="relu", b_up=U, bias_up=bias_up)
    assert plan["gated"] == 1 and plan["two_k_loads"] == expect, plan
    c2, c1 = run_both(lambda: g.fused_mm(A, B, bias=bias, act="relu", b_up=U, bias_up=bias_up, out=out))
    # integer sums are exact, relu(g) * u below 2^24 is exact in fp32: one rounding on both sides
    assert_bits(c2, oracle.gemm_fused(Ah, Bh, Uh, bh, buh, "relu", threads=oracle_threads()), f"gate/up {case[:4]}")
    assert_bits(c2, c1, "one copy per block")
    assert g.gemm_f16_device_status() == 0


def test_grouped_gate_up_two_k_block_copies():
    rows, N, K = [512, 384, 640], 256, 448
    rng = np.random.default_rng(77)
    Ah, Bh, Uh = ints(rng, (sum(rows), K)), ints(rng, (len(rows), K, N)), ints(rng, (len(rows), K, N))
    A, B, U = (torch.from_numpy(x).to(DEV) for x in (Ah, Bh, Uh))
    c2, c1 = run_both(lambda: g.grouped_fused_mm(A, B, rows, act="relu", b_up=U))
    ref = oracle.gemm_fused_grouped(Ah, Bh, rows, B_up=Uh, act="relu", threads=oracle_threads())
    assert_bits(c2, ref, "grouped gate/up two-block copies")
    assert_bits(c2, c1, "one copy per block")
    assert g.gemm_f16_device_status() == 0
