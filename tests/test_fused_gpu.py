"""Parity of the fused output stage with the CPU oracle.

Bias and activation in the output stage (TileLang tutorial ch. 14, section 6.3,
item 4; AI-infra page, section 05) and the gate/up product of two projections
sharing A (C500 review, section 17.3).  Integer inputs with the identity or
ReLU make every intermediate exact, so those cases compare bit for bit; SiLU
and GELU go through fp32 exp / erfc and are held to the propagated tolerance
of ``assert_close_fused``.
"""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from tests.parity import assert_bits, assert_close_fused, oracle_threads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for o in (g.OPT_FORCE_GATHER, g.OPT_SPLITS, g.OPT_TILE_N, g.OPT_PANEL, g.OPT_SWAP,
              g.OPT_TIMEOUT_MS, g.OPT_MAX_CTAS, g.OPT_PAIR, g.OPT_STREAMK, g.OPT_TAIL_SPLIT, g.OPT_MAX_STAGES,
              g.OPT_REPACK):
        g.gemm_f16_set_option(o, 0)


def values(rng, shape, integer):
    if integer:
        return rng.integers(-3, 4, shape).astype(np.float16)
    return rng.uniform(-1, 1, shape).astype(np.float16)


def operand(rng, rows, cols, integer, transposed=False):
    """(host view, device view) of a rows x cols operand; transposed: the view of
    a row-major cols x rows buffer (strides (1, rows))."""
    buf = values(rng, (cols, rows) if transposed else (rows, cols), integer)
    d = torch.from_numpy(buf).to(DEV)
    return (buf.T, d.t()) if transposed else (buf, d)


def check(got, ref, g_pre, u, act, K, exact, what):
    if exact:
        assert_bits(got, ref, what)
    else:
        assert_close_fused(got, ref, K, g_pre, u, act, what)


# ------------------------------------------------------------- one problem
PLAIN = [
    # (M, N, K, act, bias, integer, options, B transposed, expected plan)
    (300, 260, 200, "relu", True, True, {}, False, {"pair": 0}),
    (1000, 512, 128, "none", True, True, {}, False, {"pair": 1}),
    (700, 384, 256, "silu", True, False, {}, False, {}),
    (520, 640, 320, "gelu", False, False, {}, True, {}),
    (16, 1024, 512, "silu", True, False, {}, False, {"swap_ab": 1}),        # bias along the kernel rows
    (130, 70, 65, "relu", True, True, {}, False, {"b_tma": 0}),             # gathered operands, masked C
    (600, 256, 1024, "gelu", True, False, {g.OPT_SPLITS: 3}, False, {"splits": 3}),
    (900, 384, 640, "relu", True, True, {g.OPT_STREAMK: 2}, False, {}),
    (16, 1024, 2048, "gelu", True, False, {g.OPT_SPLITS: 4}, False, {"swap_ab": 1, "splits": 4}),
]


@pytest.mark.parametrize("case", PLAIN, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-bias{int(c[4])}-{len(c[6])}")
def test_bias_activation_matches_oracle(case):
    M, N, K, act, with_bias, integer, opts, bt, plan = case
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    Ah, A = operand(rng, M, K, integer)
    Bh, B = operand(rng, K, N, integer, bt)
    bh = values(rng, N, integer) if with_bias else None
    bias = torch.from_numpy(bh).to(DEV) if with_bias else None
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    p = g.fused_plan_for(A, B, C, bias=bias, act=act)
    assert p["fused"] == 1 and p["gated"] == 0
    for k, v in plan.items():
        assert p[k] == v, (k, p)
    if "splits" not in plan and g.OPT_STREAMK in opts:
        assert p["streamk_tiles"] > 0
    g.fused_mm(A, B, bias=bias, act=act, out=C)
    torch.cuda.synchronize()
    ref, gp, _ = oracle.gemm_fused(Ah, Bh, bias=bh, act=act, threads=oracle_threads(), parts=True)
    check(C.cpu().numpy(), ref, gp, None, act, K, integer and act in ("none", "relu"), f"fused {case}")
    assert g.gemm_f16_device_status() == 0


GATED = [
    # (M, N, K, act, biases, integer, options, B transposed, expected plan)
    (300, 264, 200, "relu", True, True, {g.OPT_PAIR: 1}, False, {"pair": 0, "tile_n": 128}),
    (1000, 512, 128, "silu", True, False, {}, False, {"pair": 1, "tile_n": 128}),
    (600, 64, 192, "gelu", False, False, {}, False, {"tile_n": 64}),
    (520, 200, 320, "relu", True, True, {}, True, {}),
    (16, 512, 256, "silu", True, False, {}, False, {"swap_ab": 0, "splits": 1}),
    (130, 70, 65, "relu", True, True, {}, False, {"b_tma": 0}),
    (400, 256, 128, "gelu", True, False, {g.OPT_FORCE_GATHER: 3}, False, {"a_tma": 0, "b_tma": 0}),
    (384, 384, 256, "silu", False, False, {g.OPT_FORCE_GATHER: 3}, True, {"a_tma": 0, "b_tma": 0}),
    (700, 300, 512, "none", True, True, {g.OPT_SPLITS: 3, g.OPT_STREAMK: 2}, False, {"splits": 1}),
]


@pytest.mark.parametrize("case", GATED, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-bias{int(c[4])}-{len(c[6])}")
def test_gate_up_matches_oracle(case):
    M, N, K, act, with_bias, integer, opts, bt, plan = case
    rng = np.random.default_rng(M * 5 + N * 11 + K)
    Ah, A = operand(rng, M, K, integer)
    Bh, B = operand(rng, K, N, integer, bt)
    Uh, U = operand(rng, K, N, integer, bt)
    bh = values(rng, N, integer) if with_bias else None
    buh = values(rng, N, integer) if with_bias else None
    bias = torch.from_numpy(bh).to(DEV) if with_bias else None
    bias_up = torch.from_numpy(buh).to(DEV) if with_bias else None
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    p = g.fused_plan_for(A, B, C, bias=bias, act=act, b_up=U, bias_up=bias_up)
    assert p["fused"] == 1 and p["gated"] == 1 and p["streamk_tiles"] == 0 and p["tail_split"] == 1
    for k, v in plan.items():
        assert p[k] == v, (k, p)
    g.fused_mm(A, B, bias=bias, act=act, b_up=U, bias_up=bias_up, out=C)
    torch.cuda.synchronize()
    ref, gp, u = oracle.gemm_fused(Ah, Bh, Uh, bh, buh, act, threads=oracle_threads(), parts=True)
    check(C.cpu().numpy(), ref, gp, u, act, K, integer and act in ("none", "relu"), f"gated {case}")
    assert g.gemm_f16_device_status() == 0


def test_gated_writes_only_the_view():
    # C inside a NaN-filled pitch-padded buffer: padding columns and the rows
    # after it stay NaN; N not a multiple of the 128-column output tile
    rng = np.random.default_rng(61)
    M, N, K, ldc = 333, 200, 96, 216
    Ah, A = operand(rng, M, K, True)
    Bh, B = operand(rng, K, N, True)
    Uh, U = operand(rng, K, N, True)
    buf = torch.full((M + 3, ldc), float("nan"), dtype=torch.float16, device=DEV)
    C = buf[:M, :N]
    g.fused_mm(A, B, act="relu", b_up=U, out=C)
    torch.cuda.synchronize()
    assert_bits(C.cpu().numpy(), oracle.gemm_fused(Ah, Bh, Uh, act="relu"), "gated in padded C")
    host = buf.cpu()
    assert torch.isnan(host[:M, N:]).all() and torch.isnan(host[M:]).all()


# ---------------------------------------------------------- several problems
def test_batched_fused_matches_oracle():
    rng = np.random.default_rng(62)
    for nb, M, N, K, act, gated, integer, shared_bias in (
            (4, 300, 264, 200, "relu", True, True, False),
            (3, 16, 512, 256, "silu", False, False, True),     # swapped per problem, one bias for all
            (5, 130, 70, 65, "gelu", False, False, False),
            (2, 520, 384, 512, "gelu", True, False, True)):
        Ah, Bh = values(rng, (nb, M, K), integer), values(rng, (nb, K, N), integer)
        Uh = values(rng, (nb, K, N), integer) if gated else None
        bh = values(rng, N if shared_bias else (nb, N), integer)
        buh = values(rng, N if shared_bias else (nb, N), integer) if gated else None
        dev = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(DEV)  # noqa: E731
        C = g.fused_mm(dev(Ah), dev(Bh), bias=dev(bh), act=act, b_up=dev(Uh), bias_up=dev(buh))
        torch.cuda.synchronize()
        ref, gp, u = oracle.gemm_fused_batched(Ah, Bh, Uh, bh, buh, act, threads=oracle_threads(), parts=True)
        got = C.cpu().numpy()
        for b in range(nb):
            check(got[b], ref[b], gp[b], None if u is None else u[b], act, K, integer and act == "relu",
                  f"batched fused b{nb} {M}x{N}x{K} {act} gated={gated} problem {b}")
    assert g.gemm_f16_device_status() == 0


GROUPED = [
    # (group rows, N, K, act, gated, integer, options)
    ([130, 0, 256, 1, 700], 320, 200, "silu", True, False, {}),
    ([512, 384, 640], 512, 136, "relu", True, True, {}),
    ([37] * 9, 128, 72, "gelu", True, False, {g.OPT_PAIR: 1}),
    ([300, 900, 77], 256, 640, "gelu", False, False, {g.OPT_STREAMK: 2}),
    ([1000, 3000, 50], 1024, 512, "silu", True, False, {}),
]


@pytest.mark.parametrize("case", GROUPED, ids=lambda c: f"g{len(c[0])}-{sum(c[0])}x{c[1]}x{c[2]}-{c[3]}-{int(c[4])}")
def test_grouped_fused_matches_oracle(case):
    rows, N, K, act, gated, integer, opts = case
    rng = np.random.default_rng(sum(rows) + N + K + 7)
    G = len(rows)
    Ah, Bh = values(rng, (sum(rows), K), integer), values(rng, (G, K, N), integer)
    Uh = values(rng, (G, K, N), integer) if gated else None
    bh = values(rng, (G, N), integer)
    buh = values(rng, (G, N), integer) if gated else None
    dev = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(DEV)  # noqa: E731
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    Cbuf = torch.full((sum(rows) + 5, N), float("nan"), dtype=torch.float16, device=DEV)
    g.grouped_fused_mm(dev(Ah), dev(Bh), rows, bias=dev(bh), act=act, b_up=dev(Uh), bias_up=dev(buh),
                       out=Cbuf[:sum(rows)])
    torch.cuda.synchronize()
    ref, gp, u = oracle.gemm_fused_grouped(Ah, Bh, rows, Uh, bh, buh, act, threads=oracle_threads(), parts=True)
    got = Cbuf.cpu().numpy()
    check(got[:sum(rows)], ref, gp, u, act, K, integer and act == "relu", f"grouped fused {case}")
    assert np.isnan(got[sum(rows):]).all()
    assert g.gemm_f16_device_status() == 0


# ----------------------------------------------------------------- errors
def test_fused_argument_errors():
    A = torch.zeros((64, 64), dtype=torch.float16, device=DEV)
    B = torch.zeros((64, 64), dtype=torch.float16, device=DEV)
    C = torch.zeros((64, 64), dtype=torch.float16, device=DEV)
    bias = torch.zeros(64, dtype=torch.float16, device=DEV)
    base = (A.data_ptr(), 64, 1, B.data_ptr(), 64, 1)
    with pytest.raises(g.GemmF16Error) as e:   # bias_up without a second projection
        g.gemm_f16_fused(*base, 0, 0, bias.data_ptr(), 0, C.data_ptr(), 64, 64, 64, 64)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemmF16Error) as e:   # unknown activation
        g.gemm_f16_fused(*base, 0, bias.data_ptr(), 0, 9, C.data_ptr(), 64, 64, 64, 64)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemmF16Error) as e:   # C overlaps the bias
        g.gemm_f16_fused(*base, 0, C.data_ptr() + 64, 0, 1, C.data_ptr(), 64, 64, 64, 64)
    assert e.value.status == g.ERR_ALIAS
    with pytest.raises(g.GemmF16Error) as e:   # C overlaps the up projection
        g.gemm_f16_fused(*base, C.data_ptr(), 0, 0, 1, C.data_ptr(), 64, 64, 64, 64)
    assert e.value.status == g.ERR_ALIAS
    with pytest.raises(ValueError):
        g.fused_mm(A, B, act="tanh")
    torch.cuda.synchronize()
