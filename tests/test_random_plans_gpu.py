"""Randomised parity sweep: shapes, operand layouts, entry points (plain,
fused, grouped, batched) and planner options drawn together from a fixed seed,
integer inputs in [-2, 2] so every result is exact and compared bit for bit
with the oracle; and real-valued inputs, plain and fused, held to the
tolerance.  Combinations that no hand-written case names are where plan
interactions hide (a grouped call with K = 1 once reached an unaligned TMA box
this way)."""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from tests.parity import assert_close, assert_close_fused, oracle_threads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
OPTIONS = (g.OPT_FORCE_GATHER, g.OPT_SPLITS, g.OPT_TILE_N, g.OPT_PANEL, g.OPT_SWAP, g.OPT_PAIR, g.OPT_STREAMK,
           g.OPT_TAIL_SPLIT, g.OPT_MAX_STAGES, g.OPT_REPACK, g.OPT_PDL,
           g.OPT_L2_A, g.OPT_L2_B, g.OPT_L2_C, g.OPT_TWO_K_LOADS)


def _reset():
    for o in OPTIONS:
        g.gemm_f16_set_option(o, 0)


@pytest.fixture(autouse=True)
def _defaults():
    yield
    _reset()


def _ints(rng, shape):
    return rng.integers(-2, 3, shape).astype(np.float16)


def _view(rng, vals, kind):
    """Device view of `vals` in one of five layouts."""
    r, c = vals.shape
    v = torch.from_numpy(np.ascontiguousarray(vals))
    if kind == 0:
        return v.to(DEV)                                      # row-major
    if kind == 1:
        return v.t().contiguous().to(DEV).t()                # transposed view
    if kind == 2:                                            # pitch not a 16-byte multiple
        buf = torch.zeros((r, c + int(rng.integers(1, 9))), dtype=torch.float16)
        buf[:, :c] = v
        return buf.to(DEV)[:, :c]
    if kind == 3:                                            # base 2 bytes off alignment
        flat = torch.zeros((r * c + 8,), dtype=torch.float16)
        flat[1:1 + r * c] = v.reshape(-1)
        return flat.to(DEV)[1:1 + r * c].view(r, c)
    buf = torch.zeros((2 * r, 2 * c), dtype=torch.float16)   # no unit stride
    buf[::2, ::2] = v
    return buf.to(DEV)[::2, ::2]


def _options(rng):
    draws = ((0.2, g.OPT_FORCE_GATHER, lambda: int(rng.integers(1, 8))),
             (0.15, g.OPT_SPLITS, lambda: int(rng.integers(2, 5))),
             (0.15, g.OPT_TILE_N, lambda: int(rng.choice([64, 128, 192, 256]))),
             (0.2, g.OPT_PANEL, lambda: int(rng.integers(1, 12))),
             (0.15, g.OPT_SWAP, lambda: int(rng.integers(1, 3))),
             (0.2, g.OPT_PAIR, lambda: int(rng.integers(1, 3))),
             (0.2, g.OPT_STREAMK, lambda: int(rng.integers(1, 3))),
             (0.1, g.OPT_TAIL_SPLIT, lambda: 1),
             (0.1, g.OPT_MAX_STAGES, lambda: int(rng.choice([2, 4, 6]))),
             (0.2, g.OPT_REPACK, lambda: int(rng.integers(1, 3))),
             (0.1, g.OPT_PDL, lambda: 1),
             (0.15, g.OPT_L2_A, lambda: int(rng.integers(1, 4))),
             (0.15, g.OPT_L2_B, lambda: int(rng.integers(1, 4))),
             (0.15, g.OPT_L2_C, lambda: int(rng.integers(1, 4))),
             (0.2, g.OPT_TWO_K_LOADS, lambda: 1))
    return {o: f() for p, o, f in draws if rng.random() < p}


def _plain(rng):
    M, N, K = (int(x) for x in rng.integers(1, 700, 3))
    if rng.random() < 0.2:
        K = int(rng.integers(700, 3000))
    if rng.random() < 0.2:
        M, N = (int(x) for x in rng.integers(700, 2000, 2))
    Ah, Bh = _ints(rng, (M, K)), _ints(rng, (K, N))
    A = _view(rng, Ah, int(rng.integers(0, 5)))
    B = _view(rng, Bh, int(rng.integers(0, 5)))
    ref = oracle.gemm(Ah, Bh, threads=oracle_threads())
    ck = int(rng.integers(0, 3))
    if ck == 0:
        return g.matmul(A, B), ref, f"plain {M}x{N}x{K}"
    # C inside a NaN buffer, pitched (ck 1) or 2 bytes off alignment (ck 2): nothing
    # outside the M x N view may change
    ldc = N + int(rng.integers(1, 17)) if ck == 1 else N
    off = 0 if ck == 1 else 1
    buf = torch.full((M * ldc + 8,), float("nan"), dtype=torch.float16, device=DEV)
    C = buf[off:off + M * ldc].view(M, ldc)[:, :N]
    g.matmul(A, B, out=C)
    torch.cuda.synchronize()
    outside = torch.ones(buf.numel(), dtype=torch.bool)
    outside[(off + torch.arange(M)[:, None] * ldc + torch.arange(N)[None, :]).reshape(-1)] = False
    assert torch.isnan(buf.cpu()[outside]).all(), f"plain {M}x{N}x{K}: wrote outside the C view"
    return C, ref, f"plain {M}x{N}x{K}, C layout {ck}, ldc {ldc}"


def _fused(rng):
    M, N, K = (int(x) for x in rng.integers(1, 600, 3))
    gated = rng.random() < 0.5
    act = ("none", "relu")[int(rng.integers(0, 2))]
    Ah, Bh = _ints(rng, (M, K)), _ints(rng, (K, N))
    Uh = _ints(rng, (K, N)) if gated else None
    bh = _ints(rng, N) if rng.random() < 0.7 else None
    buh = _ints(rng, N) if gated and rng.random() < 0.7 else None
    t = lambda x: None if x is None else torch.from_numpy(x).to(DEV)  # noqa: E731
    C = g.fused_mm(t(Ah), t(Bh), bias=t(bh), act=act, b_up=t(Uh), bias_up=t(buh))
    ref = oracle.gemm_fused(Ah, Bh, Uh, bh, buh, act, threads=oracle_threads())
    return C, ref, f"fused {M}x{N}x{K} gated={gated} {act}"


def _grouped(rng):
    G = int(rng.integers(1, 10))
    rows = [int(x) if rng.random() > 0.15 else 0 for x in rng.integers(1, 400, G)]
    if sum(rows) == 0:
        rows[0] = 5
    N, K = (int(x) for x in rng.integers(1, 400, 2))
    Ah, Bh = _ints(rng, (sum(rows), K)), _ints(rng, (G, K, N))
    A = torch.from_numpy(Ah).to(DEV)
    if rng.random() < 0.4:
        A = torch.from_numpy(np.ascontiguousarray(Ah.T)).to(DEV).t()
    C = g.grouped_mm(A, torch.from_numpy(Bh).to(DEV), rows)
    return C, oracle.gemm_grouped(Ah, Bh, rows, threads=oracle_threads()), f"grouped {rows} N={N} K={K}"


def _batched(rng):
    nb = int(rng.integers(1, 6))
    M, N, K = (int(x) for x in rng.integers(1, 400, 3))
    Ah, Bh = _ints(rng, (nb, M, K)), _ints(rng, (nb, K, N))
    C = g.bmm(torch.from_numpy(Ah).to(DEV), torch.from_numpy(Bh).to(DEV))
    return C, oracle.gemm_batched(Ah, Bh, threads=oracle_threads()), f"batched {nb}x{M}x{N}x{K}"


@pytest.mark.parametrize("seed", [101, 102, 103])
def test_random_plans_bit_exact(seed):
    rng = np.random.default_rng(seed)
    makers = (_plain, _plain, _fused, _grouped, _batched)
    for i in range(150):
        _reset()
        opts = _options(rng)
        for o, v in opts.items():
            g.gemm_f16_set_option(o, v)
        C, ref, what = makers[int(rng.integers(0, len(makers)))](rng)
        torch.cuda.synchronize()
        got = C.cpu().numpy()
        assert g.gemm_f16_device_status() == 0, (i, what, opts)
        if not np.array_equal(got.view(np.uint16), ref.view(np.uint16)):
            bad = np.argwhere(got.view(np.uint16) != ref.view(np.uint16))
            raise AssertionError(f"case {i}: {what}, options {opts}: {len(bad)} elements differ, first at "
                                 f"{bad[0].tolist()}")


def _real(rng):
    """Real-valued inputs, uniform [-1, 1] in fp16: every fp32 summation order is
    a correct result, so the plain product is held to the stated tolerance and
    the fused stage (every activation, plain and gated) to its propagated one."""
    M, N, K = (int(x) for x in rng.integers(1, 700, 3))
    if rng.random() < 0.3:
        K = int(rng.integers(700, 4000))
    Ah = rng.uniform(-1, 1, (M, K)).astype(np.float16)
    Bh = rng.uniform(-1, 1, (K, N)).astype(np.float16)
    A = _view(rng, Ah, int(rng.integers(0, 5)))
    B = _view(rng, Bh, int(rng.integers(0, 5)))
    if rng.random() < 0.4:
        C = g.matmul(A, B)
        torch.cuda.synchronize()
        assert_close(C.cpu().numpy(), oracle.gemm(Ah, Bh, threads=oracle_threads()), K, f"real {M}x{N}x{K}")
        return f"real {M}x{N}x{K}"
    act = ("none", "relu", "silu", "gelu")[int(rng.integers(0, 4))]
    gated = rng.random() < 0.5
    Uh = rng.uniform(-1, 1, (K, N)).astype(np.float16) if gated else None
    bh = rng.uniform(-1, 1, N).astype(np.float16) if rng.random() < 0.7 else None
    buh = rng.uniform(-1, 1, N).astype(np.float16) if gated and rng.random() < 0.7 else None
    t = lambda x: None if x is None else torch.from_numpy(x).to(DEV)  # noqa: E731
    U = None
    if gated:   # the up projection with B's strides
        U = torch.empty_strided(B.shape, B.stride(), dtype=torch.float16, device=DEV)
        U.copy_(torch.from_numpy(Uh))
    C = g.fused_mm(A, B, bias=t(bh), act=act, b_up=U, bias_up=t(buh))
    torch.cuda.synchronize()
    ref, gp, u = oracle.gemm_fused(Ah, Bh, Uh, bh, buh, act, threads=oracle_threads(), parts=True)
    what = f"real fused {M}x{N}x{K} gated={gated} {act}"
    assert_close_fused(C.cpu().numpy(), ref, K, gp, u, act, what)
    return what


@pytest.mark.parametrize("seed", [201, 202])
def test_random_plans_real_valued_within_tolerance(seed):
    rng = np.random.default_rng(seed)
    for i in range(60):
        _reset()
        opts = _options(rng)
        for o, v in opts.items():
            g.gemm_f16_set_option(o, v)
        what = _real(rng)
        assert g.gemm_f16_device_status() == 0, (i, what, opts)
