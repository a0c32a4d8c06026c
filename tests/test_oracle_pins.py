"""Pins for the CPU oracle: what the pages and the mathematics fix, not the oracle itself.

Each test names the passage or the property it pins.  Planted mistakes (wrong
strides, modulo K) are planted in the oracle's inputs or in the tiled
restatement, on the CPU.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import tiled
from synth import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def h(x):
    return np.asarray(x, dtype=np.float16)


# ---------------------------------------------------------------- fp16 codec
def test_decode_every_code_matches_numpy():
    codes = np.arange(65536, dtype=np.uint16)
    ours = oracle.half_to_double(codes)
    ref = codes.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # the sign of zero survives
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_encode_matches_numpy_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.uniform(-1, 1, 200000),
        rng.standard_normal(200000) * 1000,
        np.ldexp(rng.uniform(0.5, 1, 100000), rng.integers(-30, 17, 100000))
        * rng.choice([-1, 1], 100000),
    ])
    # exact midpoints between neighbouring fp16 values, to exercise ties-to-even
    codes = rng.integers(0, 0x7bff, 50000).astype(np.uint16)
    lo = codes.view(np.float16).astype(np.float64)
    hi = (codes + 1).view(np.float16).astype(np.float64)
    x = np.concatenate([x, (lo + hi) / 2, -(lo + hi) / 2])
    edges = np.array([0.0, -0.0, 65504.0, 65519.999, 65520.0, 70000.0, -65520.0,
                      2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001,
                      3 * 2.0 ** -25, 2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11,
                      1.0 + 3 * 2.0 ** -11, np.inf, -np.inf])
    x = np.concatenate([x, edges])
    ours = oracle.double_to_half(x).view(np.uint16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.isnan(oracle.double_to_half([np.nan]).astype(np.float64))[0]


# ---------------------------------------------------------- worked examples
def test_transposed_view_example():
    g = golden("transposed_view.json")
    X = h(g["X_rowmajor"]).reshape(-1)
    # A = I3 picks out the rows of B, so C[1,0] = B[1,0]
    I3 = h(np.eye(3)).reshape(-1)
    sbk, sbn = g["B_strides"]
    C = oracle.gemm_strided(I3, 0, 3, 1, X, 0, sbk, sbn, 3, 2, 3).view(np.float16)
    assert C.reshape(3, 2)[1, 0] == g["B_1_0"]
    assert np.array_equal(C.reshape(3, 2).astype(np.float64),
                          np.array(g["X_rowmajor"], dtype=np.float64).T)
    # planted mistake: assuming contiguous strides reads the wrong element
    s0, s1 = g["contiguous_strides"]
    Cw = oracle.gemm_strided(I3, 0, 3, 1, X, 0, s0, s1, 3, 2, 3).view(np.float16)
    assert Cw.reshape(3, 2)[1, 0] == g["contiguous_B_1_0"]


def test_k_tail_zero_fill_not_modulo():
    g = golden("k_tail.json")
    a = h(g["a"]).reshape(1, 3)
    b = h(g["b"]).reshape(3, 1)
    assert oracle.gemm(a, b)[0, 0] == g["correct"]
    C, _ = tiled.tiled_gemm(a, b, 1, 1, g["block_k"])
    assert C[0, 0] == g["correct"]
    Cw, _ = tiled.tiled_gemm(a, b, 1, 1, g["block_k"], k_wrap_modulo=True)
    assert Cw[0, 0] == g["modulo_wrapped"]
    assert [k % 3 for k in (2, 3)] == g["wrapped_indices_of_second_block"]


def test_read_counts_4x4():
    g = golden("read_counts_4x4.json")
    rng = np.random.default_rng(1)
    A = rng.integers(-3, 4, (4, 4))
    B = rng.integers(-3, 4, (4, 4))
    for key in ("untiled", "tile_2x2", "whole"):
        t = g[key]
        C, st = tiled.tiled_gemm(A, B, t["BM"], t["BN"], t["BK"])
        assert st.logical_reads == t["reads"], key
        assert int(st.writes.sum()) == g["output_writes"]
        assert np.array_equal(C, A @ B)
        # the closed form M*N*K*(1/BM + 1/BN) for divisible shapes
        assert st.logical_reads == 4 * 4 * 4 * (1 / t["BM"] + 1 / t["BN"])


def test_tail_130x70x65_program_model():
    g = golden("tail_130x70x65.json")
    M, N, K, BM, BN, BK = (g[k] for k in ("M", "N", "K", "BM", "BN", "BK"))
    w = workloads.TAIL_ROWMAJOR_B
    A = w.A.host_view()
    B = w.B.host_view()
    C, st = tiled.tiled_gemm(A, B, BM, BN, BK)
    assert st.programs == g["programs"] == g["grid"][0] * g["grid"][1]
    assert st.rounds_per_program == g["rounds"]
    assert tiled.corner_valid(M, N, BM, BN) == (g["corner_valid_rows"], g["corner_valid_cols"])
    assert g["corner_valid_rows"] * g["corner_valid_cols"] == g["corner_valid_outputs"]
    assert tiled.last_round_valid_k(K, BK) == g["last_round_valid_k"]
    useful = 2 * M * N * K
    assert useful / st.block_flops == pytest.approx(g["useful_fraction_approx"], abs=5e-4)
    # single writer: every valid output written exactly once
    assert st.writes.min() == 1 and st.writes.max() == 1
    # the tiled restatement equals the plain oracle bit for bit on exact inputs
    Co = oracle.gemm(A, B)
    assert np.array_equal(C.astype(np.float16).view(np.uint16), Co.view(np.uint16))


def test_int64_offset_example():
    g = golden("int64_offset.json")
    assert g["row"] * g["stride"] == g["offset"] == 2 ** 32
    assert (g["row"] * g["stride"]) & 0xFFFFFFFF == g["offset_wrapped_32bit"]
    # The oracle indexes with int64: A row 65536 with row stride 65536 lives at
    # element 2^32.  The buffer is zero-filled virtual memory; only touched pages
    # are backed.  A wrapped offset would read row 0's value instead.
    n = g["offset"] + 1
    try:
        buf = np.zeros(n, dtype=np.uint16)
    except MemoryError:
        pytest.skip("cannot reserve 8 GiB of virtual memory")
    buf[0] = np.float16(2.0).view(np.uint16)
    buf[g["offset"]] = np.float16(1.0).view(np.uint16)
    Bm = h([3.0])
    M = g["row"] + 1
    C = oracle.gemm_strided(buf, 0, g["stride"], 1, Bm, 0, 1, 1, M, 1, 1).view(np.float16)
    assert C[0] == 6.0
    assert C[g["row"]] == 3.0
    assert C[1:g["row"]].max() == 0.0


# ------------------------------------------------------------ brute force
def _exact_int_product(Ai, Bi):
    M, K = Ai.shape
    N = Bi.shape[1]
    out = [[sum(int(Ai[m, k]) * int(Bi[k, n]) for k in range(K)) for n in range(N)]
           for m in range(M)]
    return np.array(out, dtype=np.int64)


def _random_view(rng, rows, cols, values):
    """A rows x cols fp16 view with random layout: row-major, transposed or pitched."""
    layout = rng.integers(0, 3)
    if layout == 0:
        pitch = cols + int(rng.integers(0, 5))
        buf = np.zeros((rows, pitch), dtype=np.float16)
        buf[:, :cols] = values
        return buf[:, :cols]
    if layout == 1:
        pitch = rows + int(rng.integers(0, 5))
        buf = np.zeros((cols, pitch), dtype=np.float16)
        buf[:, :rows] = values.T
        return buf[:, :rows].T
    # both strides > 1
    buf = np.zeros((rows * 2, cols * 3), dtype=np.float16)
    buf[::2, ::3] = values
    return buf[::2, ::3]


def test_bruteforce_integer_inputs_exact():
    rng = np.random.default_rng(2)
    for _ in range(60):
        M, N, K = (int(x) for x in rng.integers(1, 40, 3))
        Ai = rng.integers(-3, 4, (M, K))
        Bi = rng.integers(-3, 4, (K, N))
        A = _random_view(rng, M, K, Ai.astype(np.float16))
        B = _random_view(rng, K, N, Bi.astype(np.float16))
        C = oracle.gemm(A, B)
        assert np.array_equal(C.astype(np.int64), _exact_int_product(Ai, Bi))


def test_random_real_inputs_match_numpy_double_then_round():
    # a library routine (numpy float64 matmul, then numpy's correctly rounded
    # double -> half) on the same fp16 inputs
    rng = np.random.default_rng(3)
    for _ in range(30):
        M, N, K = (int(x) for x in rng.integers(1, 120, 3))
        A = rng.uniform(-1, 1, (M, K)).astype(np.float16)
        B = rng.uniform(-1, 1, (K, N)).astype(np.float16)
        ref = (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float16)
        Av = _random_view(rng, M, K, A)
        Bv = _random_view(rng, K, N, B)
        assert np.array_equal(oracle.gemm(Av, Bv).view(np.uint16), ref.view(np.uint16))


def test_closed_forms_permutation_diagonal_identity():
    rng = np.random.default_rng(4)
    n, N = 37, 23
    B = rng.uniform(-4, 4, (n, N)).astype(np.float16)
    perm = rng.permutation(n)
    P = np.zeros((n, n), dtype=np.float16)
    P[np.arange(n), perm] = 1
    assert np.array_equal(oracle.gemm(P, B), B[perm])
    d = rng.choice([-2.0, -1.0, 0.5, 1.0, 2.0], n)
    D = np.diag(d).astype(np.float16)
    assert np.array_equal(oracle.gemm(D, B), (d[:, None] * B.astype(np.float64)).astype(np.float16))
    I = np.eye(N, dtype=np.float16)
    assert np.array_equal(oracle.gemm(B, I), B)
    # (A B)^T = B^T A^T with transposed views
    A = rng.integers(-3, 4, (11, n)).astype(np.float16)
    assert np.array_equal(oracle.gemm(A, B).T, oracle.gemm(B.T, A.T))


def test_overflow_and_nan():
    a = h([[256.0, 256.0]])
    b = h([[256.0], [256.0]])
    assert np.isposinf(oracle.gemm(a, b)[0, 0])
    assert oracle.gemm(h([[255.875]]), h([[256.0]]))[0, 0] == 65504.0  # 65504 exact
    assert np.isnan(oracle.gemm(h([[np.nan, 1.0]]), h([[1.0], [1.0]]))[0, 0])


def test_sampled_dots_equal_full_oracle():
    rng = np.random.default_rng(5)
    M, N, K = 57, 41, 93
    A = rng.uniform(-1, 1, (M, K)).astype(np.float16)
    Bt = rng.uniform(-1, 1, (N, K)).astype(np.float16)
    B = Bt.T  # column-major B: columns contiguous
    full = oracle.gemm(A, B)
    ms = rng.integers(0, M, 200)
    ns = rng.integers(0, N, 200)
    vals, exact = oracle.dots(A.reshape(-1), ms * K, 1, Bt.reshape(-1), ns * K, 1, K)
    assert np.array_equal(vals.view(np.uint16), full[ms, ns].view(np.uint16))
    ref = np.einsum("ik,ik->i", A[ms].astype(np.float64), Bt[ns].astype(np.float64))
    assert np.allclose(exact, ref, rtol=0, atol=1e-12)


def test_openmp_rows_do_not_change_results():
    rng = np.random.default_rng(6)
    A = rng.uniform(-1, 1, (64, 300)).astype(np.float16)
    B = rng.uniform(-1, 1, (300, 50)).astype(np.float16)
    assert np.array_equal(oracle.gemm(A, B, threads=1).view(np.uint16),
                          oracle.gemm(A, B, threads=4).view(np.uint16))


# ------------------------------------------------- batched and grouped GEMM
# TileLang tutorial ch. 14 "GEMM operators", sections 4.3 (grouped) and 4.4
# (batched).  Pinned against numpy's float64 einsum (a library routine) then
# numpy's rounding, per problem, and against closed forms that a wrong batch
# index or group offset would break.
def _ref_batched(A, B):
    return np.einsum("bmk,bkn->bmn", A.astype(np.float64), B.astype(np.float64)).astype(np.float16)


def test_batched_matches_einsum_per_problem():
    rng = np.random.default_rng(21)
    for _ in range(8):
        nb, M, N, K = (int(x) for x in rng.integers(1, 24, 4))
        A = rng.uniform(-1, 1, (nb, M, K)).astype(np.float16)
        B = rng.uniform(-1, 1, (nb, K, N)).astype(np.float16)
        C = oracle.gemm_batched(A, B)
        assert np.array_equal(C.view(np.uint16), _ref_batched(A, B).view(np.uint16))
    # a B shared by every problem (batch stride 0) and transposed A views
    A = rng.uniform(-1, 1, (5, 9, 13)).astype(np.float16)
    B1 = rng.uniform(-1, 1, (13, 7)).astype(np.float16)
    Bs = np.broadcast_to(B1, (5, 13, 7))
    At = np.ascontiguousarray(A.transpose(0, 2, 1)).transpose(0, 2, 1)
    C = oracle.gemm_batched(At, Bs)
    assert np.array_equal(C.view(np.uint16), _ref_batched(A, np.broadcast_to(B1, (5, 13, 7))).view(np.uint16))


def test_batched_problems_are_independent():
    # permuting the batch permutes the results: a wrong batch index (reading
    # problem b+1's B, say) fails this
    rng = np.random.default_rng(22)
    A = rng.integers(-3, 4, (6, 11, 17)).astype(np.float16)
    B = rng.integers(-3, 4, (6, 17, 5)).astype(np.float16)
    perm = rng.permutation(6)
    C = oracle.gemm_batched(A, B)
    assert np.array_equal(oracle.gemm_batched(A[perm], B[perm]), C[perm])
    for b in range(6):
        assert np.array_equal(C[b].astype(np.int64), _exact_int_product(A[b].astype(np.int64), B[b].astype(np.int64)))


def test_grouped_matches_per_group_products():
    rng = np.random.default_rng(23)
    rows = [0, 7, 1, 0, 13, 4]
    G, N, K = len(rows), 9, 15
    A = rng.uniform(-1, 1, (sum(rows), K)).astype(np.float16)
    B = rng.uniform(-1, 1, (G, K, N)).astype(np.float16)
    C = oracle.gemm_grouped(A, B, rows)
    r0 = 0
    for g, r in enumerate(rows):
        ref = (A[r0:r0 + r].astype(np.float64) @ B[g].astype(np.float64)).astype(np.float16)
        assert np.array_equal(C[r0:r0 + r].view(np.uint16), ref.view(np.uint16))
        r0 += r


def test_grouped_closed_forms():
    rng = np.random.default_rng(24)
    A = rng.integers(-3, 4, (20, 8)).astype(np.float16)
    B = rng.integers(-3, 4, (8, 6)).astype(np.float16)
    # one group is the plain product; every group sharing one B is too
    assert np.array_equal(oracle.gemm_grouped(A, B[None], [20]), oracle.gemm(A, B))
    assert np.array_equal(oracle.gemm_grouped(A, np.stack([B] * 4), [3, 0, 12, 5]), oracle.gemm(A, B))
    # group g scaled by g+1 shows which rows each group owns (an off-by-one
    # group offset fails this)
    rows = [3, 0, 12, 5]
    Bg = np.stack([B * (g + 1) for g in range(4)]).astype(np.float16)
    C = oracle.gemm_grouped(A, Bg, rows).astype(np.int64)
    base = oracle.gemm(A, B).astype(np.int64)
    scale = np.repeat(np.arange(1, 5), rows)[:, None]
    assert np.array_equal(C, base * scale)


# ------------------------------------------------------------- fused epilogue
# Bias + activation in the output stage and the gate/up product (TileLang
# tutorial ch. 14, section 6.3, item 4; AI-infra page, section 05; C500 review,
# section 17.3).  Pinned to textbook function values, library routines other
# than the ones the oracle calls, exact identities and a hand-worked example.
def test_exact_sums_round_to_the_plain_oracle():
    rng = np.random.default_rng(50)
    A, B = h(rng.uniform(-1, 1, (37, 150))), h(rng.uniform(-1, 1, (150, 29)))
    S = oracle.gemm_exact(A, B)
    assert np.array_equal(oracle.double_to_half(S).view(np.uint16), oracle.gemm(A, B).view(np.uint16))
    # integer inputs: the sums are the exact integer products
    Ai, Bi = rng.integers(-3, 4, (20, 31)), rng.integers(-3, 4, (31, 17))
    assert np.array_equal(oracle.gemm_exact(h(Ai), h(Bi)), (Ai @ Bi).astype(np.float64))


@pytest.mark.parametrize("act,table,form", [("gelu", "phi", "x*F"), ("silu", "sigma", "x*F")])
def test_activations_at_textbook_points(act, table, form):
    d = golden("fused_epilogue.json")
    for xs, F in d[table].items():
        x = float(xs)
        assert abs(oracle.activation(x, act) - x * F) <= 1e-15 * max(1.0, abs(x)), (act, x)
    assert oracle.activation(0.0, act) == 0.0


def test_activations_match_independent_library_routines():
    special = pytest.importorskip("scipy.special")
    x = np.concatenate([np.linspace(-30, 30, 4001), [-1e-6, 1e-6, 0.0]])
    silu = oracle.activation(x, "silu")
    assert np.allclose(silu, x * special.expit(x), rtol=1e-13, atol=1e-300)
    gelu = oracle.activation(x, "gelu")
    assert np.allclose(gelu, x * special.ndtr(x), rtol=1e-12, atol=1e-290)
    assert np.array_equal(oracle.activation(x, "relu"), np.maximum(x, 0.0))
    assert np.array_equal(oracle.activation(x, "none"), x)


@pytest.mark.parametrize("act", ["relu", "silu", "gelu"])
def test_activation_odd_part_is_identity(act):
    # relu, silu and gelu all satisfy f(x) - f(-x) = x (sigma(x) + sigma(-x) = 1,
    # Phi(x) + Phi(-x) = 1): a wrong sign or a dropped factor breaks it
    x = np.linspace(-12, 12, 2401)
    d = oracle.activation(x, act) - oracle.activation(-x, act)
    assert np.allclose(d, x, rtol=0, atol=1e-13 * 12)


def test_fused_without_epilogue_is_the_plain_gemm():
    rng = np.random.default_rng(51)
    A, B = h(rng.uniform(-1, 1, (45, 300))), h(rng.uniform(-1, 1, (300, 70)))
    assert np.array_equal(oracle.gemm_fused(A, B).view(np.uint16), oracle.gemm(A, B).view(np.uint16))


def test_bias_runs_along_columns():
    # A = I: C = act(B + bias[None, :]) elementwise; a bias indexed by row
    # (or added twice) gives other values since M != N and the entries differ
    rng = np.random.default_rng(52)
    B = rng.integers(-4, 5, (3, 5))
    bias = np.array([1, -2, 3, 0, -1])
    C = oracle.gemm_fused(h(np.eye(3)), h(B), bias=h(bias))
    assert np.array_equal(C.astype(np.int64), B + bias[None, :])
    C = oracle.gemm_fused(h(np.eye(3)), h(B), bias=h(bias), act="relu")
    assert np.array_equal(C.astype(np.int64), np.where(B + bias < 0, 0, B + bias))


def test_gated_hand_worked_example():
    d = golden("fused_epilogue.json")
    C, g, u = oracle.gemm_fused(h(d["A"]), h(d["B_gate"]), h(d["B_up"]), h(d["bias_gate"]), h(d["bias_up"]),
                                act="relu", parts=True)
    assert np.array_equal(g, np.array(d["gate_pre"], dtype=np.float64))
    assert np.array_equal(u, np.array(d["up"], dtype=np.float64))
    assert np.array_equal(C.astype(np.float64), np.array(d["out_relu"], dtype=np.float64))


@pytest.mark.parametrize("act", ["none", "relu", "silu", "gelu"])
def test_gate_by_constant_up_scales_the_plain_form(act):
    # B_up = 0 and bias_up = 1: the product is the non-gated result, bit for bit;
    # bias_up = 2 doubles it exactly (a power of two, far from overflow)
    rng = np.random.default_rng(53)
    A, B = h(rng.uniform(-1, 1, (30, 64))), h(rng.uniform(-1, 1, (64, 40)))
    bias = h(rng.uniform(-1, 1, 40))
    plain = oracle.gemm_fused(A, B, bias=bias, act=act)
    zero = np.zeros_like(B)
    one = oracle.gemm_fused(A, B, zero, bias, h(np.ones(40)), act=act)
    two = oracle.gemm_fused(A, B, zero, bias, h(np.full(40, 2.0)), act=act)
    assert np.array_equal(one.view(np.uint16), plain.view(np.uint16))
    # exact where the doubled value stays normal; a subnormal result is rounded
    # on a fixed grid of 2^-24, so there it may differ by one step
    p64, t64 = plain.astype(np.float64), two.astype(np.float64)
    normal = np.abs(p64) >= 2.0 ** -14
    assert np.array_equal(t64[normal], 2 * p64[normal])
    assert np.all(np.abs(t64[~normal] - 2 * p64[~normal]) <= 2.0 ** -24)


def test_fused_grouped_and_batched_compose_per_problem():
    rng = np.random.default_rng(54)
    rows = [7, 0, 12, 1]
    A = h(rng.uniform(-1, 1, (sum(rows), 24)))
    B, Bu = h(rng.uniform(-1, 1, (4, 24, 16))), h(rng.uniform(-1, 1, (4, 24, 16)))
    bias = h(rng.uniform(-1, 1, (4, 16)))
    C = oracle.gemm_fused_grouped(A, B, rows, Bu, bias, None, "silu")
    r0 = 0
    for g, r in enumerate(rows):
        ref = oracle.gemm_fused(A[r0:r0 + r], B[g], Bu[g], bias[g], None, "silu")
        assert np.array_equal(C[r0:r0 + r].view(np.uint16), ref.view(np.uint16))
        r0 += r
    A3 = h(rng.uniform(-1, 1, (3, 9, 24)))
    C3 = oracle.gemm_fused_batched(A3, B[:3], None, bias[0], None, "gelu")
    for b in range(3):
        ref = oracle.gemm_fused(A3[b], B[b], bias=bias[0], act="gelu")
        assert np.array_equal(C3[b].view(np.uint16), ref.view(np.uint16))
