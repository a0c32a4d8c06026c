"""Parity of the sm_103a GEMM with the CPU oracle, through the C ABI.

Every case runs the library on cuda:0 and compares with the oracle on the same
seeded fp16 inputs: bit for bit where the inputs are integers (every fp32 sum is
exact), within the stated tolerance otherwise.  The five configurations are
covered at full size (whole outputs where the host can afford the oracle,
4096 seeded samples plus a whole boundary tile where it cannot).
"""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
import synth
from synth import workloads
from tests.parity import assert_bits, assert_close, block_reference, oracle_threads, sampled_reference

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for o in (g.OPT_FORCE_GATHER, g.OPT_SPLITS, g.OPT_TILE_N, g.OPT_PANEL, g.OPT_SWAP,
              g.OPT_TIMEOUT_MS, g.OPT_MAX_CTAS, g.OPT_PAIR, g.OPT_STREAMK, g.OPT_TAIL_SPLIT, g.OPT_MAX_STAGES, g.OPT_REPACK,
              g.OPT_L2_A, g.OPT_L2_B, g.OPT_L2_C):
        g.gemm_f16_set_option(o, 0)


def to_dev(x: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def gpu(A, B, out=None):
    C = g.matmul(A, B, out=out)
    torch.cuda.synchronize()
    return C


def host(t):
    return t.cpu().numpy()


# ----------------------------------------------------------------- layouts
def make_view(values: np.ndarray, layout: str):
    """A device fp16 view holding `values` [r, c] in the requested layout."""
    r, c = values.shape
    v = torch.from_numpy(np.ascontiguousarray(values))
    if layout == "row":
        return v.to(DEV)
    if layout == "col":                      # transposed view of a row-major [c, r]
        return v.t().contiguous().to(DEV).t()
    if layout == "pitch":                    # row-major inside a wider buffer (pitch c+5)
        buf = torch.full((r, c + 5), float("nan"), dtype=torch.float16)
        buf[:, :c] = v
        return buf.to(DEV)[:, :c]
    if layout == "pitch16":                  # pitch rounded up to 16 elements (TMA-able)
        p = (c + 15) // 16 * 16 + 16
        buf = torch.full((r, p), float("nan"), dtype=torch.float16)
        buf[:, :c] = v
        return buf.to(DEV)[:, :c]
    if layout == "offset":                   # base 2 bytes past an aligned address
        flat = torch.full((r * c + 8,), float("nan"), dtype=torch.float16)
        flat[1:1 + r * c] = v.reshape(-1)
        return flat.to(DEV)[1:1 + r * c].view(r, c)
    if layout == "strided":                  # both strides > 1
        buf = torch.full((r * 2, c * 3), float("nan"), dtype=torch.float16)
        buf[::2, ::3] = v
        return buf.to(DEV)[::2, ::3]
    raise ValueError(layout)


LAYOUTS = ("row", "col", "pitch", "pitch16", "offset", "strided")


# -------------------------------------------------------------- tail shape
@pytest.mark.parametrize("w", [workloads.TAIL_ROWMAJOR_B, workloads.TAIL_TRANSPOSED_B], ids=lambda w: w.name)
def test_tail_shape_bit_exact(w):
    A, B = w.A.device_view(DEV), w.B.device_view(DEV)
    assert tuple(B.stride()) == w.B.strides
    C = gpu(A, B)
    ref = oracle.gemm(w.A.host_view(), w.B.host_view())
    assert_bits(host(C), ref, w.name)


@pytest.mark.parametrize("opt,val", [(g.OPT_SWAP, 2), (g.OPT_SPLITS, 2), (g.OPT_TILE_N, 64),
                                     (g.OPT_PANEL, 1), (g.OPT_MAX_CTAS, 1)])
def test_tail_shape_forced_plans_bit_exact(opt, val):
    w = workloads.TAIL_TRANSPOSED_B
    g.gemm_f16_set_option(opt, val)
    C = gpu(w.A.device_view(DEV), w.B.device_view(DEV))
    assert_bits(host(C), oracle.gemm(w.A.host_view(), w.B.host_view()), f"opt {opt}={val}")


# ------------------------------------------------------- random brute force
CASES = []
_rng = np.random.default_rng(1234)
for i in range(36):
    M, N, K = (int(x) for x in _rng.integers(1, 300, 3))
    CASES.append((i, M, N, K, LAYOUTS[_rng.integers(0, 6)], LAYOUTS[_rng.integers(0, 6)],
                  bool(_rng.integers(0, 2))))


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}-{c[4]}-{c[5]}-{'int' if c[6] else 'real'}")
def test_random_shapes_and_layouts(case):
    i, M, N, K, la, lb, integer = case
    rng = np.random.default_rng(100 + i)
    if integer:
        Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
        Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    else:
        Ah = rng.uniform(-1, 1, (M, K)).astype(np.float16)
        Bh = rng.uniform(-1, 1, (K, N)).astype(np.float16)
    C = host(gpu(make_view(Ah, la), make_view(Bh, lb)))
    ref = oracle.gemm(Ah, Bh)
    if integer and K * 9 <= 2048:
        assert_bits(C, ref, str(case))
    else:
        assert_close(C, ref, K, str(case))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 1, 1000), (1, 700, 1), (700, 1, 1), (127, 129, 63),
                                   (128, 256, 64), (129, 257, 65), (256, 512, 4096), (64, 64, 64),
                                   (3, 5000, 333), (65, 300, 129), (2000, 33, 70)])
def test_edge_sizes(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    C = host(gpu(to_dev(Ah), to_dev(Bh)))
    ref = oracle.gemm(Ah, Bh, threads=oracle_threads())
    if K * 9 <= 2048:
        assert_bits(C, ref, f"{M}x{N}x{K}")
    else:
        assert_close(C, ref, K, f"{M}x{N}x{K}")


def test_tma_and_gather_paths_agree_bit_for_bit():
    rng = np.random.default_rng(7)
    A = to_dev(rng.uniform(-1, 1, (520, 336)).astype(np.float16))
    B = to_dev(rng.uniform(-1, 1, (336, 704)).astype(np.float16))
    out = torch.empty((520, 704), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["a_tma"] and plan["b_tma"] and plan["c_tma"] and plan["b_mn_major"]
    C1 = host(gpu(A, B))
    g.gemm_f16_set_option(g.OPT_FORCE_GATHER, 7)
    plan = g.plan_for(A, B, out)
    assert not (plan["a_tma"] or plan["b_tma"] or plan["c_tma"])
    C2 = host(gpu(A, B))
    assert_bits(C1, C2, "tma vs gather")
    assert_close(C1, oracle.gemm(host(A), host(B)), 336, "vs oracle")


def test_mn_major_a_and_k_major_b_through_tma():
    rng = np.random.default_rng(8)
    Ah = rng.uniform(-1, 1, (384, 256)).astype(np.float16)
    Bh = rng.uniform(-1, 1, (256, 320)).astype(np.float16)
    A = make_view(Ah, "col")    # M-major A
    B = make_view(Bh, "col")    # K-major B
    out = torch.empty((384, 320), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["a_tma"] and plan["a_mn_major"] and plan["b_tma"] and not plan["b_mn_major"]
    assert_close(host(gpu(A, B)), oracle.gemm(Ah, Bh), 256, "mn-major A, k-major B")


# MN-major TMA operands whose MN extent is a multiple of 64 are read with one
# 3-D box per stage (all swizzle-atom columns at once); the others with one 2-D
# box per atom column.  Atom columns past the edge of the view must come in as
# zeros, never as the neighbouring elements of memory.
BOX_CASES = [
    # (M, N, K, layout A, layout B, pair option, expected a_box3d, b_box3d)
    (300, 320, 200, "row", "row", 0, 0, 1),       # pair; last tile holds one valid atom column
    (384, 136, 200, "col", "row", 0, 1, 0),       # M-major A in 3-D; N % 64 != 0 keeps B in 2-D
    (200, 576, 216, "row", "row", 1, 0, 1),       # single CTA, four atom columns per box
    (640, 512, 96, "col", "row", 0, 1, 1),        # pair; both operands in 3-D
    (32, 1024, 200, "row", "row", 0, 1, 0),       # swapped: B^T is the M-major kernel A
]


@pytest.mark.parametrize("case", BOX_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-{c[4]}-pair{c[5]}")
def test_mn_major_box_forms_bit_exact(case):
    M, N, K, la, lb, pair, a3, b3 = case
    rng = np.random.default_rng(M * 7 + N + K)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = make_view(Ah, la), make_view(Bh, lb)
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    g.gemm_f16_set_option(g.OPT_PAIR, pair)
    plan = g.plan_for(A, B, out)
    assert (plan["a_box3d"], plan["b_box3d"]) == (a3, b3), plan
    assert_bits(host(gpu(A, B, out=out)), oracle.gemm(Ah, Bh, threads=oracle_threads()), f"boxes {case}")
    assert g.gemm_f16_device_status() == 0


# ------------------------------------------------------------ pair tiles
PAIR_CASES = [
    # (M, N, K, layout A, layout B, tile_n, integer inputs)
    (512, 512, 256, "row", "row", 256, True),
    (1000, 520, 300, "pitch16", "pitch16", 256, True),
    (776, 384, 200, "col", "col", 128, True),       # M-major A, K-major B
    (300, 1000, 136, "row", "col", 256, False),
    (2048, 1024, 1024, "row", "row", 256, False),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-{c[4]}-bn{c[5]}")
def test_pair_tiles_match_oracle(case):
    M, N, K, la, lb, bn, integer = case
    rng = np.random.default_rng(M + N + K)
    if integer:
        Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
        Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    else:
        Ah = rng.uniform(-1, 1, (M, K)).astype(np.float16)
        Bh = rng.uniform(-1, 1, (K, N)).astype(np.float16)
    A, B = make_view(Ah, la), make_view(Bh, lb)
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    g.gemm_f16_set_option(g.OPT_TILE_N, bn)
    g.gemm_f16_set_option(g.OPT_SPLITS, 1)
    single = host(gpu(A, B))
    g.gemm_f16_set_option(g.OPT_PAIR, 2)
    plan = g.plan_for(A, B, out)
    assert plan["pair"] == 1 and plan["tile_m"] == 256 and plan["grid"] % 2 == 0, plan
    paired = host(gpu(A, B, out=out))
    ref = oracle.gemm(Ah, Bh, threads=oracle_threads())
    if integer and K * 9 <= 2048:
        assert_bits(paired, ref, f"pair {case}")
    else:
        assert_close(paired, ref, K, f"pair {case}")
    assert_close(single, ref, K, f"single {case}")
    assert g.gemm_f16_device_status() == 0


def test_pair_tiles_many_units_per_cluster():
    # one cluster walks every tile: exercises the TMEM double buffer and the
    # stage ring across tiles in the pair form
    g.gemm_f16_set_option(g.OPT_PAIR, 2)
    g.gemm_f16_set_option(g.OPT_MAX_CTAS, 2)
    rng = np.random.default_rng(5)
    g.gemm_f16_set_option(g.OPT_SPLITS, 1)
    Ah = rng.integers(-3, 4, (1100, 192)).astype(np.float16)
    Bh = rng.integers(-3, 4, (192, 1296)).astype(np.float16)
    A, B = to_dev(Ah), to_dev(Bh)
    out = torch.empty((1100, 1296), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["pair"] == 1 and plan["grid"] == 2 and plan["units"] > 10
    assert_bits(host(gpu(A, B, out=out)), oracle.gemm(Ah, Bh, threads=oracle_threads()), "pair, one cluster")


# ------------------------------------------------------- boundary behaviour
def test_k_tail_is_zero_filled_not_wrapped():
    # The Triton page's K-tail example (a=[1,2,3], b=[4,5,6] -> 32; wrapping K
    # would give 36).  The elements just past K are NaN in memory: reading any
    # of them would poison the result.
    a = torch.full((1, 8), float("nan"), dtype=torch.float16)
    a[0, :3] = torch.tensor([1.0, 2.0, 3.0])
    b = torch.full((8, 8), float("nan"), dtype=torch.float16)
    b[:3, 0] = torch.tensor([4.0, 5.0, 6.0])
    C = host(gpu(a.to(DEV)[:, :3], b.to(DEV)[:3, :1]))
    assert C[0, 0] == 32.0
    # same on the TMA path: 16-byte pitch, K = 65, NaN beyond K in every row
    rng = np.random.default_rng(9)
    A = torch.full((200, 72), float("nan"), dtype=torch.float16)
    A[:, :65] = torch.from_numpy(rng.integers(-3, 4, (200, 65)).astype(np.float16))
    B = torch.full((72, 136), float("nan"), dtype=torch.float16)
    B[:65, :130] = torch.from_numpy(rng.integers(-3, 4, (65, 130)).astype(np.float16))
    Av, Bv = A.to(DEV)[:, :65], B.to(DEV)[:65, :130]
    out = torch.empty((200, 130), dtype=torch.float16, device=DEV)
    assert g.plan_for(Av, Bv, out)["a_tma"]
    C = host(gpu(Av, Bv))
    assert_bits(C, oracle.gemm(A[:, :65].numpy(), B[:65, :130].numpy()), "tma k-tail")


@pytest.mark.parametrize("force", [0, 7])
def test_only_the_view_of_c_is_written(force):
    g.gemm_f16_set_option(g.OPT_FORCE_GATHER, force)
    rng = np.random.default_rng(10)
    M, N, K, ldc = 300, 200, 96, 264
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    canary = np.float16(-12345.0)
    buf = torch.full((M + 3, ldc), float(canary), dtype=torch.float16, device=DEV)
    out = buf[:M, :N]
    gpu(to_dev(Ah), to_dev(Bh), out=out)
    hb = host(buf)
    assert_bits(hb[:M, :N], oracle.gemm(Ah, Bh), "view")
    assert np.all(hb[:M, N:] == canary) and np.all(hb[M:] == canary)


@pytest.mark.parametrize("N,ldc", [(130, 136), (70, 80), (200, 208)])
def test_pitch_padding_untouched_when_n_is_not_a_multiple_of_8(N, ldc):
    # A TMA-aligned pitch but a row width that ends inside a 16-byte chunk: the
    # padding after column N keeps its NaN.
    rng = np.random.default_rng(N + ldc)
    M, K = 300, 96
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    buf = torch.full((M, ldc), float("nan"), dtype=torch.float16, device=DEV)
    gpu(to_dev(Ah), to_dev(Bh), out=buf[:, :N])
    host_buf = buf.cpu().numpy()
    assert_bits(host_buf[:, :N], oracle.gemm(Ah, Bh), f"N={N}, ldc={ldc}")
    assert np.isnan(host_buf[:, N:]).all()


def test_overflow_gives_inf_like_the_oracle():
    a = torch.full((4, 64), 16.0, dtype=torch.float16, device=DEV)
    b = torch.full((64, 4), 128.0, dtype=torch.float16, device=DEV)
    C = host(gpu(a, b))  # 64 * 2048 = 131072 > 65504
    assert np.all(np.isposinf(C))


# ----------------------------------------------------------------- split-K
def test_split_k_deterministic_and_workspace_paths():
    rng = np.random.default_rng(11)
    M, N, K = 16, 4096, 8192
    Ah = rng.uniform(-1, 1, (M, K)).astype(np.float16)
    Bh = rng.uniform(-1, 1, (K, N)).astype(np.float16)
    A, B = to_dev(Ah), to_dev(Bh)
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    g.gemm_f16_set_option(g.OPT_STREAMK, 2)
    plan = g.plan_for(A, B, out)
    assert plan["swap_ab"] and plan["streamk_tiles"] > 0 and plan["workspace_bytes"] > 0
    C1 = host(gpu(A, B))
    C2 = host(gpu(A, B))
    assert_bits(C1, C2, "split-K repeatability")
    ref = oracle.gemm(Ah, Bh, threads=oracle_threads())
    assert_close(C1, ref, K, "split-K vs oracle")
    # caller-owned workspace gives the same bits
    nbytes = g.gemm_f16_workspace_size(M, N, K)
    assert nbytes >= plan["workspace_bytes"] > 0
    ws = torch.zeros(nbytes // 4 + 64, dtype=torch.int32, device=DEV)
    out2 = torch.empty_like(out)
    g.gemm_f16_ws(A.data_ptr(), K, 1, B.data_ptr(), N, 1, out2.data_ptr(), N, M, N, K,
                  ws.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert_bits(host(out2), C1, "caller workspace")
    # too small a workspace is refused
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16_ws(A.data_ptr(), K, 1, B.data_ptr(), N, 1, out2.data_ptr(), N, M, N, K,
                      ws.data_ptr(), nbytes - 256, 0)
    assert e.value.status == g.ERR_OUT_OF_MEMORY
    # whole tiles only, and classic split-K, change the summation order only
    g.gemm_f16_set_option(g.OPT_STREAMK, 1)
    assert g.plan_for(A, B, out)["streamk_tiles"] == 0
    assert_close(host(gpu(A, B)), ref, K, "no split")
    g.gemm_f16_set_option(g.OPT_STREAMK, 2)
    g.gemm_f16_set_option(g.OPT_SPLITS, 4)
    assert g.plan_for(A, B, out)["splits"] == 4
    C3 = host(gpu(A, B))
    assert_close(C3, ref, K, "classic split-K")
    assert_bits(host(gpu(A, B)), C3, "classic split-K repeatability")


@pytest.mark.parametrize("M,N,K,layout", [(2304, 4608, 64, "row"), (1000, 1000, 100, "pitch"),
                                           (700, 1536, 136, "row"), (3000, 700, 72, "pitch16")])
def test_tail_split_bit_exact(M, N, K, layout):
    """The last partial wave of tiles is cut along N into narrower tiles; every
    output is still one complete K reduction, so integer inputs stay exact."""
    rng = np.random.default_rng(M + N + K)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = make_view(Ah, layout), make_view(Bh, layout)
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    g.gemm_f16_set_option(g.OPT_STREAMK, 1)   # whole tiles (gathered operands default to stream-K)
    plan = g.plan_for(A, B, out)
    assert plan["tail_split"] > 1, plan
    ref = oracle.gemm(Ah, Bh, threads=oracle_threads())
    assert_bits(host(gpu(A, B, out=out)), ref, f"tail split {M}x{N}x{K}")
    g.gemm_f16_set_option(g.OPT_TAIL_SPLIT, 1)
    assert g.plan_for(A, B, out)["tail_split"] == 1
    assert_bits(host(gpu(A, B, out=out)), ref, f"no tail split {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,layout", [(1000, 1000, 1000, "pitch"), (3001, 1999, 200, "offset")])
def test_gathered_operands_default_to_stream_k(M, N, K, layout):
    """Gathered (non-TMA) operands make tiles slow, so by default the last
    partial wave is balanced by stream-K; integer inputs stay bit-exact.  (The
    aligned-copy path is switched off: these products are large enough that it
    would replace the gather.)"""
    g.gemm_f16_set_option(g.OPT_REPACK, 1)
    rng = np.random.default_rng(M + 5 * N + K)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = make_view(Ah, layout), make_view(Bh, layout)
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert not (plan["a_tma"] and plan["b_tma"]) and plan["streamk_tiles"] > 0, plan
    assert_bits(host(gpu(A, B, out=out)), oracle.gemm(Ah, Bh, threads=oracle_threads()), f"gathered {M}x{N}x{K}")
    assert g.gemm_f16_device_status() == 0


def _segment_end(ptr):
    """End address of the caching-allocator segment (one cudaMalloc) holding ptr."""
    for seg in torch.cuda.memory_snapshot():
        if seg["address"] <= ptr < seg["address"] + seg["total_size"]:
            return seg["address"] + seg["total_size"]
    return None


@pytest.mark.parametrize("M,N,K,pair", [(1000, 1024, 704, 0), (1000, 1024, 704, 2), (2304, 4608, 320, 0),
                                        (2304, 4608, 320, 2), (16, 1040, 6000, 0), (200, 56, 9000, 0)])
def test_stream_k_bit_exact(M, N, K, pair):
    """Tiles cut along K by the stream-K schedule are summed exactly once, in K
    order; integer inputs make every order exact, so the result is unique."""
    g.gemm_f16_set_option(g.OPT_PAIR, pair)
    g.gemm_f16_set_option(g.OPT_STREAMK, 2)
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    hi = 3 if K * 9 <= 2048 else 1
    Ah = rng.integers(-hi, hi + 1, (M, K)).astype(np.float16)
    Bh = rng.integers(-hi, hi + 1, (K, N)).astype(np.float16)
    A, B = to_dev(Ah), to_dev(Bh)
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["streamk_tiles"] > 0, plan
    if pair == 2:
        assert plan["pair"] == 1, plan
    got = host(gpu(A, B, out=out))
    ref = oracle.gemm(Ah, Bh, threads=oracle_threads())
    if np.abs(ref.astype(np.float64)).max() <= 2048:
        assert_bits(got, ref, f"stream-K {M}x{N}x{K}")
    else:
        assert_close(got, ref, K, f"stream-K {M}x{N}x{K}")
    assert_bits(host(gpu(A, B, out=out)), got, "stream-K repeatability")
    g.gemm_f16_set_option(g.OPT_STREAMK, 1)
    assert g.plan_for(A, B, out)["streamk_tiles"] == 0
    assert_close(host(gpu(A, B, out=out)), ref, K, "whole tiles")


def test_alias_and_bad_memory_rejected_on_device():
    # Every check here goes through gemm_f16_get_plan, which validates exactly
    # like gemm_f16 but never launches, so a view that is wrong on purpose
    # cannot reach the GPU.
    A = torch.zeros((64, 64), dtype=torch.float16, device=DEV)
    B = torch.zeros((64, 64), dtype=torch.float16, device=DEV)
    C = torch.empty((64, 64), dtype=torch.float16, device=DEV)
    with pytest.raises(g.GemmF16Error) as e:
        g.matmul(A, B, out=A)
    assert e.value.status == g.ERR_ALIAS
    # the same arguments with C elsewhere are accepted
    g.gemm_f16_get_plan(A.data_ptr(), 64, 1, B.data_ptr(), 64, 1, C.data_ptr(), 64, 64, 64, 64)
    # A's view ends 2 bytes past the end of the cudaMalloc segment holding it
    end = _segment_end(A.data_ptr())
    assert end is not None
    start = end - 2 * 64 * 64 + 2
    start -= start % 16
    a_ptr = start + 2 * ((end - start) // 2 - 64 * 64 + 1)
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16_get_plan(a_ptr, 64, 1, B.data_ptr(), 64, 1, C.data_ptr(), 64, 64, 64, 64)
    assert e.value.status in (g.ERR_INVALID_VALUE, g.ERR_ALIAS)
    if not (C.data_ptr() < end + 2 and a_ptr < C.data_ptr() + 2 * 64 * 64):
        assert e.value.status == g.ERR_INVALID_VALUE
    # the view that ends exactly at the segment end is fine
    ok_ptr = end - 2 * 64 * 64
    if not (ok_ptr < C.data_ptr() + 2 * 64 * 64 and C.data_ptr() < end):
        g.gemm_f16_get_plan(ok_ptr, 64, 1, B.data_ptr(), 64, 1, C.data_ptr(), 64, 64, 64, 64)
    # host memory is refused, pageable or pinned
    h = torch.zeros((64, 64), dtype=torch.float16)
    for hp in (h, h.pin_memory()):
        with pytest.raises(g.GemmF16Error) as e:
            g.gemm_f16_get_plan(hp.data_ptr(), 64, 1, B.data_ptr(), 64, 1, C.data_ptr(), 64, 64, 64, 64)
        assert e.value.status == g.ERR_INVALID_VALUE
        with pytest.raises(g.GemmF16Error) as e:
            g.gemm_f16(A.data_ptr(), 64, 1, B.data_ptr(), 64, 1, hp.data_ptr(), 64, 64, 64, 64)
        assert e.value.status == g.ERR_INVALID_VALUE
    # memory of another GPU (when one is visible) is refused: operands must be
    # on the current device
    if torch.cuda.device_count() > 1:
        other = torch.zeros((64, 64), dtype=torch.float16, device=torch.device("cuda:1"))
        torch.cuda.set_device(DEV)
        with pytest.raises(g.GemmF16Error) as e:
            g.gemm_f16_get_plan(other.data_ptr(), 64, 1, B.data_ptr(), 64, 1, C.data_ptr(), 64, 64, 64, 64)
        assert e.value.status == g.ERR_INVALID_VALUE


# ---------------------------------------------------- the five configurations
def test_device_generator_matches_host():
    for kind, seed, n in (("uniform", 2, 1 << 20), ("int3", 1, 12345)):
        d = synth.buffer_torch(kind, seed, n, DEV).cpu().numpy()
        assert np.array_equal(d.view(np.uint16), synth.buffer_np(kind, seed, n).view(np.uint16))


def _run_workload(w):
    A, B = w.A.device_view(DEV), w.B.device_view(DEV)
    assert tuple(A.stride()) == w.A.strides and tuple(B.stride()) == w.B.strides
    C = gpu(A, B)
    del A, B
    return C


def test_decode_m16_full_output():
    w = workloads.DECODE_16x16384x8192
    C = host(_run_workload(w))
    ref = oracle.gemm(w.A.host_view(), w.B.host_view(), threads=oracle_threads())
    assert_close(C, ref, w.K, w.name)


def test_irregular_strided_full_output():
    w = workloads.IRREGULAR_3001x1999x4097
    C = host(_run_workload(w))
    ref = oracle.gemm(w.A.host_view(), w.B.host_view(), threads=oracle_threads())
    assert_close(C, ref, w.K, w.name)


def test_square_4096_full_output():
    """Every one of the 4096 x 4096 outputs against the oracle (on all host
    cores: about ten seconds), in the launch configuration the bench times."""
    w = workloads.SQUARE_4096
    C = host(_run_workload(w))
    ref = oracle.gemm(w.A.host_view(), w.B.host_view(), threads=oracle_threads())
    assert_close(C, ref, w.K, w.name)


@pytest.mark.parametrize("w", [workloads.MOE_131072x2048x7168], ids=lambda w: w.name)
def test_large_sampled_plus_boundary_tile(w):
    """The MoE-flattened shape is too large for the host oracle (1.9e12
    multiply-adds): 4096 seeded random outputs and the whole last tile."""
    C = _run_workload(w)
    rng = np.random.default_rng(20260)
    ms = rng.integers(0, w.M, 4096)
    ns = rng.integers(0, w.N, 4096)
    got = C[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)].cpu().numpy()
    assert_close(got, sampled_reference(w, ms, ns), w.K, f"{w.name} samples")
    out = torch.empty((1, 1), dtype=torch.float16, device=DEV)
    bm, bn = 128, 256
    tile = C[w.M - bm:, w.N - bn:].cpu().numpy()
    assert_close(tile, block_reference(w, w.M - bm, w.M, w.N - bn, w.N), w.K, f"{w.name} last tile")
    del out


def test_no_kernel_reported_a_timeout():
    assert g.gemm_f16_device_status(reset=True) == 0


@pytest.mark.parametrize("M,N,K", [(16, 16, (1 << 20) + 3),       # 16385 K blocks, swapped form
                                   ((1 << 20) + 5, 64, 64),       # 4097 pair tile rows
                                   (64, (1 << 20) + 7, 64),       # swapped: 8193 tiles along N
                                   (3, 3, (1 << 21) + 1)])         # long K through split-K / stream-K
def test_long_dimensions(M, N, K):
    """One very long dimension: tile and K-block counts in the thousands, int64
    offsets well past 2^31 bytes.  Integer inputs in [-1, 1]: every partial sum
    is an integer below 2^24, exact in fp32 in any order, so the one rounding to
    fp16 matches the oracle's bit for bit."""
    rng = np.random.default_rng(M + N + K)
    Ah = rng.integers(-1, 2, (M, K)).astype(np.float16)
    Bh = rng.integers(-1, 2, (K, N)).astype(np.float16)
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    C = host(gpu(to_dev(Ah), to_dev(Bh), out=out))
    assert_bits(C, oracle.gemm(Ah, Bh, threads=oracle_threads()), f"{M}x{N}x{K}")
    assert g.gemm_f16_device_status() == 0


@pytest.mark.parametrize("opts", [
    {g.OPT_STREAMK: 2, g.OPT_MAX_STAGES: 2},                  # pair form, 2-slot ring: 8-piece landing zone
    {g.OPT_STREAMK: 2, g.OPT_MAX_STAGES: 2, g.OPT_TAIL_SPLIT: 1},
    {g.OPT_STREAMK: 2, g.OPT_MAX_STAGES: 4},
    {g.OPT_SPLITS: 3, g.OPT_MAX_STAGES: 2, g.OPT_PAIR: 1},
])
def test_shallow_ring_with_k_cuts(opts):
    """Tiles cut along K with a shallow ring: the last unit of a worker collects
    the other partials in the (small) stage area, in batches narrower than a
    64-column TMA-store box; those batches must not go out as whole boxes
    (which would overwrite the next tile's columns)."""
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    rng = np.random.default_rng(4486)
    M, N, K = 1190, 1216, 2986
    Ah = rng.integers(-2, 3, (M, K)).astype(np.float16)
    Bh = rng.integers(-2, 3, (K, N)).astype(np.float16)
    A, B = to_dev(Ah), to_dev(Bh)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["streamk_tiles"] > 0 or plan["splits"] > 1, plan
    C = host(gpu(A, B, out=out))
    assert_bits(C, oracle.gemm(Ah, Bh, threads=oracle_threads()), f"shallow ring {opts}")
    assert g.gemm_f16_device_status() == 0


# ------------------------------------------------------ L2 eviction policies
@pytest.mark.parametrize("a,b,c", [(2, 3, 1), (3, 2, 2), (2, 2, 3), (1, 3, 2)])
@pytest.mark.parametrize("case", [(1100, 1288, 896, "row", "row", {}),            # pair form, 3-D B boxes
                                  (704, 520, 296, "col", "col", {g.OPT_PAIR: 1}),  # single form, MN-major A
                                  (1190, 1216, 2984, "row", "row", {g.OPT_STREAMK: 2})])
def test_l2_policies_do_not_change_results(case, a, b, c):
    """Eviction policies on the operand copies and the C stores only steer L2
    replacement: every combination gives the oracle's result bit for bit."""
    M, N, K, la, lb, opts = case
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    g.gemm_f16_set_option(g.OPT_L2_A, a)
    g.gemm_f16_set_option(g.OPT_L2_B, b)
    g.gemm_f16_set_option(g.OPT_L2_C, c)
    rng = np.random.default_rng(M + 7 * N + K + a)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = make_view(Ah, la), make_view(Bh, lb)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["a_tma"] and plan["b_tma"] and plan["c_tma"] and not plan["repack"], plan
    assert_bits(host(gpu(A, B, out=out)), oracle.gemm(Ah, Bh, threads=oracle_threads()), f"L2 {a}{b}{c} {case[:5]}")
    assert g.gemm_f16_device_status() == 0


# ----------------------------------- K segments for swapped small-M pairs
# (M, N, K, B transposed, segments: 64 pair tiles take 2, 48 take 3, 56 take 4
# when each segment keeps 8 K blocks, 40 keep stream-K)
@pytest.mark.parametrize("M,N,K,bt,S", [(16, 16384, 1024, False, 2), (40, 12288, 1600, False, 3),
                                        (16, 14336, 2048, True, 4), (16, 14336, 1024, False, 1),
                                        (16, 10240, 2048, True, 1)])
def test_swapped_pairs_take_k_segments(M, N, K, bt, S):
    """A swapped pair plan whose tiles are fewer than the clusters but at least
    half as many runs S K segments per tile (classic split-K, units numbered
    segment-major) when S fills the waves of units; the last of a tile's units
    adds the others' partials.  Bit for bit on integers, the same bits through a
    caller workspace of the size gemm_f16_workspace_size reports, and the same
    as stream-K."""
    rng = np.random.default_rng(M * 7 + N + K)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A = to_dev(Ah)
    B = make_view(Bh, "col" if bt else "row")
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["swap_ab"] and plan["pair"] and plan["splits"] == S, plan
    assert (plan["streamk_tiles"] > 0) == (S == 1) and plan["workspace_bytes"] > 0, plan
    C = host(gpu(A, B, out=out))
    assert_bits(C, oracle.gemm(Ah, Bh, threads=oracle_threads()), f"{S} K segments {M}x{N}x{K}")
    nbytes = g.gemm_f16_workspace_size(M, N, K)
    assert nbytes >= plan["workspace_bytes"]
    ws = torch.zeros(nbytes // 4 + 64, dtype=torch.int32, device=DEV)
    out2 = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    g.gemm_f16_ws(A.data_ptr(), A.stride(0), A.stride(1), B.data_ptr(), B.stride(0), B.stride(1), out2.data_ptr(), N,
                  M, N, K, ws.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert_bits(host(out2), C, "caller workspace")
    g.gemm_f16_set_option(g.OPT_STREAMK, 2)   # a forced stream-K keeps stream-K
    p2 = g.plan_for(A, B, out)
    assert p2["splits"] == 1 and p2["streamk_tiles"] > 0, p2
    assert_bits(host(gpu(A, B, out=out)), C, "stream-K")
    assert g.gemm_f16_device_status() == 0


# ---------------------------------------------- swapped form on CTA pairs
@pytest.mark.parametrize("M,N,K", [(16, 4096, 1024), (48, 2048, 520), (8, 3000, 640), (40, 16384, 2048)])
def test_swapped_small_m_on_pairs(M, N, K):
    """Small M computed as C^T = B^T A^T on 2-CTA pairs (M = 256 per MMA, each
    CTA loading half of the BN activation rows): the default for a row-major A."""
    rng = np.random.default_rng(M * 31 + N + K)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = to_dev(Ah), to_dev(Bh)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    plan = g.plan_for(A, B, out)
    assert plan["swap_ab"] and plan["pair"] and plan["tile_m"] == 256, plan
    C = host(gpu(A, B, out=out))
    assert_bits(C, oracle.gemm(Ah, Bh, threads=oracle_threads()), f"swapped pairs {M}x{N}x{K}")
    assert_bits(host(gpu(A, B, out=out)), C, "repeatable")
    assert g.gemm_f16_device_status() == 0
