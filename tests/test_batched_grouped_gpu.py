"""Parity of the batched and grouped entry points with the CPU oracle.

Batched GEMM follows the TileLang tutorial ch. 14 "GEMM operators", section 4.4;
grouped GEMM section 4.3.  Integer inputs in [-3, 3] make every sum exact, so
those cases are compared bit for bit; real inputs within the stated tolerance.
"""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from synth import workloads
from tests.parity import assert_bits, assert_close, assert_close_fused, oracle_threads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for o in (g.OPT_FORCE_GATHER, g.OPT_SPLITS, g.OPT_TILE_N, g.OPT_PANEL, g.OPT_SWAP,
              g.OPT_TIMEOUT_MS, g.OPT_MAX_CTAS, g.OPT_PAIR, g.OPT_STREAMK, g.OPT_TAIL_SPLIT, g.OPT_MAX_STAGES,
              g.OPT_REPACK):
        g.gemm_f16_set_option(o, 0)


def ints(rng, shape):
    return rng.integers(-3, 4, shape).astype(np.float16)


def reals(rng, shape):
    return rng.uniform(-1, 1, shape).astype(np.float16)


def dev(x):
    # (a writable copy: some operands are read-only broadcast views)
    return torch.from_numpy(np.array(x, order="C", copy=True)).to(DEV)


# ------------------------------------------------------------------ batched
BATCHED = [
    # (batch, M, N, K, integer, how A and B are laid out)
    (4, 300, 260, 200, True, "contiguous"),          # batch dimension in the TMA maps
    (3, 1000, 512, 128, True, "contiguous"),          # pair tiles
    (5, 130, 70, 65, True, "contiguous"),             # the ragged 130x70x65 shape per problem
    (6, 200, 192, 136, True, "shared_b"),             # one B for every problem (stride 0)
    (4, 140, 96, 72, True, "odd_stride"),             # batch strides not 16-byte multiples: gathered
    (8, 16, 1024, 512, True, "contiguous"),           # small M: swapped form per problem
    (2, 768, 768, 1024, False, "contiguous"),
]


def _batched_case(rng, nb, M, N, K, integer, layout):
    mk = ints if integer else reals
    Ah, Bh = mk(rng, (nb, M, K)), mk(rng, (nb, K, N))
    if layout == "shared_b":
        Bh = np.broadcast_to(Bh[:1], (nb, K, N))
        B = dev(Bh[0]).unsqueeze(0).expand(nb, K, N)
        A = dev(Ah)
    elif layout == "odd_stride":
        # each problem padded by 3 elements: batch strides M*K+3, K*N+3
        Abuf = torch.full((nb, M * K + 3), float("nan"), dtype=torch.float16)
        Bbuf = torch.full((nb, K * N + 3), float("nan"), dtype=torch.float16)
        Abuf[:, :M * K] = torch.from_numpy(Ah.reshape(nb, -1))
        Bbuf[:, :K * N] = torch.from_numpy(Bh.reshape(nb, -1))
        Abuf, Bbuf = Abuf.to(DEV), Bbuf.to(DEV)
        A = Abuf.as_strided((nb, M, K), (M * K + 3, K, 1))
        B = Bbuf.as_strided((nb, K, N), (K * N + 3, N, 1))
    else:
        A, B = dev(Ah), dev(Bh)
    return Ah, Bh, A, B


@pytest.mark.parametrize("case", BATCHED, ids=lambda c: f"b{c[0]}-{c[1]}x{c[2]}x{c[3]}-{c[5]}")
def test_batched_matches_oracle(case):
    nb, M, N, K, integer, layout = case
    rng = np.random.default_rng(nb * 1000 + M + N + K)
    Ah, Bh, A, B = _batched_case(rng, nb, M, N, K, integer, layout)
    C = g.bmm(A, B)
    torch.cuda.synchronize()
    ref = oracle.gemm_batched(Ah, Bh, threads=oracle_threads())
    got = C.cpu().numpy()
    for b in range(nb):
        if integer:
            assert_bits(got[b], ref[b], f"batched {case} problem {b}")
        else:
            assert_close(got[b], ref[b], K, f"batched {case} problem {b}")
    assert g.gemm_f16_device_status() == 0


def test_batched_gather_and_stream_k_agree_bit_for_bit():
    rng = np.random.default_rng(31)
    Ah, Bh = reals(rng, (3, 520, 700)), reals(rng, (3, 700, 384))
    A, B = dev(Ah), dev(Bh)
    C1 = g.bmm(A, B).cpu().numpy()
    g.gemm_f16_set_option(g.OPT_FORCE_GATHER, 7)
    C2 = g.bmm(A, B).cpu().numpy()
    assert_bits(C1, C2, "TMA vs gather")
    g.gemm_f16_set_option(g.OPT_FORCE_GATHER, 0)
    g.gemm_f16_set_option(g.OPT_STREAMK, 2)
    C3 = g.bmm(A, B).cpu().numpy()
    assert_close(C3, oracle.gemm_batched(Ah, Bh, threads=oracle_threads()), 700, "stream-K batched")
    assert g.gemm_f16_device_status() == 0


def test_batched_writes_only_the_views():
    # C problems placed with a gap of NaN between them: the gaps stay NaN
    rng = np.random.default_rng(32)
    nb, M, N, K = 3, 200, 130, 64
    Ah, Bh = ints(rng, (nb, M, K)), ints(rng, (nb, K, N))
    stride = M * 136 + 40   # ldc 136 > N, and a gap after every problem
    Cbuf = torch.full((nb * stride,), float("nan"), dtype=torch.float16, device=DEV)
    C = Cbuf.as_strided((nb, M, N), (stride, 136, 1))
    g.bmm(dev(Ah), dev(Bh), out=C)
    torch.cuda.synchronize()
    ref = oracle.gemm_batched(Ah, Bh)
    assert_bits(C.cpu().numpy(), ref, "strided batched C")
    host = Cbuf.cpu()
    written = torch.zeros(nb * stride, dtype=torch.bool)
    idx = (torch.arange(nb)[:, None, None] * stride + torch.arange(M)[None, :, None] * 136
           + torch.arange(N)[None, None, :]).reshape(-1)
    written[idx] = True
    assert torch.isnan(host[~written]).all()


def test_batched_rejects_overlapping_outputs():
    A = torch.zeros((2, 64, 64), dtype=torch.float16, device=DEV)
    B = torch.zeros((2, 64, 64), dtype=torch.float16, device=DEV)
    C = torch.zeros((64 * 64 + 10,), dtype=torch.float16, device=DEV)
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16_batched(A.data_ptr(), 64 * 64, 64, 1, B.data_ptr(), 64 * 64, 64, 1, C.data_ptr(), 10, 64,
                           64, 64, 64, 2)
    assert e.value.status == g.ERR_INVALID_VALUE


# ------------------------------------------------------------------ grouped
GROUPED = [
    # (group rows, N, K, integer)
    ([130, 0, 256, 1, 700], 320, 200, True),        # empty and one-row groups, ragged ends
    ([512, 384, 640], 512, 136, True),              # pair tiles, whole and ragged groups
    ([37] * 9, 96, 72, True),                       # many small groups
    ([1000, 3000, 50], 1024, 512, False),
]


@pytest.mark.parametrize("case", GROUPED, ids=lambda c: f"g{len(c[0])}-{sum(c[0])}x{c[1]}x{c[2]}")
def test_grouped_matches_oracle(case):
    rows, N, K, integer = case
    rng = np.random.default_rng(sum(rows) + N + K)
    mk = ints if integer else reals
    Ah, Bh = mk(rng, (sum(rows), K)), mk(rng, (len(rows), K, N))
    # C with NaN rows after the groups' rows: nothing past them may be written
    Cbuf = torch.full((sum(rows) + 5, N), float("nan"), dtype=torch.float16, device=DEV)
    g.grouped_mm(dev(Ah), dev(Bh), rows, out=Cbuf[:sum(rows)])
    torch.cuda.synchronize()
    ref = oracle.gemm_grouped(Ah, Bh, rows, threads=oracle_threads())
    got = Cbuf.cpu().numpy()
    if integer:
        assert_bits(got[:sum(rows)], ref, f"grouped {case}")
    else:
        assert_close(got[:sum(rows)], ref, K, f"grouped {case}")
    assert np.isnan(got[sum(rows):]).all()
    assert g.gemm_f16_device_status() == 0


def test_grouped_stream_k_and_gather_paths():
    rng = np.random.default_rng(41)
    rows, N, K = [300, 0, 900, 77], 256, 640
    Ah, Bh = ints(rng, (sum(rows), K)), ints(rng, (len(rows), K, N))
    ref = oracle.gemm_grouped(Ah, Bh, rows, threads=oracle_threads())
    A, B = dev(Ah), dev(Bh)
    for opt, val in ((g.OPT_STREAMK, 2), (g.OPT_FORCE_GATHER, 7), (g.OPT_SPLITS, 3)):
        g.gemm_f16_set_option(opt, val)
        assert_bits(g.grouped_mm(A, B, rows).cpu().numpy(), ref, f"grouped, option {opt}={val}")
        g.gemm_f16_set_option(opt, 0)
    assert g.gemm_f16_device_status() == 0


def test_grouped_all_empty_does_nothing():
    A = torch.zeros((0, 64), dtype=torch.float16, device=DEV)
    B = torch.zeros((3, 64, 64), dtype=torch.float16, device=DEV)
    C = torch.zeros((0, 64), dtype=torch.float16, device=DEV)
    anchor = torch.zeros(8, dtype=torch.float16, device=DEV)
    g.gemm_f16_grouped(anchor.data_ptr(), 64, 1, B.data_ptr(), 64 * 64, 64, 1, anchor.data_ptr(), 64,
                       [0, 0, 0], 64, 64)
    torch.cuda.synchronize()
    assert C.numel() == 0 and g.gemm_f16_device_status() == 0


# ------------------------------------------------------- full-size workloads
def _launch_as_bench(w, A, B, C, U=None):
    """The call bench.py times for a multi-problem workload."""
    M, N, K, n = w.M, w.N, w.K, w.count
    if U is not None or w.act != "none":
        up, act = (U.data_ptr() if U is not None else 0), g.ACTIVATIONS[w.act]
        if w.kind == "batched":
            g.gemm_f16_batched_fused(A.data_ptr(), M * K, K, 1, B.data_ptr(), K * N, N, 1, up, 0, 0, 0, act,
                                     C.data_ptr(), M * N, N, M, N, K, n)
        else:
            g.gemm_f16_grouped_fused(A.data_ptr(), K, 1, B.data_ptr(), K * N, N, 1, up, 0, 0, 0, act, C.data_ptr(),
                                     N, list(w.group_rows), N, K)
    elif w.kind == "batched":
        g.gemm_f16_batched(A.data_ptr(), M * K, K, 1, B.data_ptr(), K * N, N, 1, C.data_ptr(), M * N, N,
                           M, N, K, n)
    else:
        g.gemm_f16_grouped(A.data_ptr(), K, 1, B.data_ptr(), K * N, N, 1, C.data_ptr(), N, list(w.group_rows),
                           N, K)


def _problem_of_rows(w, rows):
    """Problem (batched) or group (grouped) index of each stacked output row."""
    if w.kind == "batched":
        return rows // w.M
    ends = np.cumsum(w.group_rows)
    return np.searchsorted(ends, rows, side="right")


@pytest.mark.parametrize("w", workloads.MULTI, ids=lambda w: w.name)
def test_full_size_workload_sampled(w):
    """Sampled outputs of the bench's batched / grouped workloads at full size,
    plus the first and last row of every problem, against the oracle's dot
    products over the regenerated rows of A and columns of B."""
    A, B = w.A.device_view(DEV), w.B.device_view(DEV)
    U = w.B_up.device_view(DEV) if w.B_up is not None else None
    C = torch.full((w.c_rows, w.N), float("nan"), dtype=torch.float16, device=DEV)
    _launch_as_bench(w, A, B, C, U)
    torch.cuda.synchronize()
    del A, B, U
    assert not torch.isnan(C).any(), "an output element was not written"
    K = w.K
    if w.kind == "batched":
        starts = np.arange(w.count, dtype=np.int64) * w.M
        ends = starts + w.M
    else:
        ends = np.cumsum(np.asarray(w.group_rows, dtype=np.int64))
        starts = ends - np.asarray(w.group_rows, dtype=np.int64)
    rng = np.random.default_rng(20261)
    edge = np.concatenate([starts, ends - 1])
    rows = np.concatenate([rng.integers(0, w.c_rows, 2048), edge])
    cols = np.concatenate([rng.integers(0, w.N, 2048), rng.integers(0, w.N, edge.size)])
    cols[-4:] = w.N - 1
    prob = _problem_of_rows(w, rows)
    k = np.arange(K, dtype=np.int64)
    A_rows = w.A.values_at(rows[:, None], k[None, :])                    # [S, K]
    B_cols = w.B.values_at(prob[:, None] * K + k[None, :], cols[:, None])  # [S, K]
    idx = np.arange(rows.size, dtype=np.int64) * K
    ref, S = oracle.dots(A_rows.reshape(-1), idx, 1, B_cols.reshape(-1), idx, 1, K, threads=oracle_threads())
    got = C[torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)].cpu().numpy()
    if w.B_up is None and w.act == "none":
        assert_close(got, ref, K, f"{w.name} samples")
    else:
        S_up = None
        if w.B_up is not None:
            U_cols = w.B_up.values_at(prob[:, None] * K + k[None, :], cols[:, None])
            _, S_up = oracle.dots(A_rows.reshape(-1), idx, 1, U_cols.reshape(-1), idx, 1, K,
                                  threads=oracle_threads())
        ref, gp, u = oracle.epilogue(S, w.act, 0.0, S_up, 0.0)
        assert_close_fused(got, ref, K, gp, u, w.act, f"{w.name} samples")
    assert g.gemm_f16_device_status() == 0


@pytest.mark.parametrize("rows,N,K,opts", [
    ([194, 241, 0, 165, 273, 217, 64, 0], 206, 1, {}),          # K = 1: A [rows, 1] has unit strides both ways
    ([215, 236], 28, 1, {g.OPT_PAIR: 1, g.OPT_TAIL_SPLIT: 1}),
    ([130, 77, 301], 256, 96, {}),                              # A column-major, group starts 130, 207
    ([130, 77, 301], 256, 96, {g.OPT_REPACK: 2}),               # ... through the aligned copy (K-major)
    ([512, 384, 640], 512, 136, {}),                            # starts on multiples of 8: MN-major TMA A
    ([8, 120, 64, 64], 256, 136, {}),                           # starts 0, 8, 128, 192: MN-major TMA A in
    ([200, 56, 256], 256, 96, {}),                              # 64-row boxes only where a group starts on one
])
def test_grouped_column_major_a(rows, N, K, opts):
    """A whose rows are contiguous in memory (a transposed view, or K = 1): in a
    grouped call each group's first row is the innermost TMA coordinate of an
    MN-major A box, which must sit on a 16-byte boundary; groups that start
    elsewhere take the gather or a K-major copy.  Bit-exact either way."""
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    rng = np.random.default_rng(sum(rows) + N + K)
    Ah, Bh = ints(rng, (sum(rows), K)), ints(rng, (len(rows), K, N))
    A = torch.from_numpy(np.ascontiguousarray(Ah.T)).to(DEV).t()     # strides (1, rows)
    C = g.grouped_mm(A, dev(Bh), rows)
    torch.cuda.synchronize()
    assert_bits(C.cpu().numpy(), oracle.gemm_grouped(Ah, Bh, rows), f"grouped, column-major A {rows}")
    U = ints(rng, (len(rows), K, N))
    C = g.grouped_fused_mm(A, dev(Bh), rows, act="relu", b_up=dev(U))
    torch.cuda.synchronize()
    assert_bits(C.cpu().numpy(), oracle.gemm_fused_grouped(Ah, Bh, rows, U, act="relu"), "fused, column-major A")
    assert g.gemm_f16_device_status() == 0


@pytest.mark.parametrize("rows,K", [([8, 120, 64, 64], 136), ([200, 56, 259], 96), ([64, 1000], 72)])
def test_grouped_column_major_a_through_the_aligned_copy(rows, K):
    """A column-major A whose pitch (total rows + 3) TMA cannot take, copied to
    an aligned MN-major buffer whose rows are padded to whole 64-row atoms and
    read with the one-box-per-stage form where the group starts allow it."""
    g.gemm_f16_set_option(g.OPT_REPACK, 2)
    N = 256
    rng = np.random.default_rng(sum(rows) * 7 + K)
    Ah, Bh = ints(rng, (sum(rows), K)), ints(rng, (len(rows), K, N))
    buf = torch.full((K, sum(rows) + 3), float("nan"), dtype=torch.float16)
    buf[:, :sum(rows)] = torch.from_numpy(np.ascontiguousarray(Ah.T))
    A = buf.to(DEV)[:, :sum(rows)].t()                                # strides (1, rows + 3)
    C = g.grouped_mm(A, dev(Bh), rows)
    torch.cuda.synchronize()
    assert_bits(C.cpu().numpy(), oracle.gemm_grouped(Ah, Bh, rows), f"grouped, copied column-major A {rows}")
    assert g.gemm_f16_device_status() == 0
