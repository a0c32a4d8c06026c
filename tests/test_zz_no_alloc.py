"""gemm_f16_noalloc: the entry point for callers that must not allocate.

Some callers cannot call cudaMalloc (all device memory already handed to their
own pool, or a code path where an allocation, and the device synchronisation
it implies, is not allowed).  gemm_f16_noalloc keeps the split-K / stream-K
partial sums in the library's fixed device array instead of a workspace it
would allocate.  This file runs after the other test files, so a failure here
does not hide theirs; it sets every option it needs and restores the defaults.
"""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from tests.parity import assert_close, oracle_threads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _defaults():
    for o in (g.OPT_FORCE_GATHER, g.OPT_SPLITS, g.OPT_TILE_N, g.OPT_PANEL, g.OPT_SWAP,
              g.OPT_TIMEOUT_MS, g.OPT_MAX_CTAS, g.OPT_PAIR, g.OPT_STREAMK, g.OPT_TAIL_SPLIT, g.OPT_MAX_STAGES):
        g.gemm_f16_set_option(o, 0)
    yield
    for o in (g.OPT_STREAMK, g.OPT_SPLITS):
        g.gemm_f16_set_option(o, 0)


def _args(A, B, C):
    M, K = A.shape
    N = B.shape[1]
    return (A.data_ptr(), A.stride(0), A.stride(1), B.data_ptr(), B.stride(0), B.stride(1),
            C.data_ptr(), C.stride(0), M, N, K)


@pytest.mark.parametrize("streamk,splits", [(2, 0), (0, 4)])
def test_no_alloc_entry_matches_gemm_f16(streamk, splits):
    torch.cuda.set_device(DEV)
    g.gemm_f16_set_option(g.OPT_STREAMK, streamk)
    g.gemm_f16_set_option(g.OPT_SPLITS, splits)
    rng = np.random.default_rng(31)
    M, N, K = 16, 4096, 8192          # small M: the plan cuts tiles along K
    Ah = rng.uniform(-1, 1, (M, K)).astype(np.float16)
    Bh = rng.uniform(-1, 1, (K, N)).astype(np.float16)
    A = torch.from_numpy(Ah).to(DEV)
    B = torch.from_numpy(Bh).to(DEV)
    ref_out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    plan = g.gemm_f16_get_plan(*_args(A, B, ref_out))
    assert 0 < plan["workspace_bytes"] <= g.NOALLOC_SCRATCH_BYTES, plan
    stream = torch.cuda.current_stream(DEV).cuda_stream
    g.gemm_f16(*_args(A, B, ref_out), stream=stream)
    torch.cuda.synchronize(DEV)
    expected = ref_out.cpu().numpy()
    for call in range(2):                       # the array keeps the last call's contents
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        g.gemm_f16_noalloc(*_args(A, B, out), stream=stream)
        torch.cuda.synchronize(DEV)
        got = out.cpu().numpy()
        assert_close(got, expected, K, f"noalloc call {call} vs gemm_f16")
    assert_close(got, oracle.gemm(Ah, Bh, threads=oracle_threads()), K, "noalloc vs oracle")
    assert g.gemm_f16_device_status() == 0


def test_no_alloc_rejects_a_plan_beyond_its_scratch():
    # 128 x 4096 x 65536 with stream-K cuts 32-wide tiles over every SM; the
    # partials need far more than 8 MiB, so the call is refused before launch.
    g.gemm_f16_set_option(g.OPT_STREAMK, 2)
    M, N, K = 256, 4096, 65536
    A = torch.zeros((M, K), dtype=torch.float16, device=DEV)
    B = torch.zeros((K, N), dtype=torch.float16, device=DEV)
    out = torch.zeros((M, N), dtype=torch.float16, device=DEV)
    plan = g.gemm_f16_get_plan(*_args(A, B, out))
    assert plan["workspace_bytes"] > g.NOALLOC_SCRATCH_BYTES, plan
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16_noalloc(*_args(A, B, out))
    assert e.value.status == g.ERR_OUT_OF_MEMORY


def test_no_alloc_gathers_unaligned_views_and_allocates_nothing():
    """An operand TMA cannot address (a transposed view whose pitch, 17
    elements, is not a multiple of 16 bytes) is gathered by this entry point
    (gemm_f16 would copy it into its workspace for a large product), and the
    tiles are cut along K, so the partial sums go to the fixed array.  Integer
    inputs make every order of the fp32 sums exact: the result must equal the
    oracle bit for bit.  Device memory in use must not change across the calls,
    which come before any gemm_f16 call of this shape."""
    torch.cuda.set_device(DEV)
    rng = np.random.default_rng(37)
    M, N, K = 16, 4096, 8192
    buf = rng.integers(-3, 4, (K, M + 1)).astype(np.float16)   # A = buf[:, :M].T, strides (1, M + 1)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A = torch.from_numpy(buf).to(DEV)[:, :M].t()
    B = torch.from_numpy(Bh).to(DEV)
    assert A.stride() == (1, M + 1)
    outs = [torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV) for _ in range(2)]
    g.gemm_f16_set_option(g.OPT_REPACK, 1)        # the plan this entry point runs
    try:
        plan = g.gemm_f16_get_plan(*_args(A, B, outs[0]))
    finally:
        g.gemm_f16_set_option(g.OPT_REPACK, 0)
    assert plan["repack"] == 0 and not (plan["a_tma"] and plan["b_tma"]), plan
    assert plan["streamk_tiles"] > 0 or plan["splits"] > 1, plan
    assert 0 < plan["workspace_bytes"] <= g.NOALLOC_SCRATCH_BYTES, plan
    stream = torch.cuda.current_stream(DEV).cuda_stream
    # warm-up on another shape that also cuts tiles along K: loads the module
    # and looks up the array's address, which are set-up, not allocations
    g.gemm_f16_noalloc(*_args(A[:, :4096], B[:4096, :2048], outs[1][:, :2048]), stream=stream)
    torch.cuda.synchronize(DEV)
    free0 = torch.cuda.mem_get_info(DEV)[0]
    for out in outs:                              # two calls in a row on the shared array
        g.gemm_f16_noalloc(*_args(A, B, out), stream=stream)
    torch.cuda.synchronize(DEV)
    assert torch.cuda.mem_get_info(DEV)[0] == free0
    ref = oracle.gemm(A.cpu().numpy(), Bh, threads=oracle_threads())
    for call, out in enumerate(outs):
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), f"noalloc call {call} vs oracle"
    assert g.gemm_f16_device_status() == 0


def test_no_alloc_with_the_default_k_segments():
    """A swapped small-M pair plan that takes K segments by default (16 x
    16384 x 1024: 64 pair tiles, 2 segments) keeps its partials in the fixed
    array: bit for bit against gemm_f16 and the oracle on integers."""
    torch.cuda.set_device(DEV)
    rng = np.random.default_rng(37)
    M, N, K = 16, 16384, 1024
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A = torch.from_numpy(Ah).to(DEV)
    B = torch.from_numpy(Bh).to(DEV)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    plan = g.gemm_f16_get_plan(*_args(A, B, out))
    assert plan["splits"] == 2 and plan["pair"] and plan["swap_ab"], plan
    assert 0 < plan["workspace_bytes"] <= g.NOALLOC_SCRATCH_BYTES, plan
    stream = torch.cuda.current_stream(DEV).cuda_stream
    g.gemm_f16_noalloc(*_args(A, B, out), stream=stream)
    torch.cuda.synchronize(DEV)
    got = out.cpu().numpy()
    ref = oracle.gemm(Ah, Bh, threads=oracle_threads())
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    out2 = torch.empty_like(out)
    g.gemm_f16(*_args(A, B, out2), stream=stream)
    torch.cuda.synchronize(DEV)
    assert np.array_equal(out2.cpu().numpy().view(np.uint16), got.view(np.uint16))
    assert g.gemm_f16_device_status() == 0
