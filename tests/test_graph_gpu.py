"""The C-ABI calls inside CUDA graph capture: after a first call has set up
the device (attributes, workspace), a call only validates on the host and
enqueues kernels (and, with a caller workspace, a memset) on the given stream,
so it can be captured and replayed."""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from tests.parity import assert_bits, assert_close, oracle_threads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _defaults():
    yield
    for o in (g.OPT_STREAMK, g.OPT_REPACK):
        g.gemm_f16_set_option(o, 0)


@pytest.mark.parametrize("M,N,K,opts", [(16, 4096, 2048, {}),                   # swapped, small M
                                        (1000, 768, 512, {}),                   # pair tiles
                                        (600, 640, 1024, {g.OPT_STREAMK: 2}),  # stream-K fixup
                                        (3001, 700, 640, {g.OPT_REPACK: 2})])  # aligned copy + GEMM
def test_captured_call_replays_correctly(M, N, K, opts):
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    rng = np.random.default_rng(M + N + K)
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    if opts.get(g.OPT_REPACK):
        buf = torch.zeros((M, K + 3), dtype=torch.float16, device=DEV)   # unaligned pitch
        A = buf[:, :K]
        A.copy_(torch.from_numpy(Ah).to(DEV))
    else:
        A = torch.from_numpy(Ah).to(DEV)
    B = torch.from_numpy(Bh).to(DEV)
    C = torch.zeros((M, N), dtype=torch.float16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.matmul(A, B, out=C, stream=s)      # first call: device set-up, workspace growth
    torch.cuda.synchronize()
    C.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.matmul(A, B, out=C, stream=s)
    torch.cuda.synchronize()
    assert float(C.float().abs().sum()) == 0.0   # capturing ran nothing
    ref = oracle.gemm(Ah, Bh, threads=oracle_threads())
    for _ in range(3):
        C.zero_()
        graph.replay()
        torch.cuda.synchronize()
        if K * 9 <= 2048:
            assert_bits(C.cpu().numpy(), ref, "graph replay")
        else:
            assert_close(C.cpu().numpy(), ref, K, "graph replay")
    assert g.gemm_f16_device_status() == 0
