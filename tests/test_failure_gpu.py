"""Failure detection without a GPU fault: every pipeline wait in the kernel is
bounded.  With GEMM_F16_OPT_TEST_STALL the MMA issuer first waits on a barrier
that nothing arrives on; the wait runs out after GEMM_F16_OPT_TIMEOUT_MS, the
CTA raises its abort flag, every other wait gives up, in-flight copies are
drained, TMEM is freed and the kernel returns.  The host then reads
GEMM_F16_ERR_TIMEOUT from the device status word, and the same context runs
the next call correctly.
"""
import numpy as np
import pytest
import torch

import dense_tiled_gemm_fp16_gb300 as g
import oracle
from tests.parity import assert_bits

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _defaults():
    g.gemm_f16_device_status(reset=True)
    yield
    for o in (g.OPT_FORCE_GATHER, g.OPT_SPLITS, g.OPT_TILE_N, g.OPT_PANEL, g.OPT_SWAP,
              g.OPT_TIMEOUT_MS, g.OPT_MAX_CTAS, g.OPT_PAIR, g.OPT_STREAMK, g.OPT_TAIL_SPLIT, g.OPT_MAX_STAGES,
              g.OPT_REPACK, g.OPT_TEST_STALL):
        g.gemm_f16_set_option(o, 0)
    g.gemm_f16_device_status(reset=True)


FORMS = [
    ("single", {g.OPT_PAIR: 1}),
    ("pair", {}),
    ("gathered", {g.OPT_FORCE_GATHER: 3}),
    ("split_k", {g.OPT_SPLITS: 2, g.OPT_PAIR: 1}),
]


@pytest.mark.parametrize("form", FORMS, ids=lambda f: f[0])
def test_stalled_wait_reports_timeout_and_the_context_survives(form):
    name, opts = form
    rng = np.random.default_rng(90)
    M, N, K = 512, 512, 256
    Ah = rng.integers(-3, 4, (M, K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (K, N)).astype(np.float16)
    A, B = torch.from_numpy(Ah).to(DEV), torch.from_numpy(Bh).to(DEV)
    C = torch.zeros((M, N), dtype=torch.float16, device=DEV)
    for o, v in opts.items():
        g.gemm_f16_set_option(o, v)
    g.gemm_f16_set_option(g.OPT_TIMEOUT_MS, 50)
    g.gemm_f16_set_option(g.OPT_TEST_STALL, 1)
    g.matmul(A, B, out=C)                        # queued: the kernel gives up on its own
    assert g.gemm_f16_device_status(reset=True) == g.ERR_TIMEOUT, name
    g.gemm_f16_set_option(g.OPT_TEST_STALL, 0)
    g.gemm_f16_set_option(g.OPT_TIMEOUT_MS, 0)
    g.matmul(A, B, out=C)
    torch.cuda.synchronize()
    assert_bits(C.cpu().numpy(), oracle.gemm(Ah, Bh), f"after the timeout ({name})")
    assert g.gemm_f16_device_status() == 0


def test_stalled_fused_grouped_call_times_out_cleanly():
    rng = np.random.default_rng(91)
    rows, N, K = [300, 0, 500], 256, 128
    Ah = rng.integers(-3, 4, (sum(rows), K)).astype(np.float16)
    Bh = rng.integers(-3, 4, (3, K, N)).astype(np.float16)
    Uh = rng.integers(-3, 4, (3, K, N)).astype(np.float16)
    A, B, U = (torch.from_numpy(x).to(DEV) for x in (Ah, Bh, Uh))
    g.gemm_f16_set_option(g.OPT_TIMEOUT_MS, 50)
    g.gemm_f16_set_option(g.OPT_TEST_STALL, 1)
    g.grouped_fused_mm(A, B, rows, act="relu", b_up=U)
    assert g.gemm_f16_device_status(reset=True) == g.ERR_TIMEOUT
    g.gemm_f16_set_option(g.OPT_TEST_STALL, 0)
    g.gemm_f16_set_option(g.OPT_TIMEOUT_MS, 0)
    C = g.grouped_fused_mm(A, B, rows, act="relu", b_up=U)
    torch.cuda.synchronize()
    assert_bits(C.cpu().numpy(), oracle.gemm_fused_grouped(Ah, Bh, rows, Uh, act="relu"), "fused after timeout")
    assert g.gemm_f16_device_status() == 0
