"""The GEMM cost ledger: useful FLOPs, minimum traffic, intensity and roofline.

Follows the TileLang tutorial ch. 14 "GEMM operators", section 1.1 (2MNK FLOP;
minimum DRAM traffic b(MK+KN+MN) with A and B read once and C written once;
arithmetic intensity their ratio) and the AI-infra knowledge base page "Matrix
multiplication and memory-access optimisation", section 04 (the same ideal
ledger with b = 2 bytes).  Throughput is always quoted on the useful 2MNK, never
on padded block work (Triton GEMM page, the closing timing paragraph).
"""
from __future__ import annotations


def flops(M: int, N: int, K: int) -> float:
    """Useful floating-point operations of C = A*B: one multiply and one add per term."""
    return 2.0 * M * N * K


def min_bytes(M: int, N: int, K: int, elem_bytes: int = 2) -> float:
    """Minimum DRAM traffic: read A and B once, write C once."""
    return float(elem_bytes) * (M * K + K * N + M * N)


def intensity(M: int, N: int, K: int, elem_bytes: int = 2) -> float:
    """Arithmetic intensity in FLOP per byte of minimum traffic."""
    return flops(M, N, K) / min_bytes(M, N, K, elem_bytes)


def roofline_tflops(M: int, N: int, K: int, peak_tflops: float, hbm_gbs: float,
                    elem_bytes: int = 2) -> float:
    """Attainable TFLOP/s: min(tensor peak, intensity * bandwidth)."""
    return min(peak_tflops, intensity(M, N, K, elem_bytes) * hbm_gbs / 1e3)


def bound(M: int, N: int, K: int, peak_tflops: float, hbm_gbs: float,
          elem_bytes: int = 2) -> str:
    """'tensor' if the tensor-core peak is the lower ceiling, else 'hbm'."""
    return "tensor" if intensity(M, N, K, elem_bytes) * hbm_gbs / 1e3 >= peak_tflops else "hbm"


def stage_bytes(BM: int, BN: int, BK: int, elem_bytes: int = 2) -> int:
    """Shared memory of one pipeline stage: an A block plus a B block."""
    return (BM * BK + BK * BN) * elem_bytes


def stage_intensity(BM: int, BN: int, elem_bytes: int = 2) -> float:
    """Per-round intensity of one output block, FLOP per loaded byte.

    One round loads elem_bytes*BK*(BM+BN) bytes and does 2*BM*BN*BK FLOP, so BK
    cancels (Triton GEMM page, section "Bigger tiles bring reuse and heavier
    accumulators").
    """
    return 2.0 * BM * BN / (elem_bytes * (BM + BN))


def accumulator_bytes(BM: int, BN: int) -> int:
    """Logical size of one fp32 output-block accumulator."""
    return 4 * BM * BN
