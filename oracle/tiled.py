"""Output-tiled restatement of C = A*B with logical-read accounting — TEST INFRASTRUCTURE.

This is not a faster oracle.  It re-states the blocked algorithm that the pages
walk through, so that their worked examples can be checked against it and it,
in turn, against the plain oracle:

* one program owns a BM x BN output block and walks K in rounds of BK, loading
  an A block and a B block per round and accumulating their product; masked
  positions (row >= M, k >= K, col >= N) load zero; the store writes only
  row < M and col < N ("Triton GEMM: from one output tile to addresses,
  boundaries and data reuse", sections "Why the output dims are parallelised
  and K stays in the accumulator" and "Three non-divisible dimensions need
  different boundary handling");
* each input element fetched into a block counts as one logical read, with no
  cache model ("Matrix multiplication and memory-access optimisation",
  sections 02 and 03: 128 reads untiled, 64 with 2x2 blocks, 32 whole);
* ``k_wrap_modulo=True`` replaces the K zero-fill by index wrap-around modulo K,
  the counter-example the Triton page gives (it turns 32 into 36); it exists
  only so that a test can show the wrong variant fails.

The per-round block product uses numpy float64 matmul as a library step; for
integer-valued inputs every sum is exact.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class TiledStats:
    programs: int = 0
    rounds_per_program: int = 0
    logical_reads: int = 0          # masked-in element loads of A and B
    masked_lanes: int = 0           # block positions that loaded the fill value
    block_flops: int = 0            # 2*BM*BN*BK per program-round (regular blocks)
    writes: np.ndarray = field(default=None)  # per-output write counts


def tiled_gemm(A: np.ndarray, B: np.ndarray, BM: int, BN: int, BK: int,
               k_wrap_modulo: bool = False):
    """Return (C as float64 [M,N] exact block sums, TiledStats).

    A and B are 2-D arrays of exact values (ints or floats).
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    gm = -(-M // BM)
    gn = -(-N // BN)
    rounds = -(-K // BK)
    st = TiledStats(programs=gm * gn, rounds_per_program=rounds,
                    writes=np.zeros((M, N), dtype=np.int64))
    C = np.full((M, N), np.nan)
    for p in range(gm * gn):
        pm, pn = divmod(p, gn)           # row-major program numbering
        rm = pm * BM + np.arange(BM)
        rn = pn * BN + np.arange(BN)
        acc = np.zeros((BM, BN))
        rk = np.arange(BK)
        for _ in range(rounds):
            if k_wrap_modulo:
                kk = rk % K
                a_mask = (rm[:, None] < M) & np.ones((1, BK), bool)
                b_mask = np.ones((BK, 1), bool) & (rn[None, :] < N)
            else:
                kk = rk
                a_mask = (rm[:, None] < M) & (rk[None, :] < K)
                b_mask = (rk[:, None] < K) & (rn[None, :] < N)
            a_blk = np.zeros((BM, BK))
            b_blk = np.zeros((BK, BN))
            ai, ak = np.nonzero(a_mask)
            a_blk[ai, ak] = A[rm[ai], kk[ak]]
            bk, bn = np.nonzero(b_mask)
            b_blk[bk, bn] = B[kk[bk], rn[bn]]
            st.logical_reads += int(a_mask.sum() + b_mask.sum())
            st.masked_lanes += int(a_mask.size - a_mask.sum() + b_mask.size - b_mask.sum())
            st.block_flops += 2 * BM * BN * BK
            acc += a_blk @ b_blk
            rk = rk + BK
        out_mask = (rm[:, None] < M) & (rn[None, :] < N)
        oi, on = np.nonzero(out_mask)
        C[rm[oi], rn[on]] = acc[oi, on]
        st.writes[rm[oi], rn[on]] += 1
    return C, st


def corner_valid(M: int, N: int, BM: int, BN: int):
    """(valid rows, valid cols) of the bottom-right program of the output grid."""
    return M - (-(-M // BM) - 1) * BM, N - (-(-N // BN) - 1) * BN


def last_round_valid_k(K: int, BK: int):
    """K indices the last round covers that are inside [0, K)."""
    start = (-(-K // BK) - 1) * BK
    return [k for k in range(start, start + BK) if k < K]
