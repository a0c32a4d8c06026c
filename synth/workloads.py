"""The GEMM workloads used by the tests and the bench: shapes, layouts, seeds.

Pure data plus helpers that materialise operands from :mod:`synth`; nothing
here performs any part of the matrix product.

Each operand is a logical ``rows x cols`` matrix that is either a row-major
buffer of that shape, or the transposed view of a row-major ``cols x rows``
buffer (strides ``(1, rows_of_view)``), which is how the Triton GEMM page's
``B = X.T`` example describes a transposed operand.  The generator fills the
*buffer*; the logical operand is the view.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import buffer_np, buffer_torch, values_np


@dataclass(frozen=True)
class Operand:
    rows: int
    cols: int
    kind: str
    seed: int
    transposed: bool = False  # logical = (row-major cols x rows buffer).T

    @property
    def buf_shape(self):
        return (self.cols, self.rows) if self.transposed else (self.rows, self.cols)

    @property
    def numel(self) -> int:
        return self.rows * self.cols

    @property
    def strides(self):
        """Element strides of the logical view over its buffer."""
        return (1, self.rows) if self.transposed else (self.cols, 1)

    def flat_index(self, r, c):
        """Flat buffer index of logical element (r, c) (numpy broadcasting)."""
        s0, s1 = self.strides
        return np.asarray(r, dtype=np.int64) * s0 + np.asarray(c, dtype=np.int64) * s1

    def host_buffer(self) -> np.ndarray:
        return buffer_np(self.kind, self.seed, self.numel)

    def host_view(self) -> np.ndarray:
        """Logical matrix as a (possibly non-contiguous) numpy float16 view."""
        buf = self.host_buffer().reshape(self.buf_shape)
        return buf.T if self.transposed else buf

    def device_view(self, device):
        """Logical matrix as a torch float16 view over a generator-filled buffer."""
        buf = buffer_torch(self.kind, self.seed, self.numel, device).view(*self.buf_shape)
        return buf.t() if self.transposed else buf

    def values_at(self, r, c) -> np.ndarray:
        return values_np(self.kind, self.seed, self.flat_index(r, c).astype(np.uint64))


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    A: Operand
    B: Operand
    description: str = ""
    bit_exact: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


def _op(rows, cols, kind, seed, transposed=False):
    return Operand(rows, cols, kind, seed, transposed)


# The five configurations: a ragged tail case, a square compute-bound case, a
# decode-like small-M case, an irregular strided case and the MoE-flattened case.
TAIL_ROWMAJOR_B = Workload(
    "tail_130x70x65_b_rowmajor", 130, 70, 65,
    _op(130, 65, "int3", 1), _op(65, 70, "int3", 10),
    "ragged tail shape, integers in [-3,3] (exact in fp32), B row-major [65,70]",
    bit_exact=True)
TAIL_TRANSPOSED_B = Workload(
    "tail_130x70x65_b_transposed", 130, 70, 65,
    _op(130, 65, "int3", 1), _op(65, 70, "int3", 11, transposed=True),
    "ragged tail shape, integers in [-3,3], B a view of row-major [70,65], strides (1,65)",
    bit_exact=True)
SQUARE_4096 = Workload(
    "square_4096", 4096, 4096, 4096,
    _op(4096, 4096, "uniform", 2), _op(4096, 4096, "uniform", 3),
    "square compute-bound, contiguous row-major, uniform[-1,1] in fp16")
DECODE_16x16384x8192 = Workload(
    "decode_m16_n16384_k8192", 16, 16384, 8192,
    _op(16, 8192, "uniform", 4), _op(8192, 16384, "uniform", 5),
    "decode-like small M: activations [16,8192] x weights [8192,16384]")
IRREGULAR_3001x1999x4097 = Workload(
    "irregular_3001x1999x4097_at", 3001, 1999, 4097,
    _op(3001, 4097, "uniform", 6, transposed=True), _op(4097, 1999, "uniform", 7),
    "irregular, A a view of row-major [4097,3001] with strides (1,3001), B row-major")
MOE_131072x2048x7168 = Workload(
    "moe_131072x2048x7168", 131072, 2048, 7168,
    _op(131072, 7168, "uniform", 8), _op(7168, 2048, "uniform", 9),
    "MoE-flattened (4 x 8192 tokens x top-4) [131072,7168] x [7168,2048]")

ALL = [TAIL_ROWMAJOR_B, TAIL_TRANSPOSED_B, SQUARE_4096, DECODE_16x16384x8192,
       IRREGULAR_3001x1999x4097, MOE_131072x2048x7168]
BY_NAME = {w.name: w for w in ALL}


# ------------------------------------------------ several problems per launch
def group_rows_for(total: int, groups: int, seed: int) -> tuple:
    """Synthetic per-expert row counts standing in for routing: expert g gets a
    share proportional to 1.5 + v_g (v_g a seeded uniform[-1,1) draw, so shares
    differ by up to 5x); the rounding remainder goes to the last expert."""
    v = values_np("uniform", seed, np.arange(groups, dtype=np.uint64)).astype(np.float64)
    w = 1.5 + v
    rows = [int(total * x / w.sum()) for x in w[:-1]]
    rows.append(total - sum(rows))
    return tuple(rows)


@dataclass(frozen=True)
class MultiWorkload:
    """Several problems in one launch.  kind "batched": `count` problems of
    M x N x K, A stacked as count*M rows of K, B as count*K rows of N.  kind
    "grouped": `count` groups sharing N and K, A the M = sum(group_rows) rows,
    B stacked as count*K rows of N (group g's B in rows g*K ..)."""
    name: str
    kind: str
    M: int
    N: int
    K: int
    count: int
    A: Operand
    B: Operand
    description: str = ""
    group_rows: tuple = ()
    # fused output stage: a second (up) projection stacked like B, and the activation
    B_up: Operand | None = None
    act: str = "none"

    @property
    def flops(self) -> float:
        problems = self.count if self.kind == "batched" else 1
        products = 2 if self.B_up is not None else 1
        return 2.0 * problems * products * self.M * self.N * self.K

    @property
    def c_rows(self) -> int:
        return self.count * self.M if self.kind == "batched" else self.M

    def first_problem(self) -> Workload:
        """Problem (or group) 0 as a one-GEMM workload over the same values: the
        stacked operands' first rows are the first problem's."""
        m0 = self.M if self.kind == "batched" else self.group_rows[0]
        return Workload(self.name + "[0]", m0, self.N, self.K, _op(m0, self.K, self.A.kind, self.A.seed),
                        _op(self.K, self.N, self.B.kind, self.B.seed), "first problem")

    def first_up(self):
        """Problem 0's up projection (K x N operand), or None."""
        if self.B_up is None:
            return None
        return _op(self.K, self.N, self.B_up.kind, self.B_up.seed)


BATCHED_32x1024 = MultiWorkload(
    "batched_32x1024x1024x1024", "batched", 1024, 1024, 1024, 32,
    _op(32 * 1024, 1024, "uniform", 12), _op(32 * 1024, 1024, "uniform", 13),
    "batched: 32 problems of 1024^3, contiguous row-major")
GROUPED_MOE = MultiWorkload(
    "grouped_moe_g8_131072x2048x7168", "grouped", 131072, 2048, 7168, 8,
    _op(131072, 7168, "uniform", 14), _op(8 * 7168, 2048, "uniform", 15),
    "grouped MoE layer: 131072 routed rows over 8 experts (seeded shares), each expert's [7168,2048] B",
    group_rows_for(131072, 8, 16))

GROUPED_GATEUP_SILU = MultiWorkload(
    "grouped_gateup_silu_g8_131072x2048x7168", "grouped", 131072, 2048, 7168, 8,
    _op(131072, 7168, "uniform", 14), _op(8 * 7168, 2048, "uniform", 15),
    "MoE gate/up layer: the routed rows of the grouped MoE workload through 8 experts' gate and up "
    "projections [7168,2048] each, out = silu(A Bg) * (A Bu)",
    group_rows_for(131072, 8, 16), B_up=_op(8 * 7168, 2048, "uniform", 17), act="silu")

MULTI = [BATCHED_32x1024, GROUPED_MOE, GROUPED_GATEUP_SILU]
BY_NAME.update({w.name: w for w in MULTI})
