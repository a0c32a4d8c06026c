"""CPU oracle for C = A*B (fp16 in, double accumulation, fp16 out) — TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg use
this package.  The GPU library never imports, links or calls it, and this
package never imports the GPU library.

The arithmetic lives in ``gemm_oracle.c`` (a plain strided triple loop, see its
header for the passages it follows); this module only compiles it with the
host C compiler and marshals numpy arrays into it.  ``tiled.py`` holds a
pure-Python restatement of the output-tiled loop used to pin the pages' worked
examples (logical read counts, the ragged-tail program counts, the K-tail
counter-example).

Every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_gemm.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, OpenMP over output rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_double_to_half.argtypes = [ctypes.c_double]
            lib.oracle_double_to_half.restype = ctypes.c_uint16
            lib.oracle_gemm_f16.argtypes = [P, I64, I64, P, I64, I64, P, I64, I64, I64, I64,
                                            ctypes.c_int]
            lib.oracle_gemm_f16.restype = None
            lib.oracle_dot_f16.argtypes = [P, P, I64, P, P, I64, I64, I64, P, P, ctypes.c_int]
            lib.oracle_dot_f16.restype = None
            lib.oracle_half_to_double_n.argtypes = [P, P, I64]
            lib.oracle_double_to_half_n.argtypes = [P, P, I64]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_init()
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _u16(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("expected float16 or uint16 bits")
    return a


def half_to_double(bits) -> np.ndarray:
    h = np.ascontiguousarray(_u16(np.asarray(bits)))
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_half_to_double_n(h.ctypes.data, out.ctypes.data, h.size)
    return out


def double_to_half(x) -> np.ndarray:
    """double -> fp16, returned as float16 (bits via ``.view(np.uint16)``)."""
    d = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(d.shape, dtype=np.uint16)
    _load().oracle_double_to_half_n(d.ctypes.data, out.ctypes.data, d.size)
    return out.view(np.float16)


def gemm_strided(A_buf: np.ndarray, a_off: int, s_am: int, s_ak: int,
                 B_buf: np.ndarray, b_off: int, s_bk: int, s_bn: int,
                 M: int, N: int, K: int, C_buf: np.ndarray | None = None,
                 c_off: int = 0, ldc: int | None = None, threads: int = 1) -> np.ndarray:
    """The oracle on raw flat buffers and element strides (the library's contract).

    ``A_buf``/``B_buf`` are flat fp16 buffers; element (m,k) of A is
    ``A_buf[a_off + m*s_am + k*s_ak]``, likewise for B.  Writes C[m*ldc+n] of the
    flat ``C_buf`` (allocated as M*N if not given) and returns it.
    """
    A_buf = np.ascontiguousarray(_u16(A_buf)).reshape(-1)
    B_buf = np.ascontiguousarray(_u16(B_buf)).reshape(-1)
    if ldc is None:
        ldc = N
    if C_buf is None:
        C_buf = np.zeros(c_off + (M - 1) * ldc + N, dtype=np.uint16)
    Cu = _u16(C_buf)
    if not Cu.flags.c_contiguous:
        raise ValueError("C_buf must be contiguous")
    # The caller's view must lie inside the buffers.
    last_a = a_off + (M - 1) * s_am + (K - 1) * s_ak
    last_b = b_off + (K - 1) * s_bk + (N - 1) * s_bn
    last_c = c_off + (M - 1) * ldc + (N - 1)
    if min(a_off, b_off, c_off) < 0 or last_a >= A_buf.size or last_b >= B_buf.size \
            or last_c >= Cu.size:
        raise ValueError("view exceeds its buffer")
    _load().oracle_gemm_f16(A_buf.ctypes.data + 2 * a_off, s_am, s_ak,
                            B_buf.ctypes.data + 2 * b_off, s_bk, s_bn,
                            Cu.ctypes.data + 2 * c_off, ldc, M, N, K, int(threads))
    return C_buf


def gemm(A: np.ndarray, B: np.ndarray, threads: int = 1) -> np.ndarray:
    """C = A @ B for 2-D float16 numpy views (any strides); returns float16 [M,N]."""
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shape mismatch")
    M, K = A.shape
    N = B.shape[1]
    Au, Bu = _u16(A), _u16(B)
    a_base, (s_am, s_ak) = _base_of(Au)
    b_base, (s_bk, s_bn) = _base_of(Bu)
    C = np.zeros((M, N), dtype=np.uint16)
    _load().oracle_gemm_f16(a_base, s_am, s_ak, b_base, s_bk, s_bn,
                            C.ctypes.data, N, M, N, K, int(threads))
    return C.view(np.float16)


def gemm_batched(A: np.ndarray, B: np.ndarray, threads: int = 1) -> np.ndarray:
    """Batched GEMM, C[b] = A[b] @ B[b] for 3-D float16 views [batch, M, K] and
    [batch, K, N] (any strides, a batch stride of 0 included).

    TileLang tutorial ch. 14 "GEMM operators", section 4.4 (batched GEMM: the
    same GEMM on every batch index).  Each problem is ``gemm`` as it stands.
    """
    if A.ndim != 3 or B.ndim != 3 or A.shape[0] != B.shape[0] or A.shape[2] != B.shape[1]:
        raise ValueError("shape mismatch")
    C = np.zeros((A.shape[0], A.shape[1], B.shape[2]), dtype=np.float16)
    for b in range(A.shape[0]):
        C[b] = gemm(A[b], B[b], threads)
    return C


def gemm_grouped(A: np.ndarray, B: np.ndarray, group_rows, threads: int = 1) -> np.ndarray:
    """Grouped GEMM: the rows of A [sum(group_rows), K] form consecutive groups and
    group g's rows are multiplied by B[g] ([G, K, N]); returns C [sum, N].

    TileLang tutorial ch. 14 "GEMM operators", section 4.3 (grouped GEMM: G
    GEMMs sharing K and N, the experts' rows concatenated and located through
    an offset table).  Each group is ``gemm`` as it stands; empty groups give
    no rows.
    """
    if A.ndim != 2 or B.ndim != 3 or B.shape[0] != len(group_rows) or A.shape[1] != B.shape[1]:
        raise ValueError("shape mismatch")
    if sum(int(r) for r in group_rows) != A.shape[0]:
        raise ValueError("group rows do not add up to A's rows")
    C = np.zeros((A.shape[0], B.shape[2]), dtype=np.float16)
    r0 = 0
    for g, rows in enumerate(int(r) for r in group_rows):
        if rows:
            C[r0:r0 + rows] = gemm(A[r0:r0 + rows], B[g], threads)
        r0 += rows
    return C


def _base_of(v: np.ndarray):
    item = v.itemsize
    if any(s % item for s in v.strides) or any(s <= 0 for s in v.strides):
        raise ValueError("the oracle takes positive element strides")
    return v.__array_interface__["data"][0], tuple(s // item for s in v.strides)


def dots(A_rows: np.ndarray, a_off, s_ak: int, B_cols: np.ndarray, b_off, s_bk: int,
         K: int, threads: int = 1):
    """Sampled outputs: fp16 and double sums of K-long strided dot products.

    ``A_rows``/``B_cols`` are flat fp16 buffers; sample i uses
    ``A_rows[a_off[i] + k*s_ak]`` and ``B_cols[b_off[i] + k*s_bk]``.
    Returns (float16 results, float64 unrounded sums).
    """
    Au = np.ascontiguousarray(_u16(A_rows)).reshape(-1)
    Bu = np.ascontiguousarray(_u16(B_cols)).reshape(-1)
    ao = np.ascontiguousarray(np.asarray(a_off, dtype=np.int64))
    bo = np.ascontiguousarray(np.asarray(b_off, dtype=np.int64))
    if ao.shape != bo.shape:
        raise ValueError("offset arrays differ in length")
    if ao.size and (ao.min() < 0 or bo.min() < 0
                    or ao.max() + (K - 1) * s_ak >= Au.size
                    or bo.max() + (K - 1) * s_bk >= Bu.size):
        raise ValueError("sample exceeds its buffer")
    out = np.empty(ao.size, dtype=np.uint16)
    exact = np.empty(ao.size, dtype=np.float64)
    _load().oracle_dot_f16(Au.ctypes.data, ao.ctypes.data, s_ak, Bu.ctypes.data, bo.ctypes.data,
                           s_bk, K, ao.size, out.ctypes.data, exact.ctypes.data, int(threads))
    return out.view(np.float16), exact
