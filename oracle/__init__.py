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

``gemm_fused`` (with its grouped and batched forms) adds the fused output
stage: bias, activation and the gate/up product, evaluated in double on the
unrounded sums from ``gemm_exact`` and rounded once.

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
            lib.oracle_gemm_f64.argtypes = [P, I64, I64, P, I64, I64, P, I64, I64, I64, I64,
                                            ctypes.c_int]
            lib.oracle_gemm_f64.restype = None
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


def gemm_exact(A: np.ndarray, B: np.ndarray, threads: int = 1) -> np.ndarray:
    """The unrounded double sums of ``gemm``: S = A @ B as float64 [M, N]."""
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shape mismatch")
    M, K = A.shape
    N = B.shape[1]
    a_base, (s_am, s_ak) = _base_of(_u16(A))
    b_base, (s_bk, s_bn) = _base_of(_u16(B))
    S = np.zeros((M, N), dtype=np.float64)
    _load().oracle_gemm_f64(a_base, s_am, s_ak, b_base, s_bk, s_bn, S.ctypes.data, N, M, N, K, int(threads))
    return S


# ---------------------------------------------------------------- fused epilogue
# The pages name the fusions without fixing their arithmetic: the TileLang
# tutorial's comparison checklist (ch. 14, section 6.3, item 4) and the AI-infra
# page's section 05 list bias and activation fused into the GEMM's output stage;
# the C500 review (section 17.3) lists a gate/up GEMM that fuses the two
# projections and one that adds the activation and the multiply.  Read plainly:
#   out = act(A @ B + bias)                                 (bias broadcast along rows)
#   out = act(A @ B_gate + bias_gate) * (A @ B_up + bias_up)  (gate/up)
# with act one of identity, ReLU, SiLU (x * logistic(x)) and GELU in its exact
# form x * Phi(x) (Phi the standard normal CDF).  All of it is evaluated here in
# double on the unrounded sums and rounded to fp16 once.
ACTIVATIONS = ("none", "relu", "silu", "gelu")


def _erfc(x: np.ndarray) -> np.ndarray:
    import math

    return np.vectorize(math.erfc, otypes=[np.float64])(x)


def activation(x, act: str) -> np.ndarray:
    """act(x) in double.  relu(x) = 0 for x < 0 and x otherwise; silu(x) =
    x / (1 + exp(-x)); gelu(x) = x * Phi(x) with Phi(x) = erfc(-x / sqrt(2)) / 2,
    the same as x/2 * (1 + erf(x / sqrt(2))) but without the cancellation in
    the far negative tail."""
    x = np.asarray(x, dtype=np.float64)
    if act == "none":
        return x.copy()
    if act == "relu":
        return np.where(x < 0, 0.0, x)
    if act == "silu":
        with np.errstate(over="ignore"):
            return x / (1.0 + np.exp(-x))
    if act == "gelu":
        return x * (0.5 * _erfc(-x / np.sqrt(2.0)))
    raise ValueError(f"unknown activation {act!r}")


def _bias_row(bias, N):
    if bias is None:
        return np.zeros(N, dtype=np.float64)
    b = half_to_double(np.ascontiguousarray(np.asarray(bias, dtype=np.float16)))
    if b.shape != (N,):
        raise ValueError("bias must hold N values")
    return b


def epilogue(S, act: str = "none", bias=0.0, S_up=None, bias_up=0.0):
    """The fused output stage on double sums: fp16 act(S + bias), or with the
    up sums ``S_up`` fp16 act(S + bias) * (S_up + bias_up); bias values in
    double, broadcast against S.  Returns (C, g, u): the fp16 result, the
    pre-activation gate g = S + bias and u = S_up + bias_up (None without)."""
    if act not in ACTIVATIONS:
        raise ValueError(f"unknown activation {act!r}")
    g = np.asarray(S, dtype=np.float64) + bias
    out = activation(g, act)
    u = None
    if S_up is not None:
        u = np.asarray(S_up, dtype=np.float64) + bias_up
        out = out * u
    return double_to_half(out), g, u


def gemm_fused(A: np.ndarray, B: np.ndarray, B_up: np.ndarray | None = None, bias=None, bias_up=None,
               act: str = "none", threads: int = 1, parts: bool = False):
    """fp16 act(A @ B + bias), or with ``B_up`` the gate/up form
    act(A @ B + bias) * (A @ B_up + bias_up); one rounding to fp16 at the end.

    With ``parts`` also returns the double pre-activation gate g = A @ B + bias
    and up u = A @ B_up + bias_up (None without B_up), for error bounds.
    """
    if act not in ACTIVATIONS:
        raise ValueError(f"unknown activation {act!r}")
    if bias_up is not None and B_up is None:
        raise ValueError("bias_up needs B_up")
    N = B.shape[1]
    S_up = None
    if B_up is not None:
        if B_up.shape != B.shape:
            raise ValueError("B_up must have B's shape")
        S_up = gemm_exact(A, B_up, threads)
    C, g, u = epilogue(gemm_exact(A, B, threads), act, _bias_row(bias, N)[None, :], S_up,
                       _bias_row(bias_up, N)[None, :])
    return (C, g, u) if parts else C


def gemm_fused_grouped(A: np.ndarray, B: np.ndarray, group_rows, B_up=None, bias=None, bias_up=None,
                       act: str = "none", threads: int = 1, parts: bool = False):
    """``gemm_fused`` per group of a grouped problem (see ``gemm_grouped``):
    group g uses B[g], B_up[g] and the bias rows bias[g], bias_up[g] ([G, N]);
    a bias of shape [N] is shared by every group."""
    G, K, N = B.shape
    if sum(int(r) for r in group_rows) != A.shape[0] or len(group_rows) != G:
        raise ValueError("group rows do not match")
    C = np.zeros((A.shape[0], N), dtype=np.float16)
    gs = np.zeros((A.shape[0], N))
    us = np.zeros((A.shape[0], N)) if B_up is not None else None

    def pick(b, g):
        if b is None:
            return None
        b = np.asarray(b)
        return b[g] if b.ndim == 2 else b

    r0 = 0
    for g, rows in enumerate(int(r) for r in group_rows):
        if rows:
            c, gg, uu = gemm_fused(A[r0:r0 + rows], B[g], None if B_up is None else B_up[g], pick(bias, g),
                                   pick(bias_up, g), act, threads, parts=True)
            C[r0:r0 + rows] = c
            gs[r0:r0 + rows] = gg
            if us is not None:
                us[r0:r0 + rows] = uu
        r0 += rows
    return (C, gs, us) if parts else C


def gemm_fused_batched(A: np.ndarray, B: np.ndarray, B_up=None, bias=None, bias_up=None, act: str = "none",
                       threads: int = 1, parts: bool = False):
    """``gemm_fused`` per problem of a batch ([batch, M, K] @ [batch, K, N]); a
    bias [batch, N] per problem or [N] shared."""
    nb, M, _ = A.shape
    N = B.shape[2]
    C = np.zeros((nb, M, N), dtype=np.float16)
    gs = np.zeros((nb, M, N))
    us = np.zeros((nb, M, N)) if B_up is not None else None
    for b in range(nb):
        pb = None if bias is None else (np.asarray(bias)[b] if np.ndim(bias) == 2 else bias)
        pu = None if bias_up is None else (np.asarray(bias_up)[b] if np.ndim(bias_up) == 2 else bias_up)
        c, gg, uu = gemm_fused(A[b], B[b], None if B_up is None else B_up[b], pb, pu, act, threads, parts=True)
        C[b] = c
        gs[b] = gg
        if us is not None:
            us[b] = uu
    return (C, gs, us) if parts else C


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
