"""GB300-native dense tiled fp16 GEMM.

Python binding of the C ABI in ``include/gemm_f16.h`` (``libgemm_f16.so``,
built in-tree by ``build.py``).  The binding only marshals arguments: every
step of the product runs in the library's sm_103a kernels.  If the library is
missing, calls raise :class:`GemmF16Error`; there is no fallback.

The ``gemm_f16*`` functions mirror the C entry points one to one (device
pointers as integers, element strides): the single product (``gemm_f16``, with
caller workspace ``gemm_f16_ws``, allocation-free ``gemm_f16_noalloc``), the
batched and grouped forms, and the fused output stage (bias, activation,
gate/up product) for each.  The torch-tensor forms read pointers, strides and
the current stream from the tensors: ``matmul``, ``bmm``, ``grouped_mm``,
``fused_mm`` (2-D or batched) and ``grouped_fused_mm``; ``plan_for`` and
``fused_plan_for`` report the execution plan.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import ledger  # noqa: F401  (pure-Python cost ledger)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgemm_f16.so")

STATUS = {
    0: "GEMM_F16_OK",
    1: "GEMM_F16_ERR_INVALID_VALUE",
    2: "GEMM_F16_ERR_ALIAS",
    3: "GEMM_F16_ERR_UNSUPPORTED_DEVICE",
    4: "GEMM_F16_ERR_OUT_OF_MEMORY",
    5: "GEMM_F16_ERR_LAUNCH",
    6: "GEMM_F16_ERR_TIMEOUT",
    7: "GEMM_F16_ERR_BOUNDS",
}
(OK, ERR_INVALID_VALUE, ERR_ALIAS, ERR_UNSUPPORTED_DEVICE, ERR_OUT_OF_MEMORY, ERR_LAUNCH, ERR_TIMEOUT,
 ERR_BOUNDS) = range(8)

# Largest M, N or K of a call (GEMM_F16_MAX_DIM: 32-bit copy coordinates).
MAX_DIM = 2**31 - 2**16

OPT_FORCE_GATHER = 1
OPT_SPLITS = 2
OPT_TILE_N = 3
OPT_PANEL = 4
OPT_SWAP = 5
OPT_TIMEOUT_MS = 6
OPT_MAX_CTAS = 7
OPT_PAIR = 8
OPT_STREAMK = 9
OPT_TAIL_SPLIT = 10
OPT_MAX_STAGES = 11
OPT_REPACK = 13
OPT_TEST_STALL = 14
OPT_PDL = 15
OPT_DEBUG_BOUNDS = 16
OPT_L2_A = 17
OPT_L2_B = 18
OPT_L2_C = 19
OPT_TWO_K_LOADS = 20

# Activations of the fused output stage (gemm_f16_fused and friends).
ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU = range(4)
ACTIVATIONS = {"none": ACT_NONE, "relu": ACT_RELU, "silu": ACT_SILU, "gelu": ACT_GELU}

# Every symbol include/gemm_f16.h declares.
EXPORTED = ("gemm_f16", "gemm_f16_ws", "gemm_f16_workspace_size", "gemm_f16_status_string",
            "gemm_f16_device_status", "gemm_f16_get_plan", "gemm_f16_set_option",
            "gemm_f16_abi_version", "gemm_f16_noalloc", "gemm_f16_batched", "gemm_f16_grouped",
            "gemm_f16_fused", "gemm_f16_batched_fused", "gemm_f16_grouped_fused", "gemm_f16_fused_get_plan")

# Most groups of one gemm_f16_grouped call.
MAX_GROUPS = 64

# Size of the fixed device scratch array behind gemm_f16_noalloc (8 MiB).
NOALLOC_SCRATCH_BYTES = 8 << 20


class GemmF16Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "swap_ab", "pair", "a_tma", "a_mn_major", "b_tma", "b_mn_major", "c_tma",
        "tile_m", "tile_n", "tiles_m", "tiles_n", "splits", "kblocks", "units", "grid",
        "stages", "streamk_tiles", "tail_split", "smem_bytes")] + [("workspace_bytes", ctypes.c_size_t)] + [
        (n, ctypes.c_int) for n in ("a_box3d", "b_box3d", "cluster_ctas", "fused", "gated", "repack", "two_k_loads")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded C library (raises GemmF16Error if it was never built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise GemmF16Error(ERR_LAUNCH, f"{LIB_PATH} is not built (run __graft_entry__.build())")
                L = ctypes.CDLL(LIB_PATH)
                P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
                L.gemm_f16.argtypes = [P, I64, I64, P, I64, I64, P, I64, I64, I64, I64, P]
                L.gemm_f16.restype = ctypes.c_int
                L.gemm_f16_ws.argtypes = [P, I64, I64, P, I64, I64, P, I64, I64, I64, I64, P, SZ, P]
                L.gemm_f16_ws.restype = ctypes.c_int
                L.gemm_f16_workspace_size.argtypes = [I64, I64, I64, ctypes.POINTER(SZ)]
                L.gemm_f16_workspace_size.restype = ctypes.c_int
                L.gemm_f16_status_string.argtypes = [ctypes.c_int]
                L.gemm_f16_status_string.restype = ctypes.c_char_p
                L.gemm_f16_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_int]
                L.gemm_f16_device_status.restype = ctypes.c_int
                L.gemm_f16_get_plan.argtypes = [P, I64, I64, P, I64, I64, P, I64, I64, I64, I64,
                                                ctypes.POINTER(Plan)]
                L.gemm_f16_get_plan.restype = ctypes.c_int
                L.gemm_f16_set_option.argtypes = [ctypes.c_int, I64]
                L.gemm_f16_set_option.restype = ctypes.c_int
                L.gemm_f16_abi_version.restype = ctypes.c_int
                L.gemm_f16_noalloc.argtypes = [P, I64, I64, P, I64, I64, P, I64, I64, I64, I64, P]
                L.gemm_f16_noalloc.restype = ctypes.c_int
                L.gemm_f16_batched.argtypes = [P, I64, I64, I64, P, I64, I64, I64, P, I64, I64, I64, I64, I64,
                                               I64, P]
                L.gemm_f16_batched.restype = ctypes.c_int
                L.gemm_f16_grouped.argtypes = [P, I64, I64, P, I64, I64, I64, P, I64, ctypes.POINTER(I64), I64,
                                               I64, I64, P]
                L.gemm_f16_grouped.restype = ctypes.c_int
                I = ctypes.c_int
                L.gemm_f16_fused.argtypes = [P, I64, I64, P, I64, I64, P, P, P, I, P, I64, I64, I64, I64, P]
                L.gemm_f16_fused.restype = ctypes.c_int
                L.gemm_f16_batched_fused.argtypes = [P, I64, I64, I64, P, I64, I64, I64, P, P, P, I64, I, P, I64,
                                                     I64, I64, I64, I64, I64, P]
                L.gemm_f16_batched_fused.restype = ctypes.c_int
                L.gemm_f16_grouped_fused.argtypes = [P, I64, I64, P, I64, I64, I64, P, P, P, I64, I, P, I64,
                                                     ctypes.POINTER(I64), I64, I64, I64, P]
                L.gemm_f16_grouped_fused.restype = ctypes.c_int
                L.gemm_f16_fused_get_plan.argtypes = [P, I64, I64, P, I64, I64, P, P, P, I, P, I64, I64, I64, I64,
                                                      ctypes.POINTER(Plan)]
                L.gemm_f16_fused_get_plan.restype = ctypes.c_int
                _lib = L
    return _lib


def _check(st: int, what: str):
    if st != OK:
        raise GemmF16Error(st, what)


# ------------------------------------------------------------ C-ABI mirrors
def gemm_f16(A: int, stride_am: int, stride_ak: int, B: int, stride_bk: int, stride_bn: int,
             C: int, ldc: int, M: int, N: int, K: int, stream: int = 0) -> None:
    """C = A*B on device pointers (see include/gemm_f16.h); raises on a non-OK status."""
    _check(lib().gemm_f16(A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K,
                          stream or None), "gemm_f16")


def gemm_f16_ws(A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K,
                workspace: int, workspace_bytes: int, stream: int = 0) -> None:
    _check(lib().gemm_f16_ws(A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K,
                             workspace or None, workspace_bytes, stream or None), "gemm_f16_ws")


def gemm_f16_noalloc(A: int, stride_am: int, stride_ak: int, B: int, stride_bk: int, stride_bn: int,
                     C: int, ldc: int, M: int, N: int, K: int, stream: int = 0) -> None:
    """gemm_f16 for callers that must not allocate device memory: split-K /
    stream-K partials go to the library's fixed 8 MiB device array instead of
    a cudaMalloc'd workspace (see include/gemm_f16.h)."""
    _check(lib().gemm_f16_noalloc(A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K,
                                  stream or None), "gemm_f16_noalloc")


def gemm_f16_batched(A: int, stride_ab: int, stride_am: int, stride_ak: int, B: int, stride_bb: int,
                     stride_bk: int, stride_bn: int, C: int, stride_cb: int, ldc: int, M: int, N: int, K: int,
                     batch: int, stream: int = 0) -> None:
    """`batch` problems C_b = A_b * B_b of one shape (see include/gemm_f16.h)."""
    _check(lib().gemm_f16_batched(A, stride_ab, stride_am, stride_ak, B, stride_bb, stride_bk, stride_bn, C,
                                  stride_cb, ldc, M, N, K, batch, stream or None), "gemm_f16_batched")


def gemm_f16_grouped(A: int, stride_am: int, stride_ak: int, B: int, stride_bg: int, stride_bk: int,
                     stride_bn: int, C: int, ldc: int, group_rows, N: int, K: int, stream: int = 0) -> None:
    """Grouped problems sharing K and N: group g owns group_rows[g] consecutive rows
    of A and C and multiplies them by B + g*stride_bg (see include/gemm_f16.h)."""
    rows = (ctypes.c_int64 * len(group_rows))(*[int(r) for r in group_rows])
    _check(lib().gemm_f16_grouped(A, stride_am, stride_ak, B, stride_bg, stride_bk, stride_bn, C, ldc, rows,
                                  len(group_rows), N, K, stream or None), "gemm_f16_grouped")


def gemm_f16_fused(A: int, stride_am: int, stride_ak: int, B: int, stride_bk: int, stride_bn: int, B_up: int,
                   bias: int, bias_up: int, act: int, C: int, ldc: int, M: int, N: int, K: int,
                   stream: int = 0) -> None:
    """C = act(A*B + bias), or with B_up (read with B's strides) the gate/up form
    act(A*B + bias) * (A*B_up + bias_up); 0 for an absent B_up / bias (see
    include/gemm_f16.h)."""
    _check(lib().gemm_f16_fused(A, stride_am, stride_ak, B, stride_bk, stride_bn, B_up or None, bias or None,
                                bias_up or None, act, C, ldc, M, N, K, stream or None), "gemm_f16_fused")


def gemm_f16_batched_fused(A: int, stride_ab: int, stride_am: int, stride_ak: int, B: int, stride_bb: int,
                           stride_bk: int, stride_bn: int, B_up: int, bias: int, bias_up: int, stride_bias: int,
                           act: int, C: int, stride_cb: int, ldc: int, M: int, N: int, K: int, batch: int,
                           stream: int = 0) -> None:
    """gemm_f16_batched with the fused output stage (see include/gemm_f16.h)."""
    _check(lib().gemm_f16_batched_fused(A, stride_ab, stride_am, stride_ak, B, stride_bb, stride_bk, stride_bn,
                                        B_up or None, bias or None, bias_up or None, stride_bias, act, C,
                                        stride_cb, ldc, M, N, K, batch, stream or None), "gemm_f16_batched_fused")


def gemm_f16_grouped_fused(A: int, stride_am: int, stride_ak: int, B: int, stride_bg: int, stride_bk: int,
                           stride_bn: int, B_up: int, bias: int, bias_up: int, stride_bias: int, act: int, C: int,
                           ldc: int, group_rows, N: int, K: int, stream: int = 0) -> None:
    """gemm_f16_grouped with the fused output stage (see include/gemm_f16.h)."""
    rows = (ctypes.c_int64 * len(group_rows))(*[int(r) for r in group_rows])
    _check(lib().gemm_f16_grouped_fused(A, stride_am, stride_ak, B, stride_bg, stride_bk, stride_bn, B_up or None,
                                        bias or None, bias_up or None, stride_bias, act, C, ldc, rows,
                                        len(group_rows), N, K, stream or None), "gemm_f16_grouped_fused")


def gemm_f16_fused_get_plan(A, stride_am, stride_ak, B, stride_bk, stride_bn, B_up, bias, bias_up, act, C, ldc, M,
                            N, K) -> dict:
    p = Plan()
    _check(lib().gemm_f16_fused_get_plan(A, stride_am, stride_ak, B, stride_bk, stride_bn, B_up or None,
                                         bias or None, bias_up or None, act, C, ldc, M, N, K, ctypes.byref(p)),
           "gemm_f16_fused_get_plan")
    return p.as_dict()


def gemm_f16_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().gemm_f16_workspace_size(M, N, K, ctypes.byref(n)), "gemm_f16_workspace_size")
    return n.value


def gemm_f16_status_string(status: int) -> str:
    return lib().gemm_f16_status_string(status).decode()


def gemm_f16_device_status(reset: bool = False) -> int:
    v = ctypes.c_int(0)
    _check(lib().gemm_f16_device_status(ctypes.byref(v), 1 if reset else 0), "gemm_f16_device_status")
    return v.value


def gemm_f16_get_plan(A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K) -> dict:
    p = Plan()
    _check(lib().gemm_f16_get_plan(A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K,
                                   ctypes.byref(p)), "gemm_f16_get_plan")
    return p.as_dict()


def gemm_f16_set_option(option: int, value: int) -> None:
    _check(lib().gemm_f16_set_option(option, value), "gemm_f16_set_option")


def gemm_f16_abi_version() -> int:
    return lib().gemm_f16_abi_version()


# ------------------------------------------------------------ torch helpers
def _check_tensors(*ts):
    """Every given tensor (None entries skipped) is float16 and all sit on one
    CUDA device: the library reads raw fp16 device memory, so anything else
    would be misread rather than refused."""
    import torch

    ts = [t for t in ts if t is not None]
    if any(t.dtype != torch.float16 for t in ts):
        raise TypeError("gemm_f16 takes float16 tensors")
    if not all(t.is_cuda for t in ts) or len({t.device for t in ts}) > 1:
        raise ValueError("tensors must share one CUDA device")


def _check_out(out, shape, what):
    if out is not None and (tuple(out.shape) != tuple(shape) or out.stride(-1) != 1):
        raise ValueError(f"out must be {what} with a unit column stride")


def _args(a, b, out):
    if a.dim() != 2 or b.dim() != 2:
        raise ValueError("expected two matrices")
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out.dim() != 2 or tuple(out.shape) != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with unit column stride")
    return (a.data_ptr(), a.stride(0), a.stride(1), b.data_ptr(), b.stride(0), b.stride(1),
            out.data_ptr(), out.stride(0), M, N, K)


def matmul(a, b, out=None, stream=None):
    """fp16 C = a @ b for CUDA torch tensors (any positive strides); returns C."""
    import torch

    if a.dim() != 2 or b.dim() != 2:
        raise ValueError("expected two matrices")
    _check_out(out, (a.shape[0], b.shape[1]), "[M, N]")
    _check_tensors(a, b, out)
    if out is None:
        out = torch.empty((a.shape[0], b.shape[1]), dtype=torch.float16, device=a.device)
    args = _args(a, b, out)
    with torch.cuda.device(a.device):
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        gemm_f16(*args, stream=s.cuda_stream)
    return out


def bmm(a, b, out=None, stream=None):
    """fp16 C[i] = a[i] @ b[i] for 3-D CUDA torch tensors (a batch dimension of
    stride 0 shares that operand); returns C."""
    import torch

    if a.dim() != 3 or b.dim() != 3 or a.shape[0] != b.shape[0] or a.shape[2] != b.shape[1]:
        raise ValueError("bmm takes [batch, M, K] and [batch, K, N]")
    _check_out(out, (a.shape[0], a.shape[1], b.shape[2]), "[batch, M, N]")
    _check_tensors(a, b, out)
    if out is None:
        out = torch.empty((a.shape[0], a.shape[1], b.shape[2]), dtype=torch.float16, device=a.device)
    with torch.cuda.device(a.device):
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        gemm_f16_batched(a.data_ptr(), a.stride(0), a.stride(1), a.stride(2), b.data_ptr(), b.stride(0),
                         b.stride(1), b.stride(2), out.data_ptr(), out.stride(0), out.stride(1), a.shape[1],
                         b.shape[2], a.shape[2], a.shape[0], stream=s.cuda_stream)
    return out


def grouped_mm(a, b, group_rows, out=None, stream=None):
    """fp16 grouped product: rows of `a` [sum(group_rows), K] in consecutive groups,
    group g times b[g] ([G, K, N]); returns C [sum(group_rows), N]."""
    import torch

    if a.dim() != 2 or b.dim() != 3 or b.shape[0] != len(group_rows) or a.shape[1] != b.shape[1]:
        raise ValueError("grouped_mm takes [rows, K], [G, K, N] and G row counts")
    if sum(int(r) for r in group_rows) != a.shape[0]:
        raise ValueError("group_rows must add up to a's rows")
    _check_out(out, (a.shape[0], b.shape[2]), "[rows, N]")
    _check_tensors(a, b, out)
    if out is None:
        out = torch.empty((a.shape[0], b.shape[2]), dtype=torch.float16, device=a.device)
    with torch.cuda.device(a.device):
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        gemm_f16_grouped(a.data_ptr(), a.stride(0), a.stride(1), b.data_ptr(), b.stride(0), b.stride(1),
                         b.stride(2), out.data_ptr(), out.stride(0), group_rows, b.shape[2], a.shape[1],
                         stream=s.cuda_stream)
    return out


def _act(act) -> int:
    if isinstance(act, str):
        if act not in ACTIVATIONS:
            raise ValueError(f"unknown activation {act!r}")
        return ACTIVATIONS[act]
    return int(act)


def _epilogue_args(b, b_up, bias, bias_up, problems: int, n: int):
    """(B_up pointer, bias pointer, bias_up pointer, bias stride) for the fused
    entry points; a bias is [n] (shared) or [problems, n] with a unit last stride."""
    import torch

    if b_up is not None:
        if b_up.shape != b.shape or b_up.stride() != b.stride() or b_up.dtype != torch.float16:
            raise ValueError("b_up must be float16 with b's shape and strides")
    if bias_up is not None and b_up is None:
        raise ValueError("bias_up needs b_up")
    strides = []
    ptrs = []
    for v in (bias, bias_up):
        if v is None:
            ptrs.append(0)
            continue
        if v.dtype != torch.float16 or v.shape[-1] != n or v.stride(-1) != 1 or v.dim() not in (1, 2):
            raise ValueError("a bias is float16 [N] or [problems, N] with unit stride")
        if v.dim() == 2:
            if v.shape[0] != problems:
                raise ValueError("a 2-D bias has one row per problem")
            strides.append(v.stride(0))
        else:
            strides.append(0)
        ptrs.append(v.data_ptr())
    if len(set(strides)) > 1:
        raise ValueError("bias and bias_up must share one layout")
    return (b_up.data_ptr() if b_up is not None else 0), ptrs[0], ptrs[1], (strides[0] if strides else 0)


def fused_mm(a, b, bias=None, act="none", b_up=None, bias_up=None, out=None, stream=None):
    """fp16 act(a @ b + bias), or with b_up the gate/up form
    act(a @ b + bias) * (a @ b_up + bias_up), for 2-D or batched 3-D CUDA
    tensors; returns C."""
    import torch

    if a.dim() != b.dim() or a.dim() not in (2, 3):
        raise ValueError("fused_mm takes two matrices or two batches of matrices")
    code = _act(act)
    if a.dim() == 2:
        _check_out(out, (a.shape[0], b.shape[1]), "[M, N]")
        bu, bp, bup, _ = _epilogue_args(b, b_up, bias, bias_up, 1, b.shape[1])
        _check_tensors(a, b, out, b_up, bias, bias_up)
        if out is None:
            out = torch.empty((a.shape[0], b.shape[1]), dtype=torch.float16, device=a.device)
        args = _args(a, b, out)
        with torch.cuda.device(a.device):
            s = stream if stream is not None else torch.cuda.current_stream(a.device)
            gemm_f16_fused(*args[:6], bu, bp, bup, code, *args[6:], stream=s.cuda_stream)
        return out
    if a.shape[0] != b.shape[0] or a.shape[2] != b.shape[1]:
        raise ValueError("fused_mm takes [batch, M, K] and [batch, K, N]")
    _check_out(out, (a.shape[0], a.shape[1], b.shape[2]), "[batch, M, N]")
    bu, bp, bup, sbias = _epilogue_args(b, b_up, bias, bias_up, a.shape[0], b.shape[2])
    _check_tensors(a, b, out, b_up, bias, bias_up)
    if out is None:
        out = torch.empty((a.shape[0], a.shape[1], b.shape[2]), dtype=torch.float16, device=a.device)
    with torch.cuda.device(a.device):
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        gemm_f16_batched_fused(a.data_ptr(), a.stride(0), a.stride(1), a.stride(2), b.data_ptr(), b.stride(0),
                               b.stride(1), b.stride(2), bu, bp, bup, sbias, code, out.data_ptr(), out.stride(0),
                               out.stride(1), a.shape[1], b.shape[2], a.shape[2], a.shape[0],
                               stream=s.cuda_stream)
    return out


def grouped_fused_mm(a, b, group_rows, bias=None, act="none", b_up=None, bias_up=None, out=None, stream=None):
    """grouped_mm with the fused output stage: group g's rows become
    act(a_g @ b[g] + bias[g]) (times a_g @ b_up[g] + bias_up[g] with b_up); a
    bias is [N] (shared) or [G, N]."""
    import torch

    if a.dim() != 2 or b.dim() != 3 or b.shape[0] != len(group_rows) or a.shape[1] != b.shape[1]:
        raise ValueError("grouped_fused_mm takes [rows, K], [G, K, N] and G row counts")
    if sum(int(r) for r in group_rows) != a.shape[0]:
        raise ValueError("group_rows must add up to a's rows")
    code = _act(act)
    _check_out(out, (a.shape[0], b.shape[2]), "[rows, N]")
    bu, bp, bup, sbias = _epilogue_args(b, b_up, bias, bias_up, b.shape[0], b.shape[2])
    _check_tensors(a, b, out, b_up, bias, bias_up)
    if out is None:
        out = torch.empty((a.shape[0], b.shape[2]), dtype=torch.float16, device=a.device)
    with torch.cuda.device(a.device):
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        gemm_f16_grouped_fused(a.data_ptr(), a.stride(0), a.stride(1), b.data_ptr(), b.stride(0), b.stride(1),
                               b.stride(2), bu, bp, bup, sbias, code, out.data_ptr(), out.stride(0), group_rows,
                               b.shape[2], a.shape[1], stream=s.cuda_stream)
    return out


def fused_plan_for(a, b, out, bias=None, act="none", b_up=None, bias_up=None) -> dict:
    """The execution plan fused_mm would use for these 2-D torch tensors."""
    args = _args(a, b, out)
    bu, bp, bup, _ = _epilogue_args(b, b_up, bias, bias_up, 1, b.shape[1])
    _check_tensors(a, b, out, b_up, bias, bias_up)
    return gemm_f16_fused_get_plan(*args[:6], bu, bp, bup, _act(act), *args[6:])


def plan_for(a, b, out) -> dict:
    """The execution plan gemm_f16 would use for these torch tensors."""
    args = _args(a, b, out)
    _check_tensors(a, b, out)
    return gemm_f16_get_plan(*args)
