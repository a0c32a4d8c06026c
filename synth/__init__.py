"""Seeded synthetic inputs for the fp16 GEMM, shared by the tests and the bench.

This module holds no GEMM arithmetic: it only produces fp16 matrices (as flat
buffers) from a counter-based random generator, so that any element can be
regenerated on the host from its flat index without materialising the rest.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style.  For a seed ``s`` the
stream base is ``b = mix(s + G)`` and element ``i`` of the buffer is
``z_i = mix(b + (i + 1) * G)`` (all mod 2**64), with ``G = 0x9E3779B97F4A7C15``
and ``mix`` the SplitMix64 finaliser (xor-shift 30, multiply, xor-shift 27,
multiply, xor-shift 31).

Distributions (both are one rounding away from an exact value):

* ``"uniform"``: ``v = (z >> 40) * 2**-23 - 1``, uniform on a 2**-23 grid in
  [-1, 1).  Every such ``v`` is exact in fp32, so rounding it to fp16 (round to
  nearest even) gives the same bits whether it goes double->half directly
  (numpy) or double->float->half (torch).
* ``"int3"``: ``((z >> 40) * 7 >> 24) - 3``, an integer in [-3, 3], exact in fp16.

Two implementations: numpy ``uint64`` (host, any subset of indices) and torch
``int64`` with two's-complement wrap-around (any device, whole buffers).  The
tests check that they agree bit for bit.
"""
from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
MUL1 = 0xBF58476D1CE4E5B9
MUL2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

KINDS = ("uniform", "int3")


def _mix_py(x: int) -> int:
    x &= MASK64
    x = ((x ^ (x >> 30)) * MUL1) & MASK64
    x = ((x ^ (x >> 27)) * MUL2) & MASK64
    return x ^ (x >> 31)


def stream_base(seed: int) -> int:
    """First SplitMix64 output for ``seed``: decorrelates neighbouring seeds."""
    return _mix_py((int(seed) + GOLDEN) & MASK64)


# --------------------------------------------------------------------- numpy
def _mix_np(x: np.ndarray) -> np.ndarray:
    x = x ^ (x >> np.uint64(30))
    x = x * np.uint64(MUL1)
    x = x ^ (x >> np.uint64(27))
    x = x * np.uint64(MUL2)
    return x ^ (x >> np.uint64(31))


def raw_np(seed: int, flat_idx) -> np.ndarray:
    """64-bit generator outputs ``z_i`` for the given flat element indices."""
    idx = np.asarray(flat_idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = np.uint64(stream_base(seed)) + (idx + np.uint64(1)) * np.uint64(GOLDEN)
        return _mix_np(x)


def values_np(kind: str, seed: int, flat_idx) -> np.ndarray:
    """fp16 values of the buffer elements at ``flat_idx`` (numpy float16)."""
    z = raw_np(seed, flat_idx)
    top = (z >> np.uint64(40)).astype(np.int64)
    if kind == "uniform":
        v = top.astype(np.float64) * (2.0 ** -23) - 1.0
        return v.astype(np.float16)
    if kind == "int3":
        return (((top * 7) >> 24) - 3).astype(np.float16)
    raise ValueError(f"unknown distribution {kind!r}")


def buffer_np(kind: str, seed: int, numel: int, chunk: int = 1 << 24) -> np.ndarray:
    """Whole flat buffer of ``numel`` fp16 elements on the host."""
    out = np.empty(int(numel), dtype=np.float16)
    for lo in range(0, int(numel), chunk):
        hi = min(int(numel), lo + chunk)
        out[lo:hi] = values_np(kind, seed, np.arange(lo, hi, dtype=np.uint64))
    return out


# --------------------------------------------------------------------- torch
def _signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


def _srl(x, s: int):
    """Logical right shift of an int64 tensor holding uint64 bit patterns."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix_torch(x):
    x = x ^ _srl(x, 30)
    x = x * _signed(MUL1)
    x = x ^ _srl(x, 27)
    x = x * _signed(MUL2)
    return x ^ _srl(x, 31)


def buffer_torch(kind: str, seed: int, numel: int, device="cpu", chunk: int = 1 << 26):
    """Whole flat fp16 buffer of ``numel`` elements as a torch tensor on ``device``.

    Same bits as :func:`buffer_np`; int64 arithmetic wraps modulo 2**64.
    """
    import torch

    if kind not in KINDS:
        raise ValueError(f"unknown distribution {kind!r}")
    numel = int(numel)
    out = torch.empty(numel, dtype=torch.float16, device=device)
    base = _signed(stream_base(seed))
    g = _signed(GOLDEN)
    for lo in range(0, numel, chunk):
        hi = min(numel, lo + chunk)
        idx = torch.arange(lo + 1, hi + 1, dtype=torch.int64, device=device)
        z = _mix_torch(idx * g + base)
        top = _srl(z, 40)
        if kind == "uniform":
            v = top.to(torch.float64) * (2.0 ** -23) - 1.0
            out[lo:hi] = v.to(torch.float32).to(torch.float16)
        else:
            out[lo:hi] = (((top * 7) >> 24) - 3).to(torch.float16)
        del idx, z, top
    return out


def matrix_np(kind: str, seed: int, rows: int, cols: int) -> np.ndarray:
    """Row-major ``rows x cols`` fp16 matrix on the host (flat index = r*cols + c)."""
    return buffer_np(kind, seed, rows * cols).reshape(rows, cols)


def matrix_torch(kind: str, seed: int, rows: int, cols: int, device="cpu"):
    """Row-major ``rows x cols`` fp16 matrix as a torch tensor on ``device``."""
    return buffer_torch(kind, seed, rows * cols, device).view(rows, cols)
