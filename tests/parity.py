"""Shared parity helpers for the GPU tests: tolerance, sampling, oracle calls.

The tolerance is the one the product is specified against: per element
|C_gpu - C_oracle| <= 2 fp16 ulp(|C_oracle|) + 1e-4*sqrt(K), and a relative
Frobenius error <= 1e-3.  ulp16(x) = 2^(floor(log2|x|) - 10) for normal |x|,
2^-24 below the normal range (including 0).  Integer-valued inputs make every
fp32 sum exact, so there the outputs must match bit for bit.
"""
from __future__ import annotations

import numpy as np

import oracle


def ulp16(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    small = a < 2.0 ** -14
    e = np.floor(np.log2(np.where(small, 1.0, a)))
    return np.where(small, 2.0 ** -24, 2.0 ** (e - 10))


def assert_close(got, ref, K, what=""):
    """got/ref float16 arrays of the same shape (ref from the oracle)."""
    g = np.asarray(got).astype(np.float64)
    r = np.asarray(ref).astype(np.float64)
    assert g.shape == r.shape, what
    assert np.all(np.isfinite(g) == np.isfinite(r)), f"{what}: non-finite mismatch"
    fin = np.isfinite(r)
    err = np.abs(g[fin] - r[fin])
    tol = 2 * ulp16(r[fin]) + 1e-4 * np.sqrt(K)
    bad = err > tol
    if bad.any():
        i = np.argmax(err - tol)
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; worst err {err[i]:.3e} "
                             f"tol {tol[i]:.3e} ref {r[fin][i]:.6g} got {g[fin][i]:.6g}")
    nr = np.linalg.norm(r[fin])
    if nr > 0:
        rel = np.linalg.norm(g[fin] - r[fin]) / nr
        assert rel <= 1e-3, f"{what}: relative Frobenius error {rel:.3e}"


def assert_bits(got, ref, what=""):
    g = np.ascontiguousarray(got).view(np.uint16)
    r = np.ascontiguousarray(ref).view(np.uint16)
    if not np.array_equal(g, r):
        idx = np.argwhere(g != r)
        raise AssertionError(f"{what}: {len(idx)} elements differ, first at {idx[0].tolist()}: "
                             f"{np.asarray(got)[tuple(idx[0])]} vs {np.asarray(ref)[tuple(idx[0])]}")


def oracle_threads():
    return max(1, oracle.max_threads())


def sampled_reference(w, ms, ns):
    """Oracle values of C[ms[i], ns[i]] for workload `w`, regenerating only the
    needed rows of A and columns of B from the seeded generator."""
    K = w.K
    ms = np.asarray(ms, dtype=np.int64)
    ns = np.asarray(ns, dtype=np.int64)
    ur, ri = np.unique(ms, return_inverse=True)
    uc, ci = np.unique(ns, return_inverse=True)
    k = np.arange(K, dtype=np.int64)
    A_rows = w.A.values_at(ur[:, None], k[None, :])          # [R, K]
    B_cols = w.B.values_at(k[None, :], uc[:, None])          # [Cn, K] (column n as a row)
    vals, _ = oracle.dots(A_rows.reshape(-1), ri * K, 1, B_cols.reshape(-1), ci * K, 1, K,
                          threads=oracle_threads())
    return vals


def block_reference(w, m0, m1, n0, n1):
    """Oracle block C[m0:m1, n0:n1] of workload `w` (regenerates rows/cols)."""
    K = w.K
    k = np.arange(K, dtype=np.int64)
    A_rows = np.ascontiguousarray(w.A.values_at(np.arange(m0, m1)[:, None], k[None, :]))
    B_cols = np.ascontiguousarray(w.B.values_at(k[None, :], np.arange(n0, n1)[:, None]))
    return oracle.gemm(A_rows, B_cols.T, threads=oracle_threads())


# Largest slope of each activation: |act'(x)| <= L (ReLU 1; SiLU peaks at
# about 1.0998 near x = 2.4; GELU at about 1.1289 near x = 1.41).
ACT_SLOPE = {"none": 1.0, "relu": 1.0, "silu": 1.1, "gelu": 1.13}


def assert_close_fused(got, ref, K, g, u=None, act="none", what=""):
    """Fused output stage: the plain tolerance's absolute term e = 1e-4*sqrt(K)
    bounds the error of each fp32 sum; carried through act (slope <= L) and,
    gated, the product act(g) * u, it becomes e*(L*|u| + |act(g)|) + L*e^2.
    Plus 2 fp16 ulps of the result, and a relative Frobenius error <= 1e-3."""
    gv = np.asarray(got).astype(np.float64)
    r = np.asarray(ref).astype(np.float64)
    assert gv.shape == r.shape, what
    assert np.all(np.isfinite(gv) == np.isfinite(r)), f"{what}: non-finite mismatch"
    e = 1e-4 * np.sqrt(K)
    L = ACT_SLOPE[act]
    if u is None:
        absb = L * e + np.zeros_like(r)
    else:
        absb = e * (L * np.abs(u) + np.abs(oracle.activation(g, act))) + L * e * e
    fin = np.isfinite(r)
    err = np.abs(gv[fin] - r[fin])
    tol = 2 * ulp16(r[fin]) + absb[fin]
    bad = err > tol
    if bad.any():
        i = np.argmax(err - tol)
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; worst err {err[i]:.3e} "
                             f"tol {tol[i]:.3e} ref {r[fin][i]:.6g} got {gv[fin][i]:.6g}")
    nr = np.linalg.norm(r[fin])
    if nr > 0:
        rel = np.linalg.norm(gv[fin] - r[fin]) / nr
        assert rel <= 1e-3, f"{what}: relative Frobenius error {rel:.3e}"
