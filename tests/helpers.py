"""Shared test utilities: device upload, padded copies, tolerance checks.

Tolerances (floating point), elementwise against the CPU oracle:
  FP16/BF16 -> FP32:  |D - D_ref| <= 1e-3 * (|A||B|)_ij + 1e-6
  FP64:               |D - D_ref| <= 1e-12 * (|A||B|)_ij + 2^-52 * |D_ref|_ij
(the second FP64 term is the final rounding of the sum with C, which the
first term does not cover when |A||B| is tiny next to |C|).  INT8 -> INT32
is bit-exact.
"""
from __future__ import annotations

import numpy as np

import oracle

TOL = {"f16": (1e-3, 1e-6), "bf16": (1e-3, 1e-6), "f64": (1e-12, 0.0)}


def torch_dev():
    import torch
    return torch.device("cuda:0")


def to_dev(x: np.ndarray, dtype_in: str | None = None):
    """Upload a numpy array; 16-bit float bit patterns become f16/bf16."""
    import torch
    dev = torch_dev()
    if x.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev)
        return t.view(torch.bfloat16 if dtype_in == "bf16" else torch.float16)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def padded(x: np.ndarray, align_bytes: int = 16, extra: int = 0,
           fill: int = 0x5A) -> np.ndarray:
    """Copy of a 2-D array whose rows are padded to a 16-byte multiple
    (plus `extra` elements), padding filled with garbage."""
    rows, cols = x.shape
    per = align_bytes // x.itemsize
    ld = ((cols + per - 1) // per) * per + extra * per
    big = np.empty((rows, ld), x.dtype)
    big.view(np.uint8)[:] = fill
    big[:, :cols] = x
    return big[:, :cols]


def dev_padded(x: np.ndarray, dtype_in: str | None = None, extra: int = 0):
    """Device tensor view (rows, cols) with a padded leading dimension."""
    p = padded(x, extra=extra)
    base = to_dev(p.base if p.base is not None else p, dtype_in)
    return base[:, : x.shape[1]]


def check(dtype_in: str, got: np.ndarray, want: np.ndarray,
          absab: np.ndarray | None, what: str = "") -> None:
    if dtype_in == "i8":
        if not np.array_equal(got, want):
            bad = np.argwhere(got != want)
            idx = tuple(int(v) for v in bad[0])
            raise AssertionError(f"{what}: {len(bad)} INT32 mismatches, first "
                                 f"at {idx}: {got[idx]} vs {want[idx]}")
        return
    rel, ab0 = TOL[dtype_in]
    g = got.astype(np.float64)
    w = want.astype(np.float64)
    err = np.abs(g - w)
    bound = rel * absab + ab0
    if dtype_in == "f64":
        bound = bound + np.abs(w) * 2.0 ** -52
    bad = err > bound
    if np.any(bad) or not np.all(np.isfinite(g)):
        idx = np.argwhere(bad | ~np.isfinite(g))
        i = tuple(idx[0])
        raise AssertionError(
            f"{what}: {len(idx)} of {got.size} outside tolerance; first at {i}: "
            f"got {g[i]!r} want {w[i]!r} bound {bound[i]:.3e}; "
            f"max err/bound {np.max(err / np.maximum(bound, 1e-300)):.3f}")


def decode16(bits: np.ndarray, dtype_in: str) -> np.ndarray:
    bits = np.asarray(bits, np.uint16)
    if dtype_in == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def check16(dtype_in: str, got_bits, want_bits, absab, what: str = "") -> None:
    """16-bit accumulate: |D - D_ref| <= 1e-3 (|A||B|)_ij + 1e-6 + one ulp of
    the 16-bit result (2^-10 |D_ref| for FP16, 2^-7 for BF16): the GPU rounds
    its FP32 sum to 16 bits, the oracle its double sum."""
    g = decode16(got_bits, dtype_in)
    w = decode16(want_bits, dtype_in)
    ulp = 2.0 ** -10 if dtype_in == "f16" else 2.0 ** -7
    bound = 1e-3 * absab + 1e-6 + ulp * np.abs(w)
    err = np.abs(g - w)
    bad = (err > bound) | ~np.isfinite(g)
    if np.any(bad):
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError(f"{what}: {len(idx)} of {g.size} outside tolerance; "
                             f"first at {i}: got {g[i]!r} want {w[i]!r} bound {bound[i]:.3e}")


def oracle_ref(g, rows=None, cols=None):
    """Oracle D (and |A||B|) for GemmInputs g, optionally on a sub-block."""
    A, B, C = g.A, g.B, g.C
    if rows is not None:
        A = np.ascontiguousarray(A[rows])
        C = np.ascontiguousarray(C[rows])
    if cols is not None:
        if g.b_layout == "col":
            B = np.ascontiguousarray(B[cols])
        else:
            B = np.ascontiguousarray(B[:, cols])
        C = np.ascontiguousarray(C[:, cols])
    if g.dtype_in == "i8":
        return oracle.gemm("i8", A, B, C, b_layout=g.b_layout), None
    return oracle.gemm(g.dtype_in, A, B, C, b_layout=g.b_layout,
                       want_absab=True)
