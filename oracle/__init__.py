"""CPU oracle for D = A*B + C -- TEST INFRASTRUCTURE ONLY.

The plain, slow, obviously-correct definition that the CUDA library is
checked against.  Only the test suite, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import it; the product path never does, and it
shares no code with the CUDA path (the one shared module is the seeded input
generator, which holds none of the method's arithmetic).

Arithmetic lives in ``mma_oracle.c`` (built with gcc, no fast-math, no FP
contraction).  This module only marshals numpy arrays into it.

Conventions (pages: "CDNA2 dense MFMA builtins" -- Naming convention and
Builtin reference; "RDNA3 dense WMMA builtins" -- Builtin reference;
"Common MFMA parameters" -- Shared parameters):

* ``A`` is M x K row-major.  ``B`` is given as stored: column-major
  (``b_layout="col"``: an N x K array whose row j is column j of B) or
  row-major (``b_layout="row"``: a K x N array).  ``C`` and ``D`` are M x N
  row-major.  Leading dimensions are taken from the arrays' strides.
* 16-bit floats are passed as their bit patterns (``uint16`` arrays, or
  ``float16`` arrays for FP16) together with ``dtype_in`` "f16" or "bf16".
* FP16/BF16 accumulate to FP32, INT8 to INT32, FP64 to FP64.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(exact rational brute force, closed forms, transpose invariance, the
broadcast worked example of "Common MFMA parameters").  No function is
parity-unpinned.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_DT = {"f16": 1, "bf16": 2, "i8": 3, "f64": 4}
_LAYOUT = {"col": 0, "row": 1}
_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_num_threads.restype = _int
        L.oracle_f16_to_double.restype = ctypes.c_double
        L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_gemm_f16f32.restype = _int
        L.oracle_gemm_f16f32.argtypes = [_int, _i64, _i64, _i64, _p, _i64, _p,
                                         _i64, _int, _p, _i64, _p, _i64, _p,
                                         _i64]
        L.oracle_gemm_f16f16.restype = _int
        L.oracle_gemm_f16f16.argtypes = [_int, _i64, _i64, _i64, _p, _i64, _p,
                                         _i64, _int, _p, _i64, _p, _i64, _p,
                                         _i64]
        L.oracle_double_to_f16.restype = ctypes.c_uint16
        L.oracle_double_to_f16.argtypes = [ctypes.c_double]
        L.oracle_double_to_bf16.restype = ctypes.c_uint16
        L.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        L.oracle_gemm_i8i32_ex.restype = _i64
        L.oracle_gemm_i8i32_ex.argtypes = [_i64, _i64, _i64, _p, _i64, _int, _p,
                                           _i64, _int, _int, _p, _i64, _p, _i64,
                                           _int]
        L.oracle_gemm_i8i32.restype = _i64
        L.oracle_gemm_i8i32.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64,
                                        _int, _p, _i64, _p, _i64]
        L.oracle_gemm_f64.restype = _int
        L.oracle_gemm_f64.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64,
                                      _int, _p, _i64, _p, _i64, _p, _i64]
        L.oracle_gemm_batched.restype = _i64
        L.oracle_gemm_batched.argtypes = [_int, _i64, _i64, _i64, _p, _i64, _p,
                                          _i64, _int, _p, _i64, _p, _i64, _i64,
                                          _i64, _i64, _int]
        L.oracle_blgp_source.restype = _int
        L.oracle_blgp_source.argtypes = [_int, _int]
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def f16_to_double(bits: int) -> float:
    return float(lib().oracle_f16_to_double(int(bits)))


def bf16_to_double(bits: int) -> float:
    return float(lib().oracle_bf16_to_double(int(bits)))


def double_to_f16(x: float) -> int:
    return int(lib().oracle_double_to_f16(float(x)))


def double_to_bf16(x: float) -> int:
    return int(lib().oracle_double_to_bf16(float(x)))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _ld(a: np.ndarray) -> int:
    """Leading dimension (elements) of a 2-D array with unit inner stride."""
    if a.ndim != 2 or a.strides[1] != a.itemsize:
        raise ValueError("2-D arrays with contiguous rows are required")
    if a.strides[0] % a.itemsize:
        raise ValueError("row stride must be a multiple of the item size")
    return a.strides[0] // a.itemsize


def _bits16(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("16-bit float operands are uint16 bit patterns or float16")
    return a


def _shape(A, B, b_layout):
    M, K = A.shape
    if b_layout == "col":
        N, Kb = B.shape
    elif b_layout == "row":
        Kb, N = B.shape
    else:
        raise ValueError(b_layout)
    if Kb != K:
        raise ValueError(f"K mismatch: A has {K}, B has {Kb}")
    return M, N, K


def gemm(dtype_in: str, A, B, C=None, *, b_layout: str = "col",
         want_absab: bool = False):
    """D = A*B + C on the CPU.

    Returns ``D`` (float32 / int32 / float64), or ``(D, absab)`` with
    ``absab[i, j] = sum_k |A[i, k]| * |B[k, j]|`` in float64 when
    ``want_absab`` is set (FP16/BF16/FP64 only).  For INT8 the count of
    outputs that overflowed INT32 is checked to be zero.
    """
    M, N, K = _shape(A, B, b_layout)
    L = lib()
    lay = _LAYOUT[b_layout]
    if C is not None and C.shape != (M, N):
        raise ValueError("C must be M x N")
    if dtype_in in ("f16", "bf16"):
        A16, B16 = _bits16(A), _bits16(B)
        Cf = None if C is None else np.asarray(C, dtype=np.float32)
        D = np.empty((M, N), np.float32)
        ab = np.empty((M, N), np.float64) if want_absab else None
        rc = L.oracle_gemm_f16f32(_DT[dtype_in], M, N, K, _ptr(A16), _ld(A16),
                                  _ptr(B16), _ld(B16), lay, _ptr(Cf),
                                  _ld(Cf) if Cf is not None else 0, _ptr(D), N,
                                  _ptr(ab), N)
        if rc != 0:
            raise RuntimeError("oracle_gemm_f16f32 failed")
        return (D, ab) if want_absab else D
    if dtype_in == "i8":
        if A.dtype != np.int8 or B.dtype != np.int8:
            raise TypeError("INT8 operands must be int8 arrays")
        Ci = None if C is None else np.asarray(C, dtype=np.int32)
        D = np.empty((M, N), np.int32)
        ov = L.oracle_gemm_i8i32(M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), lay,
                                 _ptr(Ci), _ld(Ci) if Ci is not None else 0,
                                 _ptr(D), N)
        if ov < 0:
            raise RuntimeError("oracle_gemm_i8i32 failed")
        if ov:
            raise OverflowError(f"{ov} outputs overflow INT32")
        return D
    if dtype_in == "f64":
        if A.dtype != np.float64 or B.dtype != np.float64:
            raise TypeError("FP64 operands must be float64 arrays")
        Cd = None if C is None else np.asarray(C, dtype=np.float64)
        D = np.empty((M, N), np.float64)
        ab = np.empty((M, N), np.float64) if want_absab else None
        rc = L.oracle_gemm_f64(M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), lay,
                               _ptr(Cd), _ld(Cd) if Cd is not None else 0,
                               _ptr(D), N, _ptr(ab), N)
        if rc != 0:
            raise RuntimeError("oracle_gemm_f64 failed")
        return (D, ab) if want_absab else D
    raise ValueError(f"unsupported dtype_in {dtype_in!r}")


def gemm_i8_ex(A, B, C=None, *, clamp: bool = False, b_layout: str = "col"):
    """8-bit integer D = A*B + C with A and B signed (int8 arrays) or
    unsigned (uint8 arrays) independently ("RDNA3 dense WMMA builtins" --
    INT8 and UINT8 inputs, a_neg/b_neg and clamp).  Returns (D int32, the
    number of outputs whose exact value overflowed INT32); overflowing
    outputs saturate with ``clamp``, else wrap modulo 2^32."""
    for t in (A, B):
        if t.dtype not in (np.int8, np.uint8):
            raise TypeError("8-bit integer operands are int8 or uint8 arrays")
    M, N, K = _shape(A, B, b_layout)
    Ci = None if C is None else np.asarray(C, dtype=np.int32)
    D = np.empty((M, N), np.int32)
    ov = lib().oracle_gemm_i8i32_ex(M, N, K, _ptr(A), _ld(A),
                                    int(A.dtype == np.int8), _ptr(B), _ld(B),
                                    int(B.dtype == np.int8), _LAYOUT[b_layout],
                                    _ptr(Ci), _ld(Ci) if Ci is not None else 0,
                                    _ptr(D), N, int(bool(clamp)))
    if ov < 0:
        raise RuntimeError("oracle_gemm_i8i32_ex failed")
    return D, int(ov)


def gemm_acc16(dtype_in: str, A, B, C=None, *, b_layout: str = "col",
               want_absab: bool = False):
    """D = A*B + C with a 16-bit addend and result of the input's type
    ("RDNA3 dense WMMA builtins" -- FP16/BF16-accumulate builtins).

    ``A``, ``B``, ``C`` are uint16 bit patterns (or float16 arrays for
    FP16); returns D as uint16 bit patterns, rounded once (nearest, ties to
    even) from the exact-product double sum, and optionally (|A|*|B|).
    """
    if dtype_in not in ("f16", "bf16"):
        raise ValueError(dtype_in)
    M, N, K = _shape(A, B, b_layout)
    A16, B16 = _bits16(A), _bits16(B)
    C16 = None if C is None else _bits16(np.asarray(C))
    if C16 is not None and C16.shape != (M, N):
        raise ValueError("C must be M x N")
    D = np.empty((M, N), np.uint16)
    ab = np.empty((M, N), np.float64) if want_absab else None
    rc = lib().oracle_gemm_f16f16(_DT[dtype_in], M, N, K, _ptr(A16), _ld(A16),
                                  _ptr(B16), _ld(B16), _LAYOUT[b_layout],
                                  _ptr(C16), _ld(C16) if C16 is not None else 0,
                                  _ptr(D), N, _ptr(ab), N)
    if rc != 0:
        raise RuntimeError("oracle_gemm_f16f16 failed")
    return (D, ab) if want_absab else D


def blgp_source(blgp: int, q: int) -> int:
    """Quarter whose B the entry at quarter q of a group of four reads under
    B lane-group pattern ``blgp`` ("Common MFMA parameters" -- Dense MFMA
    parameters, blgp), or -1 for an invalid pattern."""
    return int(lib().oracle_blgp_source(int(blgp), int(q)))


def gemm_batched(dtype_in: str, A, B, C, *, group: int = 1, abid: int = 0,
                 b_layout: str = "col", blgp: int = 0):
    """Batched tiles with A-block broadcast ("Common MFMA parameters" --
    Shared parameters, cbsz/abid) and B-group pattern (Dense MFMA
    parameters, blgp, read at matrix level).

    ``A``: (batch, M, K); ``B``: (batch, N, K) column-major tiles or
    (batch, K, N) row-major tiles; ``C``: (batch, M, N) or None.  Entry b
    uses A tile ``(b // group) * group + abid`` and B tile
    ``(b // 4) * 4 + blgp_source(blgp, b % 4)``.  All arrays contiguous.
    """
    batch, M, K = A.shape
    if b_layout == "col":
        _, N, Kb = B.shape
    else:
        _, Kb, N = B.shape
    if Kb != K or B.shape[0] != batch:
        raise ValueError("shape mismatch")
    for t in (A, B) + (() if C is None else (C,)):
        if not t.flags.c_contiguous:
            raise ValueError("batched operands must be contiguous")
    if dtype_in in ("f16", "bf16"):
        A, B = _bits16(A), _bits16(B)
        out_dt, c_dt = np.float32, np.float32
    elif dtype_in == "i8":
        out_dt, c_dt = np.int32, np.int32
    elif dtype_in == "f64":
        out_dt, c_dt = np.float64, np.float64
    else:
        raise ValueError(dtype_in)
    Cc = None if C is None else np.ascontiguousarray(C, dtype=c_dt)
    D = np.empty((batch, M, N), out_dt)
    rc = lib().oracle_gemm_batched(_DT[dtype_in], M, N, K, _ptr(A), K, _ptr(B),
                                   K if b_layout == "col" else N,
                                   _LAYOUT[b_layout], _ptr(Cc), N, _ptr(D), N,
                                   batch, group, abid, int(blgp))
    if rc < 0:
        raise ValueError("oracle_gemm_batched rejected its arguments")
    if rc > 0:
        raise OverflowError(f"{rc} outputs overflow INT32")
    return D


__all__ = ["gemm", "gemm_i8_ex", "gemm_acc16", "blgp_source", "gemm_batched", "num_threads",
           "f16_to_double", "bf16_to_double", "double_to_f16",
           "double_to_bf16", "lib"]
