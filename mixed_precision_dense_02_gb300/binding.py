"""Thin ctypes binding over the C ABI in ``include/mma_gb300.h``.

Argument marshalling only: every step of D = A*B + C runs in the CUDA
library ``libmma_gb300.so`` built in-tree from ``csrc/``.  PyTorch supplies
device memory and the current stream.  If the library is missing, or no
CUDA device is present, calls raise; nothing here computes on the CPU.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBNAME = "libmma_gb300.so"

MMA_F16, MMA_BF16, MMA_I8, MMA_F64, MMA_F32, MMA_I32 = 1, 2, 3, 4, 5, 6
MMA_COL_MAJOR, MMA_ROW_MAJOR = 0, 1
STATUS = {0: "MMA_OK", 1: "MMA_ERR_INVALID_ARG", 2: "MMA_ERR_UNSUPPORTED",
          3: "MMA_ERR_MISALIGNED", 4: "MMA_ERR_LAUNCH", 5: "MMA_ERR_TIMEOUT",
          6: "MMA_ERR_NO_DEVICE", 7: "MMA_ERR_NO_MEMORY"}

# The exported entry points and their ctypes signatures (kept in step with
# include/mma_gb300.h; tests check both lists against the header).
_p, _i64, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
SIGNATURES = {
    "mma_gemm": (_int, [_int, _int, _i64, _i64, _i64, _p, _i64, _p, _i64, _p,
                        _i64, _p, _i64, _p]),
    "mma_gemm_ex": (_int, [_int, _int, _i64, _i64, _i64, _p, _i64, _p, _i64,
                           _int, _p, _i64, _p, _i64, _p]),
    "mma_gemm_batched": (_int, [_int, _int, _i64, _i64, _i64, _p, _i64, _p,
                                _i64, _p, _i64, _p, _i64, _i64, _int, _int,
                                _p]),
    "mma_gemm_batched_ex": (_int, [_int, _int, _i64, _i64, _i64, _p, _i64, _p,
                                   _i64, _p, _i64, _p, _i64, _i64, _int, _int,
                                   _int, _p]),
    "mma_gemm_i8_ex": (_int, [_i64, _i64, _i64, _p, _i64, _int, _p, _i64,
                              _int, _int, _p, _i64, _p, _i64, _int, _p]),
    "mma_gemm_i8_noalloc": (_int, [_i64, _i64, _i64, _p, _i64, _p, _i64, _p,
                                   _i64, _p, _i64, _p]),
    "mma_device_status": (_int, [_p]),
    "mma_selftest_wait_timeout": (_int, [_i64, _p]),
    "mma_selftest_gemm_abort": (_int, [_int, _i64, _p, _p, _p, _p]),
    "mma_peak_probe": (_int, [_int, _i64, ctypes.POINTER(ctypes.c_double), _p]),
    "mma_profile_begin": (_int, []),
    "mma_profile_end": (_int, [ctypes.POINTER(ctypes.c_float), _int,
                               ctypes.POINTER(_int)]),
    "mma_status_string": (ctypes.c_char_p, [_int]),
    "mma_version": (_int, []),
}

_lib = None
_lock = threading.Lock()


class MMAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


def library_path() -> str:
    return os.path.join(_HERE, _LIBNAME)


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{_LIBNAME} is not built (expected at {path}); run "
                    "`python -m mixed_precision_dense_02_gb300.build`")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MMAError(fn, status)


# --------------------------------------------------------------------------
# raw-pointer entry points (same names as the C ABI)

def mma_gemm(dtype_in, dtype_acc, M, N, K, A, lda, B, ldb, C, ldc, D, ldd,
             stream) -> int:
    return load().mma_gemm(dtype_in, dtype_acc, M, N, K, A, lda, B, ldb, C,
                           ldc, D, ldd, stream)


def mma_gemm_ex(dtype_in, dtype_acc, M, N, K, A, lda, B, ldb, layout_b, C,
                ldc, D, ldd, stream) -> int:
    return load().mma_gemm_ex(dtype_in, dtype_acc, M, N, K, A, lda, B, ldb,
                              layout_b, C, ldc, D, ldd, stream)


def mma_gemm_batched(dtype_in, dtype_acc, M, N, K, A, lda, B, ldb, C, ldc, D,
                     ldd, batch, group, abid, stream) -> int:
    return load().mma_gemm_batched(dtype_in, dtype_acc, M, N, K, A, lda, B,
                                   ldb, C, ldc, D, ldd, batch, group, abid,
                                   stream)


def mma_gemm_batched_ex(dtype_in, dtype_acc, M, N, K, A, lda, B, ldb, C, ldc,
                        D, ldd, batch, group, abid, blgp, stream) -> int:
    return load().mma_gemm_batched_ex(dtype_in, dtype_acc, M, N, K, A, lda, B,
                                      ldb, C, ldc, D, ldd, batch, group, abid,
                                      blgp, stream)


def mma_gemm_i8_ex(M, N, K, A, lda, a_neg, B, ldb, b_neg, layout_b, C, ldc,
                   D, ldd, clamp, stream) -> int:
    """8-bit integer GEMM, int8 or uint8 per operand, optional saturation."""
    return load().mma_gemm_i8_ex(M, N, K, A, lda, a_neg, B, ldb, b_neg,
                                 layout_b, C, ldc, D, ldd, clamp, stream)


def mma_gemm_i8_noalloc(M, N, K, A, lda, B, ldb, C, ldc, D, ldd,
                        stream) -> int:
    """INT8 -> INT32 GEMM that allocates no device memory (fixed scratch)."""
    return load().mma_gemm_i8_noalloc(M, N, K, A, lda, B, ldb, C, ldc, D, ldd,
                                      stream)


def mma_device_status(stream) -> int:
    return load().mma_device_status(stream)


def mma_selftest_wait_timeout(limit_ns, stream) -> int:
    """Run one bounded wait that is made to run out (failure-detection
    self-test); mma_device_status then reports MMA_ERR_TIMEOUT once."""
    return load().mma_selftest_wait_timeout(limit_ns, stream)


MMA_PEAK_TC_F16, MMA_PEAK_DMMA, MMA_PEAK_IMMA, MMA_PEAK_DFMA = 1, 2, 3, 4


def mma_peak_probe(kind, iterations, stream) -> tuple:
    """Enqueue one issue-rate probe; returns (status, operations per launch)."""
    ops = ctypes.c_double(0.0)
    st = load().mma_peak_probe(kind, iterations, ctypes.byref(ops), stream)
    return st, ops.value


def mma_selftest_gemm_abort(cluster, limit_ns, A, B, D, stream) -> int:
    """Run the tcgen05 GEMM kernel with no operand loads and waits limited to
    limit_ns, so its own abort path runs; mma_device_status then reports
    MMA_ERR_TIMEOUT once."""
    return load().mma_selftest_gemm_abort(cluster, limit_ns, A, B, D, stream)


def mma_status_string(status: int) -> str:
    return load().mma_status_string(status).decode()


# --------------------------------------------------------------------------
# torch-tensor convenience layer (still marshalling only)

def _torch():
    import torch
    return torch


def _dtypes(t):
    torch = _torch()
    m = {torch.float16: (MMA_F16, MMA_F32, torch.float32),
         torch.bfloat16: (MMA_BF16, MMA_F32, torch.float32),
         torch.int8: (MMA_I8, MMA_I32, torch.int32),
         torch.float64: (MMA_F64, MMA_F64, torch.float64)}
    if t.dtype not in m:
        raise TypeError(f"unsupported input dtype {t.dtype}")
    return m[t.dtype]


def _ld(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("2-D tensors with unit inner stride are required")
    return t.stride(0)


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def gemm_ex(A, B, C=None, D=None, *, b_layout: str = "col", acc=None,
            stream=None):
    """D = A @ B + C on the GPU.

    ``A``: (M, K) row-major; ``B`` as stored: (N, K) for column-major B
    (``b_layout="col"``) or (K, N) for row-major B; ``C``/``D``: (M, N).
    Input dtype float16/bfloat16 -> float32 output, int8 -> int32,
    float64 -> float64.  FP16/BF16 inputs accumulate into a 16-bit addend
    and result of their own type when ``acc="same"`` or when C or D has
    that dtype.  ``D`` is allocated when not given.  Returns D.
    """
    torch = _torch()
    dt_in, dt_acc, out_dtype = _dtypes(A)
    if A.dtype in (torch.float16, torch.bfloat16):
        given = D if D is not None else C
        if acc == "same" or (acc is None and given is not None
                             and given.dtype == A.dtype):
            dt_acc, out_dtype = dt_in, A.dtype
    if B.dtype != A.dtype:
        raise TypeError("A and B must have the same dtype")
    M, K = A.shape
    if b_layout == "col":
        N, Kb = B.shape
        layout = MMA_COL_MAJOR
    elif b_layout == "row":
        Kb, N = B.shape
        layout = MMA_ROW_MAJOR
    else:
        raise ValueError(b_layout)
    if Kb != K:
        raise ValueError(f"K mismatch: {K} vs {Kb}")
    if D is None:
        D = torch.empty((M, N), dtype=out_dtype, device=A.device)
    for t in (C, D):
        if t is not None and (t.dtype != out_dtype or tuple(t.shape) != (M, N)):
            raise ValueError("C/D must be (M, N) of the accumulator dtype")
    st = mma_gemm_ex(dt_in, dt_acc, M, N, K, A.data_ptr(), _ld(A),
                     B.data_ptr(), _ld(B), layout,
                     None if C is None else C.data_ptr(),
                     0 if C is None else _ld(C), D.data_ptr(), _ld(D),
                     _stream(stream))
    _check("mma_gemm_ex", st)
    return D


def gemm_i8_ex(A, B, C=None, D=None, *, clamp: bool = False,
               b_layout: str = "col", stream=None):
    """8-bit integer D = A @ B + C (INT32 C and D) on the GPU.

    Each of ``A`` and ``B`` is a torch.int8 (signed) or torch.uint8
    (unsigned) tensor; shapes and layouts as in ``gemm_ex``.  With ``clamp``
    D is the exact result saturated to the INT32 range, else it wraps
    modulo 2^32.  ``D`` is allocated when not given.  Returns D.
    """
    torch = _torch()
    sign = {torch.int8: 1, torch.uint8: 0}
    if A.dtype not in sign or B.dtype not in sign:
        raise TypeError("A and B must be int8 or uint8 tensors")
    M, K = A.shape
    if b_layout == "col":
        N, Kb = B.shape
        layout = MMA_COL_MAJOR
    elif b_layout == "row":
        Kb, N = B.shape
        layout = MMA_ROW_MAJOR
    else:
        raise ValueError(b_layout)
    if Kb != K:
        raise ValueError(f"K mismatch: {K} vs {Kb}")
    if D is None:
        D = torch.empty((M, N), dtype=torch.int32, device=A.device)
    for t in (C, D):
        if t is not None and (t.dtype != torch.int32 or tuple(t.shape) != (M, N)):
            raise ValueError("C/D must be (M, N) int32")
    st = mma_gemm_i8_ex(M, N, K, A.data_ptr(), _ld(A), sign[A.dtype],
                        B.data_ptr(), _ld(B), sign[B.dtype], layout,
                        None if C is None else C.data_ptr(),
                        0 if C is None else _ld(C), D.data_ptr(), _ld(D),
                        int(bool(clamp)), _stream(stream))
    _check("mma_gemm_i8_ex", st)
    return D


def gemm(A, B, C=None, D=None, *, acc=None, stream=None):
    """D = A @ B + C with B given column-major as an (N, K) tensor."""
    return gemm_ex(A, B, C, D, b_layout="col", acc=acc, stream=stream)


def gemm_batched(A, B, C=None, D=None, *, group: int = 1, abid: int = 0,
                 blgp: int = 0, acc=None, stream=None):
    """Batched D_b = A_{(b//group)*group + abid} @ B_{bsrc(b)} + C_b with
    bsrc(b) = (b//4)*4 + (quarter read under lane-group pattern ``blgp``).

    ``A``: (batch, M, K); ``B``: (batch, N, K) column-major tiles;
    ``C``/``D``: (batch, M, N); all contiguous.  Dtypes as in ``gemm_ex``
    (FP16/BF16 accumulate into their own type with ``acc="same"`` or a C/D
    of that type).
    """
    torch = _torch()
    dt_in, dt_acc, out_dtype = _dtypes(A)
    if A.dtype in (torch.float16, torch.bfloat16):
        given = D if D is not None else C
        if acc == "same" or (acc is None and given is not None
                             and given.dtype == A.dtype):
            dt_acc, out_dtype = dt_in, A.dtype
    batch, M, K = A.shape
    _, N, Kb = B.shape
    if Kb != K or B.shape[0] != batch:
        raise ValueError("shape mismatch")
    for t in (A, B, C, D):
        if t is not None and not t.is_contiguous():
            raise ValueError("batched operands must be contiguous")
    if D is None:
        D = torch.empty((batch, M, N), dtype=out_dtype, device=A.device)
    st = mma_gemm_batched_ex(dt_in, dt_acc, M, N, K, A.data_ptr(), K,
                             B.data_ptr(), K,
                             None if C is None else C.data_ptr(), N,
                             D.data_ptr(), N, batch, group, abid, blgp,
                             _stream(stream))
    _check("mma_gemm_batched_ex", st)
    return D


def profile_begin() -> None:
    """Start recording the duration of each call's dominant kernel."""
    _check("mma_profile_begin", load().mma_profile_begin())


def profile_end(max_count: int = 4096) -> list:
    """Stop recording; durations (ms) of the recorded dominant kernels."""
    buf = (ctypes.c_float * max_count)()
    n = _int(0)
    _check("mma_profile_end", load().mma_profile_end(buf, max_count, ctypes.byref(n)))
    return [float(buf[i]) for i in range(min(n.value, max_count))]


def device_status(stream=None) -> None:
    """Raise MMAError if an in-kernel wait has run out since the last check."""
    _check("mma_device_status", mma_device_status(_stream(stream)))
