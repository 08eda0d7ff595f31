"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments before touching a device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from mixed_precision_dense_02_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mma_gb300.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mma_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    fns = header_functions()
    for f in ("mma_gemm", "mma_gemm_ex", "mma_gemm_batched", "mma_gemm_i8_ex",
              "mma_device_status", "mma_status_string", "mma_version"):
        assert f in fns


def test_every_declared_symbol_is_exported(lib):
    for f in header_functions():
        assert hasattr(lib, f), f
    assert sorted(binding.SIGNATURES) == header_functions()


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert binding.mma_status_string(code) == name
    assert binding.mma_status_string(99) == "MMA_ERR_UNKNOWN"
    assert binding.load().mma_version() == 200


F16, BF16, I8, F64, F32, I32 = 1, 2, 3, 4, 5, 6
OK, INVALID, UNSUP, MISAL, LAUNCH, TIMEOUT, NODEV = range(7)
P = 1 << 20  # 16-byte aligned fake device addresses; never dereferenced
Q = 1 << 24


def g(*, din=BF16, dacc=F32, M=64, N=64, K=64, A=P, lda=64, B=P, ldb=64,
      C=P, ldc=64, D=Q, ldd=64, layout=0):
    return binding.mma_gemm_ex(din, dacc, M, N, K, A, lda, B, ldb, layout, C,
                               ldc, D, ldd, None)


@pytest.mark.parametrize("kw,code", [
    (dict(din=BF16, dacc=I32), UNSUP),
    (dict(din=BF16, dacc=F16), UNSUP),
    (dict(din=F16, dacc=BF16), UNSUP),
    (dict(din=I8, dacc=I8), UNSUP),
    (dict(din=F32, dacc=F32), UNSUP),
    (dict(din=I8, dacc=F32), UNSUP),
    (dict(din=F64, dacc=F32), UNSUP),
    (dict(M=-1), INVALID),
    (dict(K=-5), INVALID),
    (dict(layout=2), INVALID),
    (dict(lda=32), INVALID),
    (dict(ldb=8), INVALID),
    (dict(ldc=8), INVALID),
    (dict(ldd=8), INVALID),
    (dict(D=0), INVALID),
    (dict(A=0), INVALID),
    (dict(B=0), INVALID),
    (dict(C=P, D=P, ldc=64, ldd=128), INVALID),
    (dict(A=P + 2), MISAL),
    (dict(B=P + 8), MISAL),
    (dict(C=P + 4), MISAL),
    (dict(D=Q + 4), MISAL),
    (dict(lda=68), MISAL),           # 68 * 2 bytes is not a 16-byte multiple
    (dict(din=I8, dacc=I32, lda=72, ldb=64), MISAL),
    (dict(ldd=66), MISAL),
    (dict(din=F64, dacc=F64, lda=65), MISAL),
])
def test_argument_errors_detected_before_launch(lib, kw, code):
    assert g(**kw) == code


def test_empty_problems_are_noops(lib):
    assert g(M=0, A=0, B=0, C=0, D=0) == OK
    assert g(N=0, A=0, B=0, C=0, D=0) == OK


def test_valid_arguments_reach_the_device_check(lib):
    # no GPU in this process: a fully valid call ends at the device check
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert g() == NODEV
    assert g(din=F64, dacc=F64, layout=1, lda=64, ldb=64) == NODEV
    # row-major B is provided for every pair
    assert g(layout=1) == NODEV
    assert g(din=I8, dacc=I32, layout=1, lda=64, ldb=64) == NODEV
    assert g(din=F16, dacc=F32, layout=1) == NODEV
    # 16-bit accumulate pairs
    assert g(din=F16, dacc=F16, ldc=64, ldd=64) == NODEV
    assert g(din=BF16, dacc=BF16, layout=1) == NODEV
    assert g(din=BF16, dacc=BF16, ldd=68) == MISAL   # 68 * 2 bytes
    assert g(K=0, A=0, B=0) == NODEV
    assert g(C=0) == NODEV


def i8x(*, M=64, N=64, K=64, A=P, lda=64, an=0, B=P, ldb=64, bn=0, layout=0,
        C=P, ldc=64, D=Q, ldd=64, clamp=1):
    return binding.mma_gemm_i8_ex(M, N, K, A, lda, an, B, ldb, bn, layout, C,
                                  ldc, D, ldd, clamp, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), INVALID), (dict(K=-1), INVALID), (dict(layout=3), INVALID),
    (dict(lda=32), INVALID), (dict(ldb=60), INVALID), (dict(ldc=8), INVALID),
    (dict(D=0), INVALID), (dict(A=0), INVALID), (dict(B=0), INVALID),
    (dict(C=P, D=P, ldc=64, ldd=128), INVALID),
    (dict(A=P + 1), MISAL), (dict(B=P + 8), MISAL), (dict(C=P + 4), MISAL),
    (dict(D=Q + 4), MISAL),
    (dict(lda=72), MISAL),           # 72 bytes is not a 16-byte multiple
    (dict(ldd=66), MISAL),           # 66 * 4 bytes
    # signed x signed without clamp is the plain INT8 product: same checks
    (dict(an=1, bn=1, clamp=0, lda=72), MISAL),
])
def test_i8_ex_argument_errors(lib, kw, code):
    assert i8x(**kw) == code


def test_i8_ex_empty_and_device_check(lib):
    assert i8x(M=0, A=0, B=0, C=0, D=0) == OK
    assert i8x(N=0, A=0, B=0, C=0, D=0, an=1, bn=1, clamp=0) == OK
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    for an in (0, 1):
        for bn in (0, 1):
            for clamp in (0, 1):
                assert i8x(an=an, bn=bn, clamp=clamp) == NODEV
    assert i8x(layout=1) == NODEV
    assert i8x(K=0, A=0, B=0) == NODEV
    assert i8x(C=0) == NODEV


def b(*, din=BF16, dacc=F32, M=16, N=16, K=16, A=P, B=P, C=P, D=Q, ld=16,
      batch=64, G=4, abid=1, blgp=None):
    if blgp is None:
        return binding.mma_gemm_batched(din, dacc, M, N, K, A, ld, B, ld, C, ld,
                                        D, ld, batch, G, abid, None)
    return binding.mma_gemm_batched_ex(din, dacc, M, N, K, A, ld, B, ld, C, ld,
                                       D, ld, batch, G, abid, blgp, None)


@pytest.mark.parametrize("kw,code", [
    (dict(G=3), INVALID), (dict(G=32), INVALID), (dict(G=0), INVALID),
    (dict(abid=4), INVALID), (dict(abid=-1), INVALID),
    (dict(batch=6), INVALID), (dict(batch=-4), INVALID),
    (dict(blgp=8), INVALID), (dict(blgp=-1), INVALID),
    (dict(blgp=3, batch=6, G=2), INVALID),    # patterns need groups of four
    (dict(din=BF16, dacc=I32), UNSUP),
    (dict(din=F16, dacc=BF16), UNSUP),
    (dict(din=I8, dacc=I8), UNSUP),
    (dict(M=-1), INVALID), (dict(ld=8), INVALID),
    (dict(A=0), INVALID), (dict(D=0), INVALID),
    (dict(A=P + 8), MISAL), (dict(C=P + 4), MISAL),
    (dict(M=20, N=20, K=20, ld=20), MISAL),   # 20 * 2 bytes
])
def test_batched_argument_errors(lib, kw, code):
    assert b(**kw) == code


def test_batched_empty_and_device_check(lib):
    assert b(batch=0, A=0, B=0, C=0, D=0) == OK
    assert b(M=0, A=0, B=0, C=0, D=0) == OK
    import torch
    if not torch.cuda.is_available():
        assert b() == NODEV
        assert b(C=0, G=1, abid=0, batch=5) == NODEV
        # generic shapes and every pair are provided
        assert b(M=32, N=48, K=64, ld=64) == NODEV
        assert b(din=I8, dacc=I32, M=32, N=32, K=32, ld=32) == NODEV
        assert b(din=F64, dacc=F64) == NODEV
        assert b(din=BF16, dacc=BF16, blgp=3) == NODEV
        assert b(blgp=7) == NODEV


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_HERE", str(tmp_path))
    with pytest.raises(RuntimeError, match="not built"):
        binding.load()


def test_selftest_wait_timeout_arguments(lib):
    assert binding.mma_selftest_wait_timeout(0, None) == INVALID
    assert binding.mma_selftest_wait_timeout(999, None) == INVALID
    assert binding.mma_selftest_wait_timeout(10 ** 10 + 1, None) == INVALID
    import torch
    if not torch.cuda.is_available():
        assert binding.mma_selftest_wait_timeout(50_000_000, None) == NODEV
