"""Edge cases at large extents, against the oracle.

* K = 2^20 with a small output: the K loop runs 16384 stages of 64 and the
  exact INT8 mode 1024 chunks (products of uniform int8 values summed over
  2^20 terms leave the INT32 range, so the wrap-around is exercised too).
* M = 2^20 rows with N = 16, K = 64: 8192 row tiles, more than 50 per SM.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from mixed_precision_dense_02_gb300 import binding, synth

from helpers import check, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixed_precision_dense_02_gb300 import build
    build.build()
    binding.load()
    yield
    binding.device_status()


@pytest.mark.parametrize("dtype_in", ["bf16", "f16", "i8"])
def test_long_k(dtype_in):
    import torch
    M, N, K = 24, 40, 1 << 20
    g = synth.gemm_inputs(f"long_k_{dtype_in}", dtype_in, M, N, K, dist="uniform")
    D = binding.gemm(to_dev(g.A, dtype_in), to_dev(g.B, dtype_in), to_dev(g.C))
    torch.cuda.synchronize()
    if dtype_in == "i8":
        want = oracle.gemm("i8", g.A, g.B, g.C)
        check("i8", D.cpu().numpy(), want, None, "int8 K = 2^20")
        return
    want, ab = oracle.gemm(dtype_in, g.A, g.B, g.C, want_absab=True)
    check(dtype_in, D.cpu().numpy(), want, ab, f"{dtype_in} K = 2^20")


def test_int8_long_k_wraps_like_int32():
    """All products 127 * 127 over K = 2^20 + 64: the exact sum exceeds
    2^31 many times over; D is that sum plus C modulo 2^32."""
    import torch
    M, N, K = 8, 16, (1 << 20) + 64
    A = np.full((M, K), 127, np.int8)
    B = np.full((N, K), 127, np.int8)
    C = np.arange(M * N, dtype=np.int32).reshape(M, N)
    D = binding.gemm(to_dev(A), to_dev(B), to_dev(C))
    torch.cuda.synchronize()
    exact = np.int64(K) * 127 * 127 + C.astype(np.int64)
    want = ((exact + 2 ** 31) % 2 ** 32 - 2 ** 31).astype(np.int32)
    assert np.array_equal(D.cpu().numpy(), want)


def test_tall_m():
    import torch
    M, N, K = 1 << 20, 16, 64
    g = synth.gemm_inputs("tall_m", "bf16", M, N, K, dist="uniform")
    D = binding.gemm(to_dev(g.A, "bf16"), to_dev(g.B, "bf16"), to_dev(g.C))
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.unique(np.append(rng.choice(M, 2000, replace=False), M - 1))
    want, ab = oracle.gemm("bf16", np.ascontiguousarray(g.A[rows]), g.B,
                           np.ascontiguousarray(g.C[rows]), want_absab=True)
    got = D[torch.from_numpy(rows).cuda()].cpu().numpy()
    check("bf16", got, want, ab, "bf16 M = 2^20")
