"""The allocation-free INT8 entry point, checked against the regular one.

mma_gemm_i8_noalloc is for callers that cannot let a library allocate device
memory: programs whose own pool allocator has already reserved the memory
they may use, and services that forbid cudaMalloc/cudaFree after start-up
because those calls can stall the whole device.  Its scratch is a fixed
array in the library's device image instead of a buffer grown with
cudaMalloc.  Here it is called through the C ABI twice in a row, on two
different problems (the first at the exact scratch limit, the second ragged
and smaller, so stale scratch contents from the first would show), and each
INT32 result must equal bit for bit what mma_gemm returns for the same
inputs.  A problem one step past the limit must be refused.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
from __future__ import annotations

import numpy as np
import pytest

from mixed_precision_dense_02_gb300 import binding, synth

from helpers import dev_padded

pytestmark = pytest.mark.gpu

MMA_ERR_UNSUPPORTED = 2


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixed_precision_dense_02_gb300 import build
    build.build()
    binding.load()
    return torch


def _noalloc(torch, A, B, C, D):
    M, K = A.shape
    N = B.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    return binding.mma_gemm_i8_noalloc(M, N, K, A.data_ptr(), A.stride(0),
                                       B.data_ptr(), B.stride(0), C.data_ptr(),
                                       C.stride(0), D.data_ptr(), D.stride(0),
                                       stream)


def test_noalloc_matches_mma_gemm_on_two_calls_in_a_row(torch_cuda):
    torch = torch_cuda
    cases = [(4096, 4096, 4096),   # (M + N) * K * 2 bytes = the 64 MiB limit
             (777, 1200, 1000)]    # ragged tiles, K tail, smaller footprint
    for M, N, K in cases:
        g = synth.gemm_inputs(f"noalloc_{M}_{N}_{K}", "i8", M, N, K)
        # leading dimensions padded to 16-byte multiples (K = 1000 int8
        # rows are not), as the entry point requires
        A = dev_padded(g.A)
        B = dev_padded(g.B)
        C = dev_padded(g.C)
        D = dev_padded(np.full((M, N), -7, np.int32), extra=1)
        assert _noalloc(torch, A, B, C, D) == 0
        ref = binding.gemm(A, B, C)
        torch.cuda.synchronize()
        assert ref.data_ptr() != D.data_ptr()
        binding.device_status()
        assert torch.equal(D, ref), f"{M}x{N}x{K}: differs from mma_gemm"
        # and the INT32 values are the exact ones (spot check against Python ints)
        i, j = M - 1, N - 1
        exact = int(np.dot(g.A[i].astype(np.int64), g.B[j].astype(np.int64))) + int(g.C[i, j])
        assert int(D[i, j]) == exact


def test_noalloc_refuses_problems_beyond_its_scratch(torch_cuda):
    torch = torch_cuda
    dev = torch.device("cuda:0")
    M, N, K = 4096, 4104, 4096    # 8 more rows of B than fit
    A = torch.zeros((M, K), dtype=torch.int8, device=dev)
    B = torch.zeros((N, K), dtype=torch.int8, device=dev)
    C = torch.zeros((M, N), dtype=torch.int32, device=dev)
    D = torch.full((M, N), 5, dtype=torch.int32, device=dev)
    assert _noalloc(torch, A, B, C, D) == MMA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((D == 5).all())   # nothing was launched
