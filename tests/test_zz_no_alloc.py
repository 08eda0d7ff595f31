"""The allocation-free INT8 entry point, checked against the regular one
and against the CPU oracle.

mma_gemm_i8_noalloc is for callers that cannot let a library allocate device
memory: programs whose own pool allocator has already reserved the memory
they may use, and services that forbid cudaMalloc/cudaFree after start-up
because those calls can stall the whole device.  Its scratch is a fixed
array in the library's device image instead of a buffer grown with
cudaMalloc.  Here it is called through the C ABI several times in a row:

* on two different problems (the first at the exact scratch limit, the
  second ragged and smaller), each INT32 result equal bit for bit to what
  mma_gemm returns for the same inputs and to the oracle over the whole
  output;
* after a call that fills the whole scratch with nonzero values, on a
  problem whose K is not a multiple of 8, so the scratch rows carry stale
  padding columns between K and their 16-byte-rounded width: nothing may
  read them;
* one step past the limit, which must be refused without launching.

Every output sits in a canary-filled buffer whose guard rows and padding
columns must come back untouched.  This file is named to be collected
last, so that a run stopping at the first failure has already run every
other test; it also passes on its own.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from mixed_precision_dense_02_gb300 import binding, synth

from helpers import GuardedMatrix, check, dev_padded

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
        Gd = GuardedMatrix(M, N, np.int32)
        assert _noalloc(torch, A, B, C, Gd.view) == 0
        ref = binding.gemm(A, B, C)
        torch.cuda.synchronize()
        binding.device_status()
        Gd.verify(f"noalloc {M}x{N}x{K} D guard")
        assert torch.equal(Gd.view, ref), f"{M}x{N}x{K}: differs from mma_gemm"
        check("i8", Gd.view.cpu().numpy(), oracle.gemm("i8", g.A, g.B, g.C), None,
              f"noalloc {M}x{N}x{K} against the oracle")


def test_noalloc_ignores_stale_scratch_beyond_k(torch_cuda):
    torch = torch_cuda
    dev = torch.device("cuda:0")
    # fill the whole scratch with BF16 -1 (every row at its full width)
    M = N = K = 4096
    A = torch.full((M, K), -1, dtype=torch.int8, device=dev)
    B = torch.full((N, K), -1, dtype=torch.int8, device=dev)
    C = torch.zeros((M, N), dtype=torch.int32, device=dev)
    D = torch.empty((M, N), dtype=torch.int32, device=dev)
    assert _noalloc(torch, A, B, C, D) == 0
    torch.cuda.synchronize()
    assert bool((D == K).all())
    # K = 1003: scratch rows are 1008 wide, columns 1003..1007 stale
    M, N, K = 300, 520, 1003
    g = synth.gemm_inputs("noalloc_k1003", "i8", M, N, K)
    A2, B2, C2 = dev_padded(g.A), dev_padded(g.B), dev_padded(g.C)
    assert A2.stride(0) == 1008 and B2.stride(0) == 1008
    Gd = GuardedMatrix(M, N, np.int32)
    assert _noalloc(torch, A2, B2, C2, Gd.view) == 0
    torch.cuda.synchronize()
    binding.device_status()
    Gd.verify("noalloc K=1003 D guard")
    check("i8", Gd.view.cpu().numpy(), oracle.gemm("i8", g.A, g.B, g.C), None,
          "noalloc K=1003 after a full-scratch call")


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
