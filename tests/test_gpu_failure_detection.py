"""Failure detection on the GPU without a fault: a bounded in-kernel wait is
made to run out and the host reads the status.

Every pipeline wait of the kernels (operand stage, accumulator hand-off, C
block) is the same bounded mbarrier wait: when it runs out it records
MMA_ERR_TIMEOUT in the library's device status word and the kernel drains
and returns.  mma_selftest_wait_timeout runs that wait on a barrier nothing
ever signals, with a 50 ms limit.  The test checks that the wait ends by
itself, that mma_device_status reports the timeout exactly once, and that
the context is still usable: a GEMM afterwards gives the oracle's result.
"""
from __future__ import annotations

import time

import numpy as np
import pytest

import oracle
from mixed_precision_dense_02_gb300 import binding, synth

from helpers import check, to_dev

pytestmark = pytest.mark.gpu

MMA_OK, MMA_ERR_TIMEOUT = 0, 5


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixed_precision_dense_02_gb300 import build
    build.build()
    binding.load()
    return torch


def test_bounded_wait_times_out_and_is_reported_once(torch_cuda):
    torch = torch_cuda
    stream = torch.cuda.current_stream().cuda_stream
    assert binding.mma_device_status(stream) == MMA_OK    # start clean
    t0 = time.perf_counter()
    assert binding.mma_selftest_wait_timeout(50_000_000, stream) == MMA_OK
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 0.04 <= waited < 5.0, waited                    # ran out by itself
    assert binding.mma_device_status(stream) == MMA_ERR_TIMEOUT
    assert binding.mma_device_status(stream) == MMA_OK     # cleared
    # the context is still usable
    g = synth.gemm_inputs("after_timeout", "bf16", 200, 136, 264, dist="uniform")
    D = binding.gemm(to_dev(g.A, "bf16"), to_dev(g.B, "bf16"), to_dev(g.C))
    torch.cuda.synchronize()
    want, ab = oracle.gemm("bf16", g.A, g.B, g.C, want_absab=True)
    check("bf16", D.cpu().numpy(), want, ab, "GEMM after a timeout")
    assert binding.mma_device_status(stream) == MMA_OK


def test_device_status_raises_after_timeout(torch_cuda):
    torch = torch_cuda
    stream = torch.cuda.current_stream().cuda_stream
    assert binding.mma_selftest_wait_timeout(2_000_000, stream) == MMA_OK
    with pytest.raises(binding.MMAError) as e:
        binding.device_status()
    assert e.value.status == MMA_ERR_TIMEOUT
    binding.device_status()    # cleared: no raise


def test_scratch_buffer_shared_by_two_streams(torch_cuda):
    """Tensor-pipe INT8 products on two streams share the library's scratch
    buffer; the library orders them by an event, and growing the buffer for
    a larger problem waits for its previous user.  Enqueued back to back
    without host synchronisation, both results must be exact."""
    torch = torch_cuda
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    g1 = synth.gemm_inputs("streams_a", "i8", 512, 512, 4096)     # 2^30 MACs
    g2 = synth.gemm_inputs("streams_b", "i8", 640, 768, 6144)     # more scratch
    ins = [(to_dev(g.A), to_dev(g.B), to_dev(g.C)) for g in (g1, g2)]
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        for (A, B, C), s in zip(ins, (s1, s2)):
            with torch.cuda.stream(s):
                outs.append(binding.gemm(A, B, C))
    torch.cuda.synchronize()
    binding.device_status()
    for k, g in enumerate((g1, g2)):
        want = oracle.gemm("i8", g.A, g.B, g.C)
        for rep in range(3):
            got = outs[2 * rep + k].cpu().numpy()
            assert np.array_equal(got, want), (k, rep)


@pytest.mark.parametrize("cluster", [1, 2])
def test_gemm_kernel_abort_path(torch_cuda, cluster):
    """The tcgen05 GEMM kernel itself, on single CTAs and on a CTA pair, with
    its producer issuing no loads and its waits limited to 50 ms: the call
    returns, the kernel ends by itself, the timeout is reported exactly once,
    its output buffer is untouched, and the tensor memory it held was freed:
    the same kernel shapes then run twice more and match the oracle."""
    torch = torch_cuda
    stream = torch.cuda.current_stream().cuda_stream
    assert binding.mma_device_status(stream) == MMA_OK
    dev = torch.device("cuda:0")
    A = torch.zeros((256, 256), dtype=torch.bfloat16, device=dev)
    B = torch.zeros_like(A)
    D = torch.full((256, 256), 7.0, dtype=torch.float32, device=dev)
    for _ in range(2):
        t0 = time.time()
        assert binding.mma_selftest_gemm_abort(cluster, 50_000_000, A.data_ptr(),
                                               B.data_ptr(), D.data_ptr(), stream) == MMA_OK
        torch.cuda.synchronize()
        assert time.time() - t0 < 10.0
        assert binding.mma_device_status(stream) == MMA_ERR_TIMEOUT
        assert binding.mma_device_status(stream) == MMA_OK
    assert bool((D == 7.0).all())
    # afterwards: products on single CTAs (256^3) and on CTA pairs
    # (2048 x 2560 x 512, a full wave of pair tiles) are exact again
    for (M, N, K) in [(256, 256, 256), (2048, 2560, 512)]:
        g = synth.gemm_inputs(f"abort_after_{M}", "bf16", M, N, K, dist="uniform")
        out = binding.gemm(to_dev(g.A, "bf16"), to_dev(g.B, "bf16"), to_dev(g.C))
        torch.cuda.synchronize()
        rows = np.arange(0, M, 7)
        want, ab = oracle.gemm("bf16", np.ascontiguousarray(g.A[rows]), g.B,
                               np.ascontiguousarray(g.C[rows]), want_absab=True)
        check("bf16", out.cpu().numpy()[rows], want, ab, f"after abort {M}x{N}x{K}")
    assert binding.mma_device_status(stream) == MMA_OK
