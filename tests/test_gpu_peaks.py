"""The per-pipe issue-rate probes (mma_peak_probe) through the C ABI: each
kind runs on every SM and reports its operation count; the rate it gives
(operations / CUDA-event time) must be positive and within a wide band
around the pipe's nominal figure, and the probes leave the device status
clean.  Invalid kinds and iteration counts are refused before any launch.
"""
from __future__ import annotations

import pytest

from mixed_precision_dense_02_gb300 import binding

pytestmark = pytest.mark.gpu

MMA_ERR_INVALID_ARG = 1

# kind, iterations, band of plausible rates (10^12 operations per second):
# dense BF16 tensor pipe ~2250 nominal, FP64 ~1.25, the warp-level INT8
# pipe ~150 measured, scalar FP64 ~1.25
CASES = [(binding.MMA_PEAK_TC_F16, 4096, (200.0, 4000.0)),
         (binding.MMA_PEAK_DMMA, 200, (0.1, 20.0)),
         (binding.MMA_PEAK_IMMA, 2000, (10.0, 2000.0)),
         (binding.MMA_PEAK_DFMA, 2000, (0.1, 20.0))]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixed_precision_dense_02_gb300 import build
    build.build()
    binding.load()


@pytest.mark.parametrize("kind,iters,band", CASES)
def test_probe_rate_is_plausible(kind, iters, band):
    import torch
    stream = torch.cuda.current_stream()
    st, _ = binding.mma_peak_probe(kind, 16, stream.cuda_stream)  # warm-up
    assert st == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    st, ops = binding.mma_peak_probe(kind, iters, stream.cuda_stream)
    e1.record(stream)
    e1.synchronize()
    assert st == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ops > 0 and ops % sms == 0
    rate = ops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    assert band[0] < rate < band[1], rate
    binding.device_status()


def test_probe_rejects_bad_arguments():
    import torch
    s = torch.cuda.current_stream().cuda_stream
    assert binding.mma_peak_probe(9, 10, s)[0] == MMA_ERR_INVALID_ARG
    assert binding.mma_peak_probe(binding.MMA_PEAK_DMMA, 0, s)[0] == MMA_ERR_INVALID_ARG
    assert binding.mma_peak_probe(binding.MMA_PEAK_TC_F16, (1 << 21) + 1, s)[0] == \
        MMA_ERR_INVALID_ARG
