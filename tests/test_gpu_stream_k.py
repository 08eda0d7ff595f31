"""Parity of the stream-K tcgen05 GEMM (FP16/BF16 -> FP32 with fewer than
half as many 128 x 128 output tiles as SMs and deep K; the tiles' K steps
are split over every SM and the pieces of a tile are added in a fixed order
by the CTA holding its first piece) with the CPU oracle, through the C ABI.

Covers ragged M, N and K, tiles split into two, three and up to ~150
pieces, C absent and C = D in place, a column count whose rows end off a
16-byte boundary, run-to-run identical results, and products that the
automatic choice keeps on the regular kernel but MMA_GB300_STREAMK=1 sends
here (several whole tiles per CTA between the split ones, and the tall
16384 x 128 x 4096 shape).  Products at least 256 wide in M and N run on
CTA pairs with 256 x 256 tiles (their partial sums passed between the
CTAs of the same rank, and with whole ranges per tile summed by all of
the tile's pairs, each a share); MMA_GB300_STREAMK_CL=1 sends them to
single CTAs instead.  Every output sits inside guard bands.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from mixed_precision_dense_02_gb300 import binding, synth

from helpers import GuardedMatrix, check, dev_padded, to_dev

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


def run(g, *, use_c=True, inplace=False, pad=1):
    A = dev_padded(g.A, g.dtype_in)
    B = dev_padded(g.B, g.dtype_in)
    if inplace:
        Gd = GuardedMatrix(g.M, g.N, np.float32, init=g.C, pad=pad)
        C = Gd.view
    else:
        Gd = GuardedMatrix(g.M, g.N, np.float32, pad=pad)
        C = dev_padded(g.C) if use_c else None
    binding.gemm(A, B, C, Gd.view)
    Gd.verify(f"stream-K {g.dtype_in} {g.M}x{g.N}x{g.K} D guard")
    return Gd.view.cpu().numpy()


# (M, N, K): tiles < 76 (half the SMs) and deep K, so the automatic choice
# splits K
SHAPES = [
    (4096, 128, 4096),    # two or three pieces per tile
    (1000, 136, 4000),    # ragged M, N and K
    (300, 130, 8200),     # rows of 130 FP32 (off a 16-byte boundary)
    (128, 128, 65536),    # one tile split over every SM
    (777, 200, 1536),
]


# M and N >= 256: CTA pairs on 256 x 256 tiles (ragged in M, N and K)
PAIR_SHAPES = [
    (1024, 768, 8192),    # 12 pair tiles, 6 whole ranges each: the
                          # tile's pairs finish it together
    (1200, 700, 8200),    # 15 ragged pair tiles, 5 ranges each
    (512, 768, 6000),
    (300, 520, 9000),     # tiles half outside M, a ragged last column tile
    (1000, 300, 4000),
    (256, 256, 16384),    # one pair tile split over every pair
]


@pytest.mark.parametrize("dtype_in", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", SHAPES + PAIR_SHAPES)
def test_stream_k_shapes(dtype_in, M, N, K):
    g = synth.gemm_inputs(f"sk_{M}_{N}_{K}", dtype_in, M, N, K, dist="normal")
    want, ab = oracle.gemm(dtype_in, g.A, g.B, g.C, want_absab=True)
    check(dtype_in, run(g), want, ab, f"stream-K {dtype_in} {M}x{N}x{K}")


def test_stream_k_no_c_in_place_and_repeatable():
    M, N, K = 1000, 136, 4000
    g = synth.gemm_inputs("sk_modes", "bf16", M, N, K, dist="uniform")
    want, ab = oracle.gemm("bf16", g.A, g.B, g.C, want_absab=True)
    first = run(g)
    check("bf16", first, want, ab, "stream-K")
    # the pieces are added in a fixed order: identical bits on a rerun
    assert np.array_equal(first.view(np.uint32), run(g).view(np.uint32))
    check("bf16", run(g, inplace=True), want, ab, "stream-K in place")
    want0, ab0 = oracle.gemm("bf16", g.A, g.B, np.zeros_like(g.C), want_absab=True)
    check("bf16", run(g, use_c=False), want0, ab0, "stream-K, C = NULL")


@pytest.mark.parametrize("M,N,K", [(520, 600, 5000), (1200, 700, 8200)])
def test_stream_k_pairs_no_c_in_place_and_repeatable(M, N, K):
    """Single CTAs (9 pair tiles would be too few for pairs) and pairs whose
    tiles are finished by all of their units, each a share."""
    g = synth.gemm_inputs(f"skp_modes_{M}", "bf16", M, N, K, dist="uniform")
    want, ab = oracle.gemm("bf16", g.A, g.B, g.C, want_absab=True)
    first = run(g)
    check("bf16", first, want, ab, "stream-K pairs")
    assert np.array_equal(first.view(np.uint32), run(g).view(np.uint32))
    check("bf16", run(g, inplace=True), want, ab, "stream-K pairs in place")
    want0, ab0 = oracle.gemm("bf16", g.A, g.B, np.zeros_like(g.C), want_absab=True)
    check("bf16", run(g, use_c=False), want0, ab0, "stream-K pairs, C = NULL")


def test_full_size_skinny_repeatable():
    """The skinny workload (its rows spread over every SM) twice: the whole
    output identical bit for bit."""
    import torch
    name = "gemm_bf16_skinny_16384x128x4096"
    w = synth.WORKLOADS[name]
    g = synth.gemm_inputs(name, "bf16", w["M"], w["N"], w["K"], dist=w.get("dist", "normal"))
    A, B, C = to_dev(g.A, "bf16"), to_dev(g.B, "bf16"), to_dev(g.C)
    D1 = binding.gemm(A, B, C)
    D2 = binding.gemm(A, B, C)
    torch.cuda.synchronize()
    assert torch.equal(D1.view(torch.int32), D2.view(torch.int32))


_FORCED_SCRIPT = """
import sys, numpy as np, torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + '/tests']
from mixed_precision_dense_02_gb300 import binding, synth
from helpers import GuardedMatrix, dev_padded
binding.load()
out = {}
for (M, N, K) in [(2100, 2300, 3000), (512, 640, 192), (256, 256, 64), (16384, 128, 4096)]:
    g = synth.gemm_inputs(f'skf_{M}_{N}_{K}', 'bf16', M, N, K, dist='uniform')
    Gd = GuardedMatrix(M, N, np.float32)
    binding.gemm(dev_padded(g.A, 'bf16'), dev_padded(g.B, 'bf16'), dev_padded(g.C), Gd.view)
    Gd.verify('forced stream-K guard')
    out[f'{M}_{N}_{K}'] = Gd.view.cpu().numpy()
binding.device_status()
np.savez(sys.argv[2], **out)
"""


_SINGLE_SCRIPT = """
import sys, numpy as np, torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + '/tests']
from mixed_precision_dense_02_gb300 import binding, synth
from helpers import GuardedMatrix, dev_padded
binding.load()
M, N, K = 1024, 768, 8192
g = synth.gemm_inputs(f'sk_{M}_{N}_{K}', 'bf16', M, N, K, dist='normal')
Gd = GuardedMatrix(M, N, np.float32)
binding.gemm(dev_padded(g.A, 'bf16'), dev_padded(g.B, 'bf16'), dev_padded(g.C), Gd.view)
Gd.verify('single-CTA stream-K guard')
binding.device_status()
np.save(sys.argv[2], Gd.view.cpu().numpy())
"""


def test_stream_k_pairs_and_single_ctas_agree_with_oracle(tmp_path):
    """The same product on pairs (automatic) and, in a child process with
    MMA_GB300_STREAMK_CL=1, on single CTAs: both within the tolerance of
    the oracle (their sums are split differently, so their bits differ)."""
    import os
    import pathlib
    import subprocess
    import sys
    root = str(pathlib.Path(__file__).resolve().parents[1])
    out = tmp_path / "single.npy"
    env = dict(os.environ, MMA_GB300_STREAMK_CL="1")
    r = subprocess.run([sys.executable, "-c", _SINGLE_SCRIPT, root, str(out)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    M, N, K = 1024, 768, 8192
    g = synth.gemm_inputs(f"sk_{M}_{N}_{K}", "bf16", M, N, K, dist="normal")
    want, ab = oracle.gemm("bf16", g.A, g.B, g.C, want_absab=True)
    check("bf16", np.load(out), want, ab, "stream-K single CTAs")
    check("bf16", run(g), want, ab, "stream-K pairs")


_PAIRS_SCRIPT = """
import sys, numpy as np, torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + '/tests']
from mixed_precision_dense_02_gb300 import binding, synth
from helpers import GuardedMatrix, dev_padded
binding.load()
out = {}
for (M, N, K) in [(256, 512, 16384), (300, 260, 5000), (512, 256, 3000)]:
    g = synth.gemm_inputs(f'skq_{M}_{N}_{K}', 'bf16', M, N, K, dist='uniform')
    Gd = GuardedMatrix(M, N, np.float32)
    binding.gemm(dev_padded(g.A, 'bf16'), dev_padded(g.B, 'bf16'), dev_padded(g.C), Gd.view)
    Gd.verify('forced pairs guard')
    out[f'{M}_{N}_{K}'] = Gd.view.cpu().numpy()
binding.device_status()
np.savez(sys.argv[2], **out)
"""


def test_stream_k_forced_pairs_many_ranges(tmp_path):
    """MMA_GB300_STREAMK_CL=2 (child process) on products with one to two
    pair tiles, so each tile is cut into 25 to 76 whole ranges and has more
    ranges than finishing items (some units add nothing), ragged in M, N
    and K; against the oracle."""
    import os
    import pathlib
    import subprocess
    import sys
    root = str(pathlib.Path(__file__).resolve().parents[1])
    out = tmp_path / "forced_pairs.npz"
    env = dict(os.environ, MMA_GB300_STREAMK_CL="2")
    r = subprocess.run([sys.executable, "-c", _PAIRS_SCRIPT, root, str(out)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = np.load(out)
    for (M, N, K) in [(256, 512, 16384), (300, 260, 5000), (512, 256, 3000)]:
        g = synth.gemm_inputs(f"skq_{M}_{N}_{K}", "bf16", M, N, K, dist="uniform")
        want, ab = oracle.gemm("bf16", g.A, g.B, g.C, want_absab=True)
        check("bf16", got[f"{M}_{N}_{K}"], want, ab, f"forced pairs {M}x{N}x{K}")


def test_stream_k_forced_on_many_tiles(tmp_path):
    """MMA_GB300_STREAMK=1 (read once per process, so in a child process):
    products with more tiles than SMs (whole tiles between each CTA's split
    ones) and with few K steps per CTA, against the oracle here."""
    import os
    import pathlib
    import subprocess
    import sys
    root = str(pathlib.Path(__file__).resolve().parents[1])
    out = tmp_path / "forced_sk.npz"
    env = dict(os.environ, MMA_GB300_STREAMK="1")
    r = subprocess.run([sys.executable, "-c", _FORCED_SCRIPT, root, str(out)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = np.load(out)
    for (M, N, K) in [(2100, 2300, 3000), (512, 640, 192), (256, 256, 64),
                      (16384, 128, 4096)]:
        g = synth.gemm_inputs(f"skf_{M}_{N}_{K}", "bf16", M, N, K, dist="uniform")
        rows = np.unique(np.append(np.random.default_rng(3).choice(M, 100, replace=False), M - 1))
        want, ab = oracle.gemm("bf16", np.ascontiguousarray(g.A[rows]), g.B,
                               np.ascontiguousarray(g.C[rows]), want_absab=True)
        check("bf16", got[f"{M}_{N}_{K}"][rows], want, ab, f"forced stream-K {M}x{N}x{K}")
