"""Parity of mma_gemm_i8_ex (8-bit integer inputs, each int8 or uint8, with
optional INT32 saturation) with the CPU oracle, bit for bit.

The operation is the iu8 builtin of "RDNA3 dense WMMA builtins" (sections
"INT32-accumulate builtins" and "INT8 and UINT8 inputs"): a_neg / b_neg pick
signed or unsigned inputs, `clamp` saturates the INT32 result on overflow.
On the tensor pipe an unsigned operand is stored shifted by -128 (so every
product keeps the signed bound and K is cut into 1024-deep chunks whose FP32
partial sums stay exact) and the exact product is restored by per-row and
per-column correction terms.  The cases below cover single and many chunks,
ragged tails, the largest stored products of every signedness, results
beyond INT32 in both directions (wrapped and saturated), row-major B (whose
column sums come from the transposing pass), and K long enough that the
saturating mode folds its chunk sums into 64-bit sums several times.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from mixed_precision_dense_02_gb300 import binding, synth

from helpers import GuardedMatrix, check, dev_padded, to_dev

pytestmark = pytest.mark.gpu

I32_MIN, I32_MAX = -(1 << 31), (1 << 31) - 1
SIGNS = [(True, True), (True, False), (False, True), (False, False)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixed_precision_dense_02_gb300 import build
    build.build()
    binding.load()
    yield
    binding.device_status()


def _tag(sa, sb):
    return ("s" if sa else "u") + ("s" if sb else "u")


def run_i8x(A, B, C, *, clamp, b_layout="col", pad=0):
    import torch
    Ad = dev_padded(A, extra=pad)
    Bd = dev_padded(B, extra=pad)
    Cd = None if C is None else dev_padded(C, extra=pad)
    M, N = A.shape[0], (B.shape[0] if b_layout == "col" else B.shape[1])
    Gd = GuardedMatrix(M, N, np.int32, pad=pad + 1)
    out = binding.gemm_i8_ex(Ad, Bd, Cd, Gd.view, clamp=clamp, b_layout=b_layout)
    Gd.verify(f"8-bit {M}x{N}x{A.shape[1]} clamp={clamp} {b_layout}-B D guard")
    return out.cpu().numpy()


SHAPES = [(1, 1, 1), (16, 16, 16), (127, 129, 65), (200, 300, 600),
          (333, 257, 1000), (130, 17, 3), (257, 384, 2100)]


@pytest.mark.parametrize("sa,sb", SIGNS, ids=[_tag(*s) for s in SIGNS])
@pytest.mark.parametrize("clamp", [False, True])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_small_shapes(sa, sb, clamp, M, N, K):
    g = synth.gemm_inputs(f"i8x_{M}_{N}_{K}", "i8", M, N, K, a_signed=sa,
                          b_signed=sb)
    want, ov = oracle.gemm_i8_ex(g.A, g.B, g.C, clamp=clamp)
    assert ov == 0
    got = run_i8x(g.A, g.B, g.C, clamp=clamp, pad=1)
    check("i8", got, want, None, f"{_tag(sa, sb)} clamp={clamp} {M}x{N}x{K}")


@pytest.mark.parametrize("sa,sb", SIGNS, ids=[_tag(*s) for s in SIGNS])
def test_row_major_b_and_no_c(sa, sb):
    M, N, K = 190, 136, 777
    g = synth.gemm_inputs("i8x_row", "i8", M, N, K, a_signed=sa, b_signed=sb,
                          b_layout="row")
    for clamp in (False, True):
        want, _ = oracle.gemm_i8_ex(g.A, g.B, g.C, clamp=clamp, b_layout="row")
        got = run_i8x(g.A, g.B, g.C, clamp=clamp, b_layout="row")
        check("i8", got, want, None, f"{_tag(sa, sb)} row-major B clamp={clamp}")
        want0, _ = oracle.gemm_i8_ex(g.A, g.B, None, clamp=clamp, b_layout="row")
        got0 = run_i8x(g.A, g.B, None, clamp=clamp, b_layout="row")
        check("i8", got0, want0, None, f"{_tag(sa, sb)} C=None clamp={clamp}")


@pytest.mark.parametrize("sa,sb", SIGNS, ids=[_tag(*s) for s in SIGNS])
@pytest.mark.parametrize("b_layout", ["col", "row"])
def test_extreme_values(sa, sb, b_layout):
    """Rows and columns held at the ends of each type's range (-128 and 127
    for int8, 0 and 255 for uint8): the stored products reach 2^14, so each
    1024-deep chunk's FP32 sum reaches 2^24, and the correction terms take
    their largest values."""
    M, N, K = 160, 144, 4096 + 17
    lo_a, hi_a = (-128, 127) if sa else (0, 255)
    lo_b, hi_b = (-128, 127) if sb else (0, 255)
    A = np.full((M, K), lo_a, np.int8 if sa else np.uint8)
    A[1::2] = hi_a
    B = np.full((N, K), lo_b, np.int8 if sb else np.uint8)
    B[1::2] = hi_b
    # a few rows of smaller values so that not every output is the same
    A[::9, : K // 3] = 1
    if b_layout == "row":
        B = np.ascontiguousarray(B.T)
    C = synth.int_uniform(0, 17, M * N, -(1 << 20), 1 << 20).astype(np.int32).reshape(M, N)
    for clamp in (False, True):
        want, _ = oracle.gemm_i8_ex(A, B, C, clamp=clamp, b_layout=b_layout)
        got = run_i8x(A, B, C, clamp=clamp, b_layout=b_layout)
        check("i8", got, want, None,
              f"{_tag(sa, sb)} extreme values B {b_layout} clamp={clamp}")


@pytest.mark.parametrize("sa,sb", SIGNS, ids=[_tag(*s) for s in SIGNS])
def test_overflow_wraps_or_saturates(sa, sb):
    """C near both ends of INT32 with large products: outputs beyond the
    range wrap without clamp and stick at INT32_MIN / INT32_MAX with it."""
    M, N, K = 136, 264, 3000
    g = synth.gemm_inputs("i8x_ovf", "i8", M, N, K, a_signed=sa, b_signed=sb,
                          c_int_range=(I32_MIN, I32_MAX))
    A, B = g.A.copy(), g.B.copy()
    # rows with large same-sign products and rows with large opposite-sign
    # products, so that both ends of the range are crossed
    A[: M // 2] = 127
    B[: N // 2] = 127
    if sa:
        A[M // 2:] = -128
    n_total = 0
    for clamp in (False, True):
        want, ov = oracle.gemm_i8_ex(A, B, g.C, clamp=clamp)
        n_total += ov
        got = run_i8x(A, B, g.C, clamp=clamp)
        check("i8", got, want, None, f"{_tag(sa, sb)} overflow clamp={clamp}")
        if clamp:
            assert np.any(got == I32_MAX)
            if sa:
                assert np.any(got == I32_MIN)
    assert n_total > 0


@pytest.mark.parametrize("sa,sb", [(False, False), (False, True), (True, True)],
                         ids=["uu", "us", "ss"])
def test_long_k_folds_and_saturates_once(sa, sb):
    """K long enough for several 64-bit folds of the chunk sums (one every
    127 chunks).  With signed B the running sum of the constant rows rises
    past 2^31 in the first half of K and falls back in the second, so
    saturating once at the end gives the exact in-range value, not a clamped
    intermediate; with unsigned B it stays beyond 2^31 and saturates."""
    M, N = 72, 80
    K = 2 * 130 * 1024 + 77      # 261 chunks: folds after 127, 254 and 261
    rng = np.random.default_rng(7)
    A = np.full((M, K), 127 if sa else 255, np.int8 if sa else np.uint8)
    if sb:
        B = np.full((N, K), 127, np.int8)
        B[:, K // 2:] = -128
    else:
        B = np.full((N, K), 255, np.uint8)
        B[:, K // 2:] = 0
    # half of the rows/columns random, so that sums are varied
    A[M // 2:] = rng.integers(0 if not sa else -128, 128 if sa else 256,
                              (M - M // 2, K)).astype(A.dtype)
    B[N // 2:] = rng.integers(0 if not sb else -128, 128 if sb else 256,
                              (N - N // 2, K)).astype(B.dtype)
    C = synth.int_uniform(0, 19, M * N, -(1 << 30), 1 << 30).astype(np.int32).reshape(M, N)
    for clamp in (False, True):
        want, _ = oracle.gemm_i8_ex(A, B, C, clamp=clamp)
        got = run_i8x(A, B, C, clamp=clamp)
        check("i8", got, want, None, f"{_tag(sa, sb)} K={K} clamp={clamp}")


def test_full_size_u8_clamp_workload():
    """The 4096^3 unsigned saturating workload, D inside guard bands: every
    one of the 16.8 M outputs against the oracle, bit for bit (the oracle
    needs a few seconds), and the properties that hold at any size for
    nonnegative products: C <= D, and D - C <= K * 255^2 unless D
    saturated."""
    import torch
    name = "gemm_u8_4096_clamp"
    g = synth.workload_gemm_inputs(name)
    A, B, C = to_dev(g.A), to_dev(g.B), to_dev(g.C)
    Gd = GuardedMatrix(g.M, g.N, np.int32)
    D = binding.gemm_i8_ex(A, B, C, Gd.view, clamp=True)
    Gd.verify(f"{name} D guard")
    d64, c64 = D.long(), C.long()
    assert bool((d64 >= c64).all())
    assert bool(((d64 == I32_MAX) | (d64 - c64 <= g.K * 255 * 255)).all())
    assert int((d64 == I32_MAX).sum()) > 0
    want, ov = oracle.gemm_i8_ex(g.A, g.B, g.C, clamp=True)
    check("i8", D.cpu().numpy(), want, None, name)
    assert ov > 0


@pytest.mark.parametrize("K", [32000, 33024])
def test_saturating_modes_either_side_of_the_int32_reach(K):
    """Unsigned x unsigned with clamp: up to about K = 32000 the INT32 sums
    start from the correction terms and never wrap (wide tiles); beyond, the
    chunk sums are folded into 64-bit sums in tensor memory (128-wide
    tiles).  Values at both ends of uint8 push the terms and partial sums
    to their extremes on either side of the switch."""
    M, N = 136, 200
    A = np.zeros((M, K), np.uint8)
    A[1::2] = 255
    A[::5, : K // 2] = 7
    B = np.zeros((N, K), np.uint8)
    B[::2] = 255
    B[::7, K // 3:] = 128
    C = synth.int_uniform(0, 23, M * N, I32_MIN, I32_MAX).astype(np.int32).reshape(M, N)
    for clamp in (False, True):
        want, _ = oracle.gemm_i8_ex(A, B, C, clamp=clamp)
        got = run_i8x(A, B, C, clamp=clamp)
        check("i8", got, want, None, f"uu K={K} clamp={clamp}")


def _routes_to_early_c_saturation(M, N, K, sa, sb, num_sms):
    """Whether a saturating product runs with C added during the chunk
    phase: 224-wide CTA-pair tiles (the library's tile-width choice: at
    least one 256-wide tile per SM, and fewer columns of waves with 224),
    three or more 1024-deep chunks, and K * max|a| * max|b| < 2^30."""
    wide = -(-M // 128) * -(-N // 256)
    if not (N > 128 and wide >= num_sms):
        return False
    pairs, m_units = num_sms // 2, -(-M // 256)
    cost = lambda bn: -(-(m_units * -(-N // bn)) // pairs) * bn
    amax, bmax = (128 if sa else 255), (128 if sb else 255)
    return cost(224) < cost(256) and K > 2048 and K * amax * bmax < (1 << 30)


def _aimed_c(S, seed):
    """C for which S + C lands on the edges of the INT32 range and on the
    values +-2^30 where the wrapped sum changes meaning: each output draws a
    target from the list and takes C = target - S when that C is itself an
    INT32, otherwise a uniform C."""
    targets = np.array([I32_MAX, I32_MAX + 1, I32_MAX + 7, I32_MIN, I32_MIN - 1,
                        I32_MIN - 9, (1 << 30) - 1, 1 << 30, -(1 << 30),
                        -(1 << 30) - 1, I32_MAX + (1 << 30) - 3,
                        I32_MIN - (1 << 30) + 3, 0], np.int64)
    rng = np.random.default_rng(seed)
    t = targets[rng.integers(0, len(targets), S.shape)]
    c = t - S.astype(np.int64)
    fallback = rng.integers(I32_MIN, I32_MAX, S.shape, endpoint=True)
    ok = (c >= I32_MIN) & (c <= I32_MAX)
    return np.where(ok, c, fallback).astype(np.int32)


@pytest.mark.parametrize("sa,sb", SIGNS, ids=[_tag(*s) for s in SIGNS])
@pytest.mark.parametrize("b_layout", ["col", "row"])
def test_saturation_with_c_added_during_the_chunks(sa, sb, b_layout):
    """Saturating products on 224-wide pair tiles: C is added to the INT32
    sums while the chunks run, so the sums hold S + C modulo 2^32 and the
    sign of C decides, at emission, whether the result crossed an end of the
    range.  Outputs are aimed at both ends (in range by one, out of range by
    one), at the values +-2^30 and at the farthest reachable overflows, on a
    ragged shape (edge tiles cut in M and N, three chunks and a tail in K),
    with and without C."""
    import torch
    M, N, K = 2000, 3900, 3000 + 40
    assert _routes_to_early_c_saturation(
        M, N, K, sa, sb, torch.cuda.get_device_properties(0).multi_processor_count)
    g = synth.gemm_inputs("i8x_sate", "i8", M, N, K, a_signed=sa, b_signed=sb,
                          b_layout=b_layout)
    S, ov = oracle.gemm_i8_ex(g.A, g.B, None, clamp=False, b_layout=b_layout)
    assert ov == 0 and int(np.abs(S.astype(np.int64)).max()) < (1 << 30)
    C = _aimed_c(S, 41 + 2 * sa + sb)
    want, n_over = oracle.gemm_i8_ex(g.A, g.B, C, clamp=True, b_layout=b_layout)
    got = run_i8x(g.A, g.B, C, clamp=True, b_layout=b_layout)
    check("i8", got, want, None, f"{_tag(sa, sb)} early-C saturation {b_layout}-B")
    assert n_over > 0 and np.any(got == I32_MAX)
    if sa or sb:
        # products of either sign: the low end is crossed too (with both
        # operands unsigned S >= 0, so S + C never falls below INT32_MIN)
        assert np.any(got == I32_MIN)
    # in-range results on either side of +-2^30 are present too
    assert np.any(got == (1 << 30)) and np.any(got == -(1 << 30))
    got0 = run_i8x(g.A, g.B, None, clamp=True, b_layout=b_layout)
    check("i8", got0, S, None, f"{_tag(sa, sb)} early-C saturation C=None")


@pytest.mark.parametrize("K", [16512, 16513])
def test_early_c_saturation_bound_on_k(K):
    """Unsigned x unsigned: K * 255^2 stays below 2^30 up to K = 16512,
    where C joins the sums during the chunks; from K = 16513 the sums
    keep S exact and C is added at emission.  Rows and columns of 255 give
    the largest S; C is aimed at the range's edges."""
    import torch
    M, N = 2048, 2432
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _routes_to_early_c_saturation(M, N, K, False, False, sms) == (K == 16512)
    rng = np.random.default_rng(K)
    A = rng.integers(0, 256, (M, K), dtype=np.uint8)
    B = rng.integers(0, 256, (N, K), dtype=np.uint8)
    A[::3] = 255
    B[::4] = 255
    S, _ = oracle.gemm_i8_ex(A, B, None, clamp=False)
    C = _aimed_c(S, K)
    want, n_over = oracle.gemm_i8_ex(A, B, C, clamp=True)
    got = run_i8x(A, B, C, clamp=True)
    check("i8", got, want, None, f"uu K={K} saturation")
    # S >= 0 here, so only the top of the range can be crossed
    assert n_over > 0 and np.any(got == I32_MAX)
