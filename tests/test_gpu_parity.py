"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small and ragged shapes are compared element by element over the whole
output; the full-size workloads are compared on random row x column blocks
of the output (the oracle computes each block from the gathered rows of A
and columns of B), except the batched workload, which is compared in full.
Tolerances are in tests/helpers.py.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from mixed_precision_dense_02_gb300 import binding, synth

from helpers import (TOL, GuardedBatch, GuardedMatrix, check, check16, decode16, dev_padded,
                     oracle_ref, to_dev)

pytestmark = pytest.mark.gpu

OUT_NP = {"f16": np.float32, "bf16": np.float32, "i8": np.int32, "f64": np.float64}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixed_precision_dense_02_gb300 import build
    build.build()
    binding.load()
    yield
    binding.device_status()


def run_gemm(g, *, pad=0, use_c=True, inplace=False):
    """Run the GPU GEMM for GemmInputs g with padded leading dimensions; D
    (or C = D in place) sits in a canary-filled buffer whose guard rows and
    padding columns must come back untouched."""
    A = dev_padded(g.A, g.dtype_in, extra=pad)
    B = dev_padded(g.B, g.dtype_in, extra=pad)
    out_dt = OUT_NP[g.dtype_in]
    if inplace:
        G = GuardedMatrix(g.M, g.N, out_dt, init=g.C, pad=pad + 1)
        C = G.view
    else:
        G = GuardedMatrix(g.M, g.N, out_dt, pad=pad + 1)
        C = dev_padded(g.C, extra=pad) if use_c else None
    out = binding.gemm_ex(A, B, C, G.view, b_layout=g.b_layout)
    G.verify(f"{g.dtype_in} {g.M}x{g.N}x{g.K} {g.b_layout}-B D guard")
    return out.cpu().numpy()


SHAPES = [(1, 1, 1), (16, 16, 16), (128, 128, 64), (127, 129, 65),
          (256, 256, 256), (200, 300, 100), (333, 257, 1000), (64, 520, 40),
          (1000, 136, 520), (130, 17, 3)]


@pytest.mark.parametrize("dtype_in", ["f16", "bf16", "i8", "f64"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_small_shapes(dtype_in, M, N, K):
    g = synth.gemm_inputs(f"par_{M}_{N}_{K}", dtype_in, M, N, K, dist="uniform")
    want, ab = oracle_ref(g)
    check(dtype_in, run_gemm(g), want, ab, f"{dtype_in} {M}x{N}x{K}")


@pytest.mark.parametrize("dtype_in", ["f16", "bf16", "i8", "f64"])
def test_padding_no_c_and_in_place(dtype_in):
    M, N, K = 260, 392, 328
    g = synth.gemm_inputs("par_pad", dtype_in, M, N, K, dist="normal")
    want, ab = oracle_ref(g)
    check(dtype_in, run_gemm(g, pad=3), want, ab, "padded")
    check(dtype_in, run_gemm(g, inplace=True), want, ab, "in place")
    g0 = synth.GemmInputs(dtype_in, M, N, K, g.A, g.B, np.zeros_like(g.C))
    want0, ab0 = oracle_ref(g0)
    check(dtype_in, run_gemm(g, use_c=False), want0, ab0, "C = NULL")


@pytest.mark.parametrize("dtype_in", ["f16", "bf16", "i8", "f64"])
def test_row_major_b(dtype_in):
    """mma_gemm_ex with B stored K x N row-major (FP64 reads it directly, the
    others transpose it first into the library's scratch buffer)."""
    for (M, N, K) in [(1, 1, 1), (65, 63, 17), (256, 192, 300), (300, 520, 1000),
                      (1024, 768, 2048)]:
        g = synth.gemm_inputs(f"par_row_{dtype_in}_{M}", dtype_in, M, N, K,
                              b_layout="row")
        want, ab = oracle_ref(g)
        check(dtype_in, run_gemm(g, pad=1), want, ab, f"{dtype_in} row-B {M}x{N}x{K}")
    g0 = synth.GemmInputs(dtype_in, M, N, K, g.A, g.B, np.zeros_like(g.C), "row")
    want0, ab0 = oracle_ref(g0)
    check(dtype_in, run_gemm(g, use_c=False), want0, ab0, "row-B, C = NULL")
    check(dtype_in, run_gemm(g, inplace=True), want, ab, "row-B, in place")


@pytest.mark.parametrize("dtype_in", ["f16", "bf16", "i8", "f64"])
def test_k_zero_gives_c(dtype_in):
    M, N = 37, 44
    g = synth.gemm_inputs("par_k0", dtype_in, M, N, 8)
    g = synth.GemmInputs(dtype_in, M, N, 0, g.A[:, :0], g.B[:, :0], g.C)
    import torch
    C = to_dev(g.C)
    A = to_dev(np.zeros((M, 8), g.A.dtype), dtype_in)[:, :0]
    B = to_dev(np.zeros((N, 8), g.B.dtype), dtype_in)[:, :0]
    D = binding.gemm(A, B, C)
    torch.cuda.synchronize()
    assert np.array_equal(D.cpu().numpy(), g.C)


@pytest.mark.parametrize("dtype_in", ["f16", "bf16", "i8"])
def test_all_ones_closed_form_exact(dtype_in):
    """A = B = 1: D_ij = K + C_ij.  Integer partial sums below 2^24 are exact
    in FP32, so FP16/BF16 must match bit for bit as well."""
    M, N, K = 300, 260, 4096
    one = {"f16": np.uint16(0x3C00), "bf16": np.uint16(0x3F80), "i8": np.int8(1)}[dtype_in]
    A = np.full((M, K), one)
    B = np.full((N, K), one)
    g0 = synth.gemm_inputs("par_ones", dtype_in, M, N, 16)
    C = g0.C
    if dtype_in != "i8":
        C = np.round(C * 64).astype(np.float32)  # integers: K + C exact
    g = synth.GemmInputs(dtype_in, M, N, K, A, B, C)
    got = run_gemm(g)
    assert np.array_equal(got, (C.astype(np.float64) + K).astype(got.dtype))


@pytest.mark.parametrize("dtype_in", ["bf16", "f64"])
def test_identity_closed_form(dtype_in):
    """B = I: D = A + C (one rounding)."""
    n = 384
    g = synth.gemm_inputs("par_eye", dtype_in, n, n, n)
    if dtype_in == "bf16":
        eye = np.where(np.eye(n, dtype=bool), np.uint16(0x3F80), np.uint16(0)).astype(np.uint16)
        a = synth.bf16_bits_to_f32(g.A).astype(np.float64)
    else:
        eye = np.eye(n)
        a = g.A
    g = synth.GemmInputs(dtype_in, n, n, n, g.A, eye, g.C)
    got = run_gemm(g)
    assert np.array_equal(got, (a + g.C.astype(np.float64)).astype(got.dtype))


@pytest.mark.parametrize("dtype_in", ["bf16", "i8"])
def test_transpose_property(dtype_in):
    """(A B + C)^T computed as B^T A^T + C^T agrees within tolerance."""
    M, N, K = 384, 272, 520
    g = synth.gemm_inputs("par_T", dtype_in, M, N, K)
    gT = synth.GemmInputs(dtype_in, N, M, K, g.B, g.A, np.ascontiguousarray(g.C.T))
    want, ab = oracle_ref(g)
    check(dtype_in, run_gemm(gT).T, want, None if ab is None else ab, "transposed")


def test_i8_extremes_exact():
    M, N, K = 256, 256, 4096
    C = synth.int_uniform(0, 3, M * N, -(1 << 20), 1 << 20).astype(np.int32).reshape(M, N)
    for a, b in ((-128, -128), (-128, 127), (127, 127)):
        g = synth.GemmInputs("i8", M, N, K, np.full((M, K), a, np.int8),
                             np.full((N, K), b, np.int8), C)
        assert np.array_equal(run_gemm(g), C + K * a * b)


def test_i8_every_value_through_the_tensor_pipe():
    """A[i][k] = int8(i + k) holds all 256 int8 values in every row; with
    B = I (256 x 256, on the tensor-pipe path) D = A + C exactly."""
    n = 256
    A = ((np.arange(n)[:, None] + np.arange(n)[None, :]) % 256).astype(np.uint8).view(np.int8)
    eye = np.eye(n, dtype=np.int8)
    C = synth.int_uniform(0, 11, n * n, -(1 << 20), 1 << 20).astype(np.int32).reshape(n, n)
    g = synth.GemmInputs("i8", n, n, n, A, eye, C)
    assert np.array_equal(run_gemm(g), A.astype(np.int32) + C)
    g = synth.GemmInputs("i8", n, n, n, eye, np.ascontiguousarray(A.T), C)
    assert np.array_equal(run_gemm(g), A.astype(np.int32) + C)


def test_i8_exact_large_partial_sums_then_unit_steps():
    """Each 1024-deep K chunk first accumulates 512 products of 2^14 (partial
    sum 2^23) and then 512 products of +-1, so every unit step must land
    exactly on a value near 2^23..2^24 -- where FP32 has no spare bits."""
    M, N, K = 256, 384, 4096
    rng = np.random.default_rng(77)
    A = rng.choice(np.array([-1, 1], np.int8), size=(M, K))
    B = rng.choice(np.array([-1, 1], np.int8), size=(N, K))
    for k0 in range(0, K, 1024):
        A[:, k0:k0 + 512] = -128
        B[:, k0:k0 + 512] = -128
    A[::7, 1024:1536] = 127          # mixed signs in some rows
    C = synth.int_uniform(0, 5, M * N, -(1 << 20), 1 << 20).astype(np.int32).reshape(M, N)
    g = synth.GemmInputs("i8", M, N, K, A, B, C)
    want, _ = oracle_ref(g)
    check("i8", run_gemm(g), want, None, "large partial sums then unit steps")


def _mixed_step_operands(M, N, K, seed):
    """8-bit operands whose 16-deep K steps mix 2^14-sized products with
    +-1 products while each 1024-deep chunk's running sum climbs towards
    the exact-FP32 limit 2^24.  Rows of A and columns of B come in four
    families (index mod 4); a family fixes where the unit entries sit in
    every chunk and the value of all other entries:
      0: all steps 2^14 products, then the last 16 steps of the chunk each
         hold one +-1 product (chunk sum 2^24 - 16 * 2^14 +- 16);
      1: one +-1 product in every step (chunk sum 64 * 15 * 2^14 +- 64);
      2: a single +-1 product at step 37 (chunk sum 2^24 - 2^14 +- 1, the
         closest to 2^24 a unit product allows: every int8 product other
         than (-128)^2 is at least 128 below 2^14, so a chunk of 1024
         products reaches no integer strictly between 2^24 - 128 and 2^24);
      3: as 1, with B's other entries +127, so the sums fall towards
         -64 * 15 * 16256.
    Rows and columns of different families meet at +-128 products as
    well.  The unit signs are random per entry."""
    rng = np.random.default_rng(seed)
    step = np.arange(64)
    units = [
        np.concatenate([np.zeros(48 * 16, bool),
                        np.eye(16, dtype=bool)[(step[48:] * 5) % 16].ravel()]),
        np.eye(16, dtype=bool)[(step * 3) % 16].ravel(),
        np.zeros(1024, bool),
        np.eye(16, dtype=bool)[(step * 7 + 1) % 16].ravel(),
    ]
    units[2][37 * 16 + 9] = True
    big_a = [-128, -128, -128, -128]
    big_b = [-128, -128, -128, 127]

    def operand(rows, big):
        X = np.empty((rows, K), np.int8)
        for f in range(4):
            mask = np.resize(units[f], K)
            sign = rng.choice(np.array([-1, 1], np.int8), size=(len(range(f, rows, 4)), K))
            X[f::4] = np.where(mask[None, :], sign, np.int8(big[f]))
        return X

    return operand(M, big_a), operand(N, big_b)


@pytest.mark.parametrize("M,N,K", [(256, 384, 4096), (2100, 2300, 4096)])
@pytest.mark.parametrize("use_c", [False, True])
def test_i8_exact_mixed_steps_near_the_fp32_limit(M, N, K, use_c):
    """Exact INT8 on the tensor pipe where every 16-deep K step of a
    1024-deep chunk mixes 2^14 products with +-1 products and the chunk's
    partial sums approach +-2^24, on single CTAs (256 x 384) and on CTA
    pairs (2100 x 2300, ragged), with and without C; bit-exact against the
    oracle over the whole output."""
    A, B = _mixed_step_operands(M, N, K, seed=M + N + int(use_c))
    C = (synth.int_uniform(0, 29, M * N, -(1 << 20), 1 << 20).astype(np.int32).reshape(M, N)
         if use_c else np.zeros((M, N), np.int32))
    g = synth.GemmInputs("i8", M, N, K, A, B, C)
    want = oracle.gemm("i8", A, B, C)
    # the families reach the intended chunk sums (first chunk, C excluded)
    c0 = A[:4, :1024].astype(np.int64) @ B[:4, :1024].T.astype(np.int64)
    assert abs(int(c0[0, 0]) - ((1 << 24) - 16 * 16384)) <= 16
    assert abs(int(c0[1, 1]) - 64 * 15 * 16384) <= 64
    assert abs(int(c0[2, 2]) - ((1 << 24) - 16384)) == 1
    assert abs(int(c0[3, 3]) + 64 * 15 * 16256) <= 64
    if use_c:
        check("i8", run_gemm(g, pad=1), want, None, f"i8 mixed steps {M}x{N}x{K} with C")
    else:
        check("i8", run_gemm(g, use_c=False), want, None, f"i8 mixed steps {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (129, 300, 1025), (513, 257, 3000),
                                   (1024, 1024, 8192), (2100, 2300, 3000)])
def test_i8_tensor_pipe_shapes_exact(M, N, K):
    """Shapes on the tcgen05 exact-INT8 path: ragged tiles, K tails and
    several K chunks.  From three chunks up C joins the INT32 sums during
    the chunk phase: 513 x 257 x 3000 on single CTAs, 2100 x 2300 x 3000 on
    CTA pairs (ragged in M, N and K)."""
    g = synth.gemm_inputs(f"i8tc_{M}_{N}_{K}", "i8", M, N, K)
    want, _ = oracle_ref(g)
    check("i8", run_gemm(g, pad=1), want, None, f"i8 {M}x{N}x{K}")


def test_i8_early_c_without_c_on_pairs():
    """The chunk-phase C path with C absent (D = A*B) on CTA pairs."""
    import torch
    M, N, K = 2100, 2300, 3072  # unpadded rows: K a multiple of 16
    g = synth.gemm_inputs("i8tc_noc", "i8", M, N, K)
    D = binding.gemm(to_dev(g.A), to_dev(g.B))
    torch.cuda.synchronize()
    want = oracle.gemm("i8", g.A, g.B, np.zeros((M, N), np.int32))
    check("i8", D.cpu().numpy(), want, None, "i8 pairs, no C")


# ----------------------------------------- FP16/BF16 with 16-bit accumulate

def acc16_inputs(name, dtype_in, M, N, K, b_layout="col"):
    g = synth.gemm_inputs(name, dtype_in, M, N, K, dist="uniform", b_layout=b_layout)
    rnd = synth.round_f16_bits if dtype_in == "f16" else synth.round_bf16_bits
    return synth.GemmInputs(dtype_in, M, N, K, g.A, g.B, rnd(g.C.astype(np.float64)),
                            b_layout)


def run_gemm16(g, *, pad=0, use_c=True, inplace=False):
    import torch
    A = dev_padded(g.A, g.dtype_in, extra=pad)
    B = dev_padded(g.B, g.dtype_in, extra=pad)
    if inplace:
        G = GuardedMatrix(g.M, g.N, np.uint16, dtype_in=g.dtype_in, init=g.C,
                          pad=pad + 1)
        C = G.view
    else:
        G = GuardedMatrix(g.M, g.N, np.uint16, dtype_in=g.dtype_in, pad=pad + 1)
        C = dev_padded(g.C, g.dtype_in, extra=pad) if use_c else None
    out = binding.gemm_ex(A, B, C, G.view, b_layout=g.b_layout, acc="same")
    G.verify(f"{g.dtype_in}->16-bit {g.M}x{g.N}x{g.K} D guard")
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def oracle16(g, rows=None, cols=None):
    A, B, C = g.A, g.B, g.C
    if rows is not None:
        A, C = np.ascontiguousarray(A[rows]), np.ascontiguousarray(C[rows])
    if cols is not None:
        B = np.ascontiguousarray(B[cols] if g.b_layout == "col" else B[:, cols])
        C = np.ascontiguousarray(C[:, cols])
    return oracle.gemm_acc16(g.dtype_in, A, B, C, b_layout=g.b_layout, want_absab=True)


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (16, 16, 16), (127, 129, 65),
                                   (256, 256, 256), (333, 257, 1000), (1000, 136, 520),
                                   (300, 264, 2500)])
def test_acc16_small_shapes(dtype_in, M, N, K):
    g = acc16_inputs(f"acc16_{M}_{N}_{K}", dtype_in, M, N, K)
    want, ab = oracle16(g)
    check16(dtype_in, run_gemm16(g), want, ab, f"{dtype_in}->{dtype_in} {M}x{N}x{K}")


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_acc16_padding_no_c_in_place_row_b(dtype_in):
    M, N, K = 260, 392, 328
    g = acc16_inputs("acc16_pad", dtype_in, M, N, K)
    want, ab = oracle16(g)
    check16(dtype_in, run_gemm16(g, pad=3), want, ab, "padded")
    check16(dtype_in, run_gemm16(g, inplace=True), want, ab, "in place")
    g0 = synth.GemmInputs(dtype_in, M, N, K, g.A, g.B, np.zeros_like(g.C))
    want0, ab0 = oracle16(g0)
    check16(dtype_in, run_gemm16(g, use_c=False), want0, ab0, "C = NULL")
    gr = acc16_inputs("acc16_row", dtype_in, M, N, K, b_layout="row")
    want, ab = oracle16(gr)
    check16(dtype_in, run_gemm16(gr, pad=1), want, ab, "row-major B")


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_acc16_exact_closed_form(dtype_in):
    """All ones, K = 256, integer C: D = K + C exactly representable."""
    M, N, K = 300, 260, 256
    one = np.uint16(0x3C00 if dtype_in == "f16" else 0x3F80)
    rnd = synth.round_f16_bits if dtype_in == "f16" else synth.round_bf16_bits
    Cv = np.random.default_rng(2).integers(-64, 64, (M, N)).astype(np.float64)
    g = synth.GemmInputs(dtype_in, M, N, K, np.full((M, K), one), np.full((N, K), one),
                         rnd(Cv))
    assert np.array_equal(run_gemm16(g), rnd(Cv + K))


def test_acc16_full_size_sampled():
    """BF16 -> BF16 at 8192^3 (the large BF16 workload's shape), sampled."""
    import torch
    M = N = K = 8192
    g = acc16_inputs("acc16_8192", "bf16", M, N, K)
    Gd = GuardedMatrix(M, N, np.uint16, dtype_in="bf16")
    D = binding.gemm_ex(to_dev(g.A, "bf16"), to_dev(g.B, "bf16"), to_dev(g.C, "bf16"),
                        Gd.view, acc="same")
    Gd.verify("bf16->bf16 8192^3 D guard")
    rng = np.random.default_rng(99)
    rows = np.unique(np.append(rng.choice(M, 64, replace=False), M - 1))
    cols = np.unique(np.append(rng.choice(N, 64, replace=False), N - 1))
    got = D[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()]
    got = got.view(torch.int16).cpu().numpy().view(np.uint16)
    want, ab = oracle16(g, rows, cols)
    check16("bf16", got, want, ab, "bf16->bf16 8192^3")


# ------------------------------------------------------------ batched

def run_batched(bi):
    G = GuardedBatch(bi.batch, bi.M, bi.N, OUT_NP[bi.dtype_in])
    binding.gemm_batched(to_dev(bi.A, bi.dtype_in), to_dev(bi.B, bi.dtype_in),
                         to_dev(bi.C), G.view, group=bi.group, abid=bi.abid)
    G.verify(f"batched {bi.dtype_in} x{bi.batch} D guard")
    return G.result()


def batched_absab(bi):
    return oracle.gemm_batched(bi.dtype_in, bi.A & 0x7FFF, bi.B & 0x7FFF, None,
                               group=bi.group, abid=bi.abid).astype(np.float64)


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("G,abid,batch", [(1, 0, 1), (1, 0, 7), (2, 1, 6), (4, 1, 64),
                                          (4, 3, 1028), (8, 5, 80), (16, 0, 160)])
def test_batched_small(dtype_in, G, abid, batch):
    bi = synth.batched_inputs(f"par_b_{G}_{batch}", dtype_in, batch, group=G, abid=abid)
    want = oracle.gemm_batched(dtype_in, bi.A, bi.B, bi.C, group=G, abid=abid)
    check(dtype_in, run_batched(bi), want, batched_absab(bi), f"batched G={G}")


def test_batched_worked_example_on_gpu():
    """The broadcast example of "Common MFMA parameters" (cbsz = 2, abid = 1):
    A tile t = (t+1) I and B = I, so D_b = (src(b)+1) I identifies src(b)."""
    import torch
    batch, n = 16, 16
    A = np.zeros((batch, n, n), np.uint16)
    for t in range(batch):
        A[t] = np.where(np.eye(n, dtype=bool), synth.round_bf16_bits(np.array([t + 1.0]))[0], 0)
    B = np.broadcast_to(np.where(np.eye(n, dtype=bool), np.uint16(0x3F80), np.uint16(0)),
                        (batch, n, n)).astype(np.uint16)
    D = binding.gemm_batched(to_dev(A, "bf16"), to_dev(B, "bf16"), None, group=4, abid=1)
    torch.cuda.synchronize()
    D = D.cpu().numpy()
    for b, src in [(0, 1), (1, 1), (2, 1), (3, 1), (4, 5), (5, 5), (6, 5), (7, 5)]:
        assert np.array_equal(D[b], (src + 1) * np.eye(n, dtype=np.float32))


# ------------------------------------------------- full-size workloads

def _sample_blocks(g, rng, nrow, ncol):
    rows = np.sort(rng.choice(g.M, size=min(nrow, g.M), replace=False))
    cols = np.sort(rng.choice(g.N, size=min(ncol, g.N), replace=False))
    # always include the last row/column (ragged tile edges)
    rows[-1], cols[-1] = g.M - 1, g.N - 1
    return np.unique(rows), np.unique(cols)


FULL_COMPARE = {"gemm_i8_4096", "gemm_bf16_skinny_16384x128x4096"}


@pytest.mark.parametrize("name", ["gemm_f16_256", "gemm_i8_4096", "gemm_bf16_8192",
                                  "gemm_f64_4096_rowB",
                                  "gemm_bf16_skinny_16384x128x4096",
                                  "gemm_bf16_deepk_1024x1024x32768"])
def test_full_size_workload(name):
    """The workloads at full size, D inside guard bands.  The INT8 headline
    (16.8 M outputs, bit-exact) and the skinny BF16 product are compared in
    full (the oracle needs a few seconds for each); the 8192^3 BF16 and the
    4096^3 FP64 products on sampled row x column blocks."""
    import torch
    w = synth.WORKLOADS[name]
    g = synth.gemm_inputs(name, w["dtype_in"], w["M"], w["N"], w["K"],
                          dist=w.get("dist", "normal"),
                          b_layout=w.get("b_layout", "col"))
    Gd = GuardedMatrix(g.M, g.N, OUT_NP[g.dtype_in])
    D = binding.gemm_ex(to_dev(g.A, g.dtype_in), to_dev(g.B, g.dtype_in),
                        to_dev(g.C), Gd.view, b_layout=g.b_layout)
    Gd.verify(f"{name} D guard")
    if g.M * g.N * g.K <= 256 ** 3 or name in FULL_COMPARE:
        want, ab = oracle_ref(g)
        check(g.dtype_in, D.cpu().numpy(), want, ab, name)
        return
    rng = np.random.default_rng(1234)
    rows, cols = _sample_blocks(g, rng, 96, 96)
    got = D[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
    want, ab = oracle_ref(g, rows, cols)
    check(g.dtype_in, got, want, ab, name)
    assert bool(torch.isfinite(D.double()).all()) if g.dtype_in != "i8" else True


def test_full_size_batched_workload():
    name = "batched_bf16_16x16x16_b262144_g4_abid1"
    w = synth.WORKLOADS[name]
    bi = synth.batched_inputs(name, "bf16", w["batch"], group=w["group"], abid=w["abid"])
    got = run_batched(bi)
    want = oracle.gemm_batched("bf16", bi.A, bi.B, bi.C, group=bi.group, abid=bi.abid)
    check("bf16", got, want, batched_absab(bi), name)


@pytest.mark.parametrize("dtype_in", ["bf16", "f16", "i8"])
def test_ragged_shapes_on_cta_pairs(dtype_in):
    """A problem the automatic choice runs on CTA pairs (M > 128, more than
    2^30 multiply-adds, at least one 256 x 256 pair tile per pair), ragged
    in every dimension: M = 2000 (= 7 * 256 + 208), N = 2600, K = 1000.
    Sampled rows (with the last) against the oracle."""
    import torch
    M, N, K = 2000, 2600, 1000
    g = synth.gemm_inputs(f"pair_ragged_{dtype_in}", dtype_in, M, N, K, dist="uniform")
    Gd = GuardedMatrix(M, N, OUT_NP[dtype_in], pad=2)
    D = binding.gemm(dev_padded(g.A, dtype_in), dev_padded(g.B, dtype_in),
                     dev_padded(g.C), Gd.view)
    Gd.verify(f"{dtype_in} ragged pairs D guard")
    rng = np.random.default_rng(11)
    rows = np.unique(np.append(rng.choice(M, 90, replace=False), [M - 1, M - 208]))
    A = np.ascontiguousarray(g.A[rows])
    C = np.ascontiguousarray(g.C[rows])
    got = D[torch.from_numpy(rows).cuda()].cpu().numpy()
    if dtype_in == "i8":
        check("i8", got, oracle.gemm("i8", A, g.B, C), None, "i8 ragged pairs")
    else:
        want, ab = oracle.gemm(dtype_in, A, g.B, C, want_absab=True)
        check(dtype_in, got, want, ab, f"{dtype_in} ragged pairs")



# One row of tiles (M at most one pair row, or one 128-row tile) or one
# column (N at most one tile): the producer loads both operands with an
# evict-first L2 policy, on CTA pairs (256 x 20480 x 1000: 80 pair tiles)
# and on single CTAs (128 x 8192 x 2040; 1000 x 128 x 1000), ragged in K.
@pytest.mark.parametrize("dtype_in", ["bf16", "i8"])
@pytest.mark.parametrize("M,N,K", [(256, 20480, 1000), (128, 8192, 2040),
                                   (1000, 128, 1000)])
def test_single_row_or_column_of_tiles(dtype_in, M, N, K):
    g = synth.gemm_inputs(f"stream_ops_{M}_{N}_{K}_{dtype_in}", dtype_in, M, N, K,
                          dist="uniform")
    got = run_gemm(g, pad=1)
    if dtype_in == "i8":
        check("i8", got, oracle.gemm("i8", g.A, g.B, g.C), None,
              f"i8 {M}x{N}x{K} single row/column of tiles")
    else:
        want, ab = oracle.gemm(dtype_in, g.A, g.B, g.C, want_absab=True)
        check(dtype_in, got, want, ab, f"{dtype_in} {M}x{N}x{K} single row/column of tiles")


# IEEE special values through the tensor pipe: a NaN in A, an infinity in A
# whose K column of B holds zeros, positives and negatives (NaN, +inf and
# -inf results), an infinity in B met by a zero column of A, and a NaN and
# an infinity in C.  NaN positions and infinity signs must match the
# oracle's double arithmetic exactly; the finite outputs keep the usual
# tolerance.  64 x 96 x 128 runs on the regular kernel, 256 x 320 x 9000 on
# the stream-K kernel (the specials meet inside split tiles).
_SPECIAL = {"f16": (0x7E00, 0x7C00, 0xFC00), "bf16": (0x7FC0, 0x7F80, 0xFF80)}


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(64, 96, 128), (256, 320, 9000)])
def test_special_values_propagate(dtype_in, M, N, K):
    nan, pinf, ninf = _SPECIAL[dtype_in]
    g = synth.gemm_inputs(f"special_{M}_{N}_{K}_{dtype_in}", dtype_in, M, N, K,
                          dist="uniform")
    A, B, C = g.A.copy(), g.B.copy(), g.C.copy()   # B is column-major: N x K
    A[3, 5] = nan                                  # row 3 all NaN
    A[7, 0] = pinf                                 # row 7: inf * B[:, 0]
    B[0:N:3, 0] = 0                                # ... NaN where B is 0
    B[1:N:3, 0] = 0x3C00 if dtype_in == "f16" else 0x3F80   # +1: +inf
    B[2:N:3, 0] = 0xBC00 if dtype_in == "f16" else 0xBF80   # -1: -inf
    B[10, K - 1] = ninf                            # column 10: -inf * A[:, K-1]
    A[0:M:2, K - 1] = 0                            # ... NaN in even rows
    C[20, 30] = np.nan
    C[21, 31] = np.inf
    gs = synth.GemmInputs(dtype_in, M, N, K, A, B, C)
    want, ab = oracle.gemm(dtype_in, A, B, C, want_absab=True)
    got = run_gemm(gs)
    assert np.array_equal(np.isnan(got), np.isnan(want)), "NaN positions differ"
    inf_w = np.isinf(want)
    assert np.array_equal(np.isinf(got), inf_w), "infinity positions differ"
    assert np.array_equal(np.sign(got[inf_w]), np.sign(want[inf_w])), "infinity signs differ"
    # the cases the inputs were built for (column 10 of row 7 also meets
    # the -inf of B, so it is left out)
    cols = np.arange(N) != 10
    assert np.isnan(want[3]).all() and np.isnan(want[7, 0::3]).all()
    assert (want[7, 1::3][cols[1::3]] == np.inf).all()
    assert (want[7, 2::3][cols[2::3]] == -np.inf).all()
    assert np.isnan(want[0:M:2, 10]).all()
    fin = np.isfinite(want) & np.isfinite(ab)
    rel, ab0 = TOL[dtype_in]
    err = np.abs(got[fin].astype(np.float64) - want[fin])
    assert (err <= rel * ab[fin] + ab0).all(), f"finite outputs off by up to {err.max()}"


@pytest.mark.parametrize("M,N,K", [(64, 96, 128), (200, 136, 520)])
def test_special_values_propagate_f64(M, N, K):
    """The same specials through the FP64 (DMMA) kernel."""
    g = synth.gemm_inputs(f"special64_{M}_{N}_{K}", "f64", M, N, K, dist="uniform")
    A, B, C = g.A.copy(), g.B.copy(), g.C.copy()
    A[3, 5] = np.nan
    A[7, 0] = np.inf
    B[0:N:3, 0] = 0.0
    B[1:N:3, 0] = 1.0
    B[2:N:3, 0] = -1.0
    B[10, K - 1] = -np.inf
    A[0:M:2, K - 1] = 0.0
    C[20, 30] = np.nan
    C[21, 31] = np.inf
    gs = synth.GemmInputs("f64", M, N, K, A, B, C)
    want, ab = oracle.gemm("f64", A, B, C, want_absab=True)
    got = run_gemm(gs)
    assert np.array_equal(np.isnan(got), np.isnan(want)), "NaN positions differ"
    inf_w = np.isinf(want)
    assert np.array_equal(np.isinf(got), inf_w), "infinity positions differ"
    assert np.array_equal(np.sign(got[inf_w]), np.sign(want[inf_w])), "infinity signs differ"
    assert np.isnan(want[3]).all() and np.isnan(want[0:M:2, 10]).all()
    fin = np.isfinite(want) & np.isfinite(ab)
    rel, ab0 = TOL["f64"]
    err = np.abs(got[fin] - want[fin])
    assert (err <= rel * ab[fin] + ab0 + np.abs(want[fin]) * 2.0 ** -52).all()


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_special_values_propagate_acc16(dtype_in):
    """The same specials with a 16-bit addend and result (the kernel rounds
    its FP32 sum once to 16 bits, the oracle its double sum), plus a finite
    row whose sum overflows the 16-bit range (+inf in both)."""
    M, N, K = 64, 96, 128
    nan, pinf, ninf = _SPECIAL[dtype_in]
    big = 0x7BFF if dtype_in == "f16" else 0x7F7F        # the largest finite
    one = 0x3C00 if dtype_in == "f16" else 0x3F80
    g = acc16_inputs(f"special16_{dtype_in}", dtype_in, M, N, K)
    A, B, C = g.A.copy(), g.B.copy(), g.C.copy()
    A[3, 5] = nan
    A[7, 0] = pinf
    B[0:N:3, 0] = 0
    B[1:N:3, 0] = one
    B[2:N:3, 0] = one | 0x8000
    B[10, K - 1] = ninf
    A[0:M:2, K - 1] = 0
    C[20, 30] = nan
    C[21, 31] = pinf
    A[9, :] = 0                                          # row 9: 4 * big
    A[9, 4:8] = big
    B[:, 4:8] = one
    gs = synth.GemmInputs(dtype_in, M, N, K, A, B, C)
    want_bits, ab = oracle16(gs)
    got = decode16(run_gemm16(gs), dtype_in)
    want = decode16(want_bits, dtype_in)
    assert np.array_equal(np.isnan(got), np.isnan(want)), "NaN positions differ"
    inf_w = np.isinf(want)
    assert np.array_equal(np.isinf(got), inf_w), "infinity positions differ"
    assert np.array_equal(np.sign(got[inf_w]), np.sign(want[inf_w])), "infinity signs differ"
    assert (want[9, np.arange(N) != 10] == np.inf).all()   # overflowed
    fin = np.isfinite(want) & np.isfinite(ab)
    ulp = 2.0 ** -10 if dtype_in == "f16" else 2.0 ** -7
    err = np.abs(got[fin] - want[fin])
    assert (err <= 1e-3 * ab[fin] + 1e-6 + ulp * np.abs(want[fin])).all()
