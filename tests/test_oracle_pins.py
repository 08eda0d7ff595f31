"""Pins of the CPU oracle to facts fixed outside itself.

Each test checks the oracle against something other than its own code:
exact rational arithmetic (Python ``fractions``/ints) on small inputs, closed
forms (identity, all-ones), invariants (transpose), library conversions of
the 16-bit formats, and the worked broadcast example printed on the page
"Common MFMA parameters" (section "Shared parameters").  A dropped term,
wrong sign, swapped index or transposed operand in the oracle fails at
least one of them.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

from mixed_precision_dense_02_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- helpers

def frac_of_f16(bits):
    return Fraction(float(np.uint16(bits).view(np.float16)))


def frac_of_bf16(bits):
    return Fraction(float(np.array([np.uint32(bits) << np.uint32(16)],
                                   np.uint32).view(np.float32)[0]))


def round_fraction_f32(q: Fraction) -> np.float32:
    """Round an exact rational to float32, nearest with ties to even."""
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length() - 24
    while a / Fraction(2) ** e >= 2 ** 24:
        e += 1
    while a / Fraction(2) ** e < 2 ** 23:
        e -= 1
    e = max(e, -149)
    scaled = a / Fraction(2) ** e
    m = math.floor(scaled)
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return np.float32(sign * float(m * Fraction(2) ** e))


def exact_gemm(A, Bcol, C, dec):
    """Exact rational D = A*B + C, B given column-major (N x K)."""
    M, K = A.shape
    N = Bcol.shape[0]
    out = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += dec(A[i, k]) * dec(Bcol[j, k])
            out[i][j] = s + (Fraction(float(C[i, j])) if C is not None else 0)
    return out


def f16_grid(rng, shape, dtype_in):
    """Values on the 2^-10 grid in [-1, 1): sums stay exact in double."""
    v = rng.integers(-1024, 1024, size=shape) / 1024.0
    return (synth.round_f16_bits(v) if dtype_in == "f16"
            else synth.round_bf16_bits(np.round(v * 128) / 128))


# ------------------------------------------------------ c1 decode pins

def test_f16_decode_matches_numpy_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.f16_to_double(int(b)) for b in bits])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_bf16_decode_matches_float32_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    got = np.array([oracle_mod.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


# ------------------------------------------- c2 FP16/BF16 -> FP32 pins

SMALL = [(1, 1, 1), (2, 3, 5), (3, 2, 1), (5, 5, 16), (16, 17, 3),
         (17, 16, 17), (1, 17, 16)]


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_f16_exact_bruteforce_on_grid(oracle_mod, dtype_in, M, N, K):
    """On grid inputs the double sum is exact, so the oracle must equal the
    exact rational result rounded once to FP32."""
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = f16_grid(rng, (M, K), dtype_in)
    B = f16_grid(rng, (N, K), dtype_in)
    C = rng.standard_normal((M, N)).astype(np.float32)
    D = oracle_mod.gemm(dtype_in, A, B, C)
    dec = frac_of_f16 if dtype_in == "f16" else frac_of_bf16
    ex = exact_gemm(A, B, C, dec)
    want = np.array([[round_fraction_f32(q) for q in row] for row in ex],
                    np.float32)
    assert np.array_equal(D.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_f16_bruteforce_general_inputs_within_one_rounding(oracle_mod, dtype_in):
    """Any fp16/bf16 inputs (subnormals included): at most one FP32 rounding
    away from the exact value (plus a double-precision term)."""
    rng = np.random.default_rng(7)
    M, N, K = 6, 5, 17
    rnd = synth.round_f16_bits if dtype_in == "f16" else synth.round_bf16_bits
    A = rnd(rng.standard_normal((M, K)) * np.exp2(rng.integers(-20, 5, (M, K))))
    B = rnd(rng.standard_normal((N, K)) * np.exp2(rng.integers(-20, 5, (N, K))))
    C = rng.standard_normal((M, N)).astype(np.float32)
    D = oracle_mod.gemm(dtype_in, A, B, C)
    dec = frac_of_f16 if dtype_in == "f16" else frac_of_bf16
    ex = exact_gemm(A, B, C, dec)
    for i in range(M):
        for j in range(N):
            q = ex[i][j]
            err = abs(Fraction(float(D[i, j])) - q)
            assert err <= abs(q) * Fraction(1, 2 ** 24) + Fraction(1, 2 ** 60)


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_f16_all_ones_closed_form(oracle_mod, dtype_in):
    M, N, K = 7, 9, 300
    one = 0x3C00 if dtype_in == "f16" else 0x3F80
    A = np.full((M, K), one, np.uint16)
    B = np.full((N, K), one, np.uint16)
    C = np.random.default_rng(0).standard_normal((M, N)).astype(np.float32)
    D = oracle_mod.gemm(dtype_in, A, B, C)
    want = (np.float64(K) + C.astype(np.float64)).astype(np.float32)
    assert np.array_equal(D, want)


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_f16_identity_closed_forms(oracle_mod, dtype_in):
    """B = I gives D = A + C; A = I gives D = B + C (B read as K x N)."""
    rng = np.random.default_rng(1)
    n = 24
    rnd = synth.round_f16_bits if dtype_in == "f16" else synth.round_bf16_bits
    to32 = synth.f16_bits_to_f32 if dtype_in == "f16" else synth.bf16_bits_to_f32
    one = 0x3C00 if dtype_in == "f16" else 0x3F80
    eye = np.where(np.eye(n, dtype=bool), one, 0).astype(np.uint16)
    X = rnd(rng.uniform(-1, 1, (n, n)))          # not symmetric
    C = rng.standard_normal((n, n)).astype(np.float32)
    # B = I (column-major storage of I is I)
    D = oracle_mod.gemm(dtype_in, X, eye, C)
    assert np.array_equal(D, (to32(X).astype(np.float64) + C).astype(np.float32))
    # A = I, B column-major stored as X (N x K): B[k][j] = X[j][k]
    D2 = oracle_mod.gemm(dtype_in, eye, X, C)
    assert np.array_equal(D2, (to32(X).T.astype(np.float64) + C).astype(np.float32))
    # A = I, B row-major stored as X (K x N): B[k][j] = X[k][j]
    D3 = oracle_mod.gemm(dtype_in, eye, X, C, b_layout="row")
    assert np.array_equal(D3, (to32(X).astype(np.float64) + C).astype(np.float32))


@pytest.mark.parametrize("dtype_in", ["f16", "bf16", "i8", "f64"])
def test_transpose_invariance(oracle_mod, dtype_in):
    """(A*B + C)^T == B^T * A^T + C^T.  With A row-major and B column-major,
    the operand buffers swap roles unchanged, so the oracle must agree with
    itself bit for bit (it sums in the same k order)."""
    M, N, K = 13, 21, 37
    g = synth.gemm_inputs("transpose_pin", dtype_in, M, N, K, dist="uniform")
    D = oracle_mod.gemm(dtype_in, g.A, g.B, g.C)
    DT = oracle_mod.gemm(dtype_in, g.B, g.A, np.ascontiguousarray(g.C.T))
    assert np.array_equal(D.T, DT)


@pytest.mark.parametrize("dtype_in", ["f16", "bf16", "i8", "f64"])
def test_layout_and_padding_invariance(oracle_mod, dtype_in):
    """Row-major B == column-major B transposed; padded leading dimensions
    (garbage in the padding) do not change the result; C=None == C=0."""
    M, N, K = 9, 11, 19
    g = synth.gemm_inputs("layout_pin", dtype_in, M, N, K, dist="uniform")
    D = oracle_mod.gemm(dtype_in, g.A, g.B, g.C)
    Brow = np.ascontiguousarray(g.B.T)
    assert np.array_equal(D, oracle_mod.gemm(dtype_in, g.A, Brow, g.C, b_layout="row"))

    def pad(x, extra):
        big = np.empty((x.shape[0], x.shape[1] + extra), x.dtype)
        big.view(np.uint8)[:] = 0xA5
        big[:, : x.shape[1]] = x
        return big[:, : x.shape[1]]

    Dp = oracle_mod.gemm(dtype_in, pad(g.A, 7), pad(g.B, 3), pad(g.C, 5))
    assert np.array_equal(D, Dp)
    Z = np.zeros_like(g.C)
    assert np.array_equal(oracle_mod.gemm(dtype_in, g.A, g.B, None),
                          oracle_mod.gemm(dtype_in, g.A, g.B, Z))


def test_absab_is_sum_of_absolute_products(oracle_mod):
    rng = np.random.default_rng(3)
    A = synth.round_bf16_bits(rng.standard_normal((4, 9)))
    B = synth.round_bf16_bits(rng.standard_normal((5, 9)))
    _, ab = oracle_mod.gemm("bf16", A, B, None, want_absab=True)
    a = synth.bf16_bits_to_f32(A).astype(np.float64)
    b = synth.bf16_bits_to_f32(B).astype(np.float64)
    for i in range(4):
        for j in range(5):
            ex = sum(Fraction(abs(a[i, k])) * Fraction(abs(b[j, k])) for k in range(9))
            assert abs(Fraction(ab[i, j]) - ex) <= ex * Fraction(1, 2 ** 50)


# ----------------------------------------------------- c3 INT8 pins

@pytest.mark.parametrize("M,N,K", SMALL + [(8, 8, 64)])
def test_i8_exact_bruteforce(oracle_mod, M, N, K):
    g = synth.gemm_inputs(f"i8_pin_{M}_{N}_{K}", "i8", M, N, K)
    D = oracle_mod.gemm("i8", g.A, g.B, g.C)
    for i in range(M):
        for j in range(N):
            s = sum(int(g.A[i, k]) * int(g.B[j, k]) for k in range(K)) + int(g.C[i, j])
            assert int(D[i, j]) == s


def test_i8_closed_forms(oracle_mod):
    M, N, K = 5, 6, 4096
    C = synth.int_uniform(0, 99, M * N, -(1 << 20), 1 << 20).astype(np.int32).reshape(M, N)
    ones = np.ones((M, K), np.int8)
    D = oracle_mod.gemm("i8", ones, np.ones((N, K), np.int8), C)
    assert np.array_equal(D, K + C)
    # the largest product magnitude everywhere: (-128) * (-128) = 2^14
    neg = np.full((M, K), -128, np.int8)
    D = oracle_mod.gemm("i8", neg, np.full((N, K), -128, np.int8), C)
    assert np.array_equal(D.astype(np.int64), K * 16384 + C.astype(np.int64))
    # mixed signs: (-128) * 127
    D = oracle_mod.gemm("i8", neg, np.full((N, K), 127, np.int8), C)
    assert np.array_equal(D.astype(np.int64), -K * 16256 + C.astype(np.int64))


def test_i8_overflow_is_reported(oracle_mod):
    K = 1 << 17  # 2^17 * 2^14 = 2^31 does not fit in int32
    A = np.full((1, K), -128, np.int8)
    B = np.full((1, K), -128, np.int8)
    with pytest.raises(OverflowError):
        oracle_mod.gemm("i8", A, B, None)


# ----------------------------------------------------- c4 FP64 pins

@pytest.mark.parametrize("M,N,K", SMALL)
def test_f64_bruteforce_one_rounding(oracle_mod, M, N, K):
    """Dot2 plus C: within one rounding of the exact rational result, up to
    an eps^2-sized term (Ogita, Rump, Oishi 2005, Prop. 5.5)."""
    g = synth.gemm_inputs(f"f64_pin_{M}_{N}_{K}", "f64", M, N, K)
    D = oracle_mod.gemm("f64", g.A, g.B, g.C)
    for i in range(M):
        for j in range(N):
            q = sum(Fraction(g.A[i, k]) * Fraction(g.B[j, k]) for k in range(K))
            sab = sum(abs(Fraction(g.A[i, k]) * Fraction(g.B[j, k])) for k in range(K))
            q += Fraction(g.C[i, j])
            err = abs(Fraction(D[i, j]) - q)
            assert err <= abs(q) * Fraction(1, 2 ** 53) + sab * Fraction(1, 2 ** 90)


def test_f64_compensation_recovers_cancelled_terms(oracle_mod):
    """Naive summation loses the small terms here; the exact answer is 2.5."""
    A = np.array([[1e16, 1.0, -1e16, 1.5, 3e20, -3e20]])
    B = np.ones((1, 6))
    assert oracle_mod.gemm("f64", A, B, None)[0, 0] == 2.5
    # the product error term: (1 + 2^-30)^2 = 1 + 2^-29 + 2^-60, minus 1 + 2^-29
    a = 1.0 + 2.0 ** -30
    A = np.array([[a, -1.0, -(2.0 ** -29)]])
    B = np.array([[a, 1.0, 1.0]])
    assert oracle_mod.gemm("f64", A, B, None)[0, 0] == 2.0 ** -60


def test_f64_special_values_extended_reals(oracle_mod):
    """IEEE semantics of D = A*B + C with non-finite terms (arithmetic over
    the extended reals): an infinity plus finite terms is that infinity,
    infinities of both signs or a NaN give NaN, 0 * inf is NaN; the same
    for the batched branch (which shares the row kernel)."""
    inf, nan = np.inf, np.nan
    A = np.array([[inf, 1.0, 2.0],        # +inf + 3 + 8        -> +inf
                  [inf, -inf, 0.5],       # +inf - inf          -> NaN
                  [nan, 1.0, 1.0],        # NaN                 -> NaN
                  [0.0, 1.0, 1.0],        # 0 * (-inf) in col 1 -> NaN
                  [-inf, 1.0, 1.0],       # -inf * 3 = -inf     -> -inf
                  [1.0, 1.0, 1.0]])       # finite; C decides
    B = np.array([[1.0, 3.0, 4.0],        # column 0 (N x K layout)
                  [-inf, 1.0, 1.0],       # column 1: starts with -inf
                  [3.0, 0.0, 0.0]])       # column 2
    C = np.zeros((6, 3))
    C[5, 0] = inf
    C[5, 1] = -inf
    C[5, 2] = nan
    D = oracle_mod.gemm("f64", A, B, C)
    assert D[0, 0] == inf and np.isnan(D[1, 0]) and np.isnan(D[2, 0])
    assert D[4, 0] == -inf and D[3, 0] == 7.0
    # column 1 starts with -inf: inf * -inf = -inf, -inf * -inf = +inf
    assert np.isnan(D[3, 1]) and D[4, 1] == inf and D[0, 1] == -inf
    assert D[1, 1] == -inf
    # column 2 is (3, 0, 0): -inf * 0 in row 1 gives NaN
    assert D[0, 2] == inf and D[4, 2] == -inf and np.isnan(D[2, 2])
    assert np.isnan(D[1, 2])
    assert D[5, 0] == inf and D[5, 1] == -inf and np.isnan(D[5, 2])
    # finite entries keep the compensated (exact here) value
    assert D[3, 2] == 0.0 and D[5, 0] == inf
    # the batched branch on the same tile (batch of 1)
    Db = oracle_mod.gemm_batched("f64", A[None], B[None], C[None], group=1, abid=0)
    assert np.array_equal(np.isnan(Db[0]), np.isnan(D))
    assert np.array_equal(Db[0][np.isfinite(D)], D[np.isfinite(D)])
    assert np.array_equal(Db[0][np.isinf(D)], D[np.isinf(D)])


def test_f64_closed_forms(oracle_mod):
    n = 32
    rng = np.random.default_rng(5)
    X = rng.standard_normal((n, n))
    C = rng.standard_normal((n, n))
    I = np.eye(n)
    assert np.array_equal(oracle_mod.gemm("f64", X, I, C), X + C)
    assert np.array_equal(oracle_mod.gemm("f64", I, X, C, b_layout="row"), X + C)
    D = oracle_mod.gemm("f64", np.ones((3, 1000)), np.ones((4, 1000)), C[:3, :4].copy())
    assert np.array_equal(D, 1000.0 + C[:3, :4])


# ------------------------------------------------- c5 broadcast pins

def _golden_broadcast():
    rows = []
    with open(os.path.join(HERE, "golden", "broadcast_worked_example.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                rows.append(line)
    return rows


def _tagged_tiles(batch, n=16):
    """A tile t = (t+1) * I (exact in bf16 for t < 256), B_b = I, C = 0:
    D_b = (src(b) + 1) * I, so the source index is read off D."""
    one = 0x3F80
    A = np.zeros((batch, n, n), np.uint16)
    for t in range(batch):
        A[t] = np.where(np.eye(n, dtype=bool),
                        synth.round_bf16_bits(np.array([t + 1.0]))[0], 0)
    B = np.broadcast_to(np.where(np.eye(n, dtype=bool), one, 0).astype(np.uint16),
                        (batch, n, n)).copy()
    C = np.zeros((batch, n, n), np.float32)
    return A, B, C


def test_broadcast_worked_example(oracle_mod):
    rows = _golden_broadcast()
    assert rows, "golden fixture is empty"
    batch = 16
    A, B, C = _tagged_tiles(batch)
    for r in rows:
        if r[0] == "src":
            G, abid, block, source = map(int, r[1:])
            D = oracle_mod.gemm_batched("bf16", A, B, C, group=G, abid=abid)
            assert D[block, 0, 0] == source + 1
            assert D[block, 3, 3] == source + 1 and D[block, 0, 1] == 0
        elif r[0] == "same":
            G = int(r[1])
            blocks = list(map(int, r[2:]))
            for abid in range(G):
                D = oracle_mod.gemm_batched("bf16", A, B, C, group=G, abid=abid)
                for b in blocks[1:]:
                    assert np.array_equal(D[b], D[blocks[0]])
                # and a different group sees different A
                other = (blocks[0] + G) % batch
                assert not np.array_equal(D[other], D[blocks[0]])


@pytest.mark.parametrize("G,abid", [(1, 0), (2, 1), (4, 1), (4, 3), (8, 0), (16, 15)])
def test_broadcast_equals_replicated_a(oracle_mod, G, abid):
    batch = 32
    bi = synth.batched_inputs("bcast_pin", "bf16", batch, group=G, abid=abid)
    D = oracle_mod.gemm_batched("bf16", bi.A, bi.B, bi.C, group=G, abid=abid)
    src = (np.arange(batch) // G) * G + abid
    Arep = np.ascontiguousarray(bi.A[src])
    D1 = oracle_mod.gemm_batched("bf16", Arep, bi.B, bi.C, group=1, abid=0)
    assert np.array_equal(D, D1)
    # G = 1 is a plain batch of independent products
    for b in (0, batch - 1):
        assert np.array_equal(D1[b], oracle_mod.gemm("bf16", Arep[b], bi.B[b], bi.C[b]))


@pytest.mark.parametrize("G,abid,batch", [(4, 4, 8), (4, -1, 8), (3, 0, 9), (4, 0, 6), (0, 0, 4)])
def test_broadcast_rejects_bad_groups(oracle_mod, G, abid, batch):
    A = np.zeros((batch, 16, 16), np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.gemm_batched("bf16", A, A.copy(), None, group=G, abid=abid)


# ------------------------------------- c2b FP16/BF16 -> 16-bit accumulate

def round_fraction_16(q: Fraction, mant: int, bias: int, emax_field: int) -> int:
    """Exact round-to-nearest-even of a rational to a 16-bit float format."""
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    if a == 0:
        return sign
    emin = 1 - bias
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - mant)
    m = math.floor(a / quantum)
    rem = a / quantum - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    v = m * quantum
    if v >= Fraction(2) ** (emax_field - bias):
        return sign | (emax_field << mant)
    if v < Fraction(2) ** emin:
        return sign | int(v / Fraction(2) ** (emin - mant))
    ev = e if v < Fraction(2) ** (e + 1) else e + 1
    frac = int(v / Fraction(2) ** (ev - mant)) - (1 << mant)
    return sign | ((ev + bias) << mant) | frac


F16_FMT, BF16_FMT = (10, 15, 31), (7, 127, 255)


@pytest.mark.parametrize("kind", ["f16", "bf16"])
def test_double_to_16bit_rounding(oracle_mod, kind):
    """The oracle's encoder against exact rational rounding: random values
    over the whole range, exact ties, subnormals, the overflow boundary."""
    fmt = F16_FMT if kind == "f16" else BF16_FMT
    enc = oracle_mod.double_to_f16 if kind == "f16" else oracle_mod.double_to_bf16
    rng = np.random.default_rng(21)
    lo, hi = (-28, 17) if kind == "f16" else (-136, 128)
    xs = list(rng.uniform(-1, 1, 3000) * np.exp2(rng.integers(lo, hi, 3000)))
    mant, bias, _ = fmt
    for e in (-14 if kind == "f16" else -126, -1, 0, 5):
        for m in range(0, 12):
            # exact ties between neighbours, and their neighbours
            base = (1 + m * 2.0 ** -mant) * 2.0 ** e
            tie = base + 2.0 ** (e - mant - 1)
            xs += [tie, -tie, np.nextafter(tie, 0), np.nextafter(tie, np.inf)]
    xs += [65504.0, 65519.9, 65520.0, 1e9, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]
    for x in xs:
        want = round_fraction_16(Fraction(float(x)), *fmt)
        assert enc(x) == want, (kind, x, hex(enc(x)), hex(want))
    if kind == "f16":  # and against numpy's own double -> binary16
        arr = np.array(xs[:3000])
        assert np.array_equal(np.array([enc(x) for x in arr], np.uint16),
                              arr.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 16), (17, 16, 17)])
def test_acc16_exact_bruteforce(oracle_mod, dtype_in, M, N, K):
    """Exact rational A*B + C rounded once to the 16-bit format."""
    rng = np.random.default_rng(M * 31 + K)
    A = f16_grid(rng, (M, K), dtype_in)
    B = f16_grid(rng, (N, K), dtype_in)
    rnd = synth.round_f16_bits if dtype_in == "f16" else synth.round_bf16_bits
    C = rnd(rng.standard_normal((M, N)))
    D = oracle_mod.gemm_acc16(dtype_in, A, B, C)
    dec = frac_of_f16 if dtype_in == "f16" else frac_of_bf16
    fmt = F16_FMT if dtype_in == "f16" else BF16_FMT
    for i in range(M):
        for j in range(N):
            q = sum(dec(A[i, k]) * dec(B[j, k]) for k in range(K)) + dec(C[i, j])
            assert int(D[i, j]) == round_fraction_16(q, *fmt)


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_acc16_closed_forms(oracle_mod, dtype_in):
    n = 24
    one = 0x3C00 if dtype_in == "f16" else 0x3F80
    eye = np.where(np.eye(n, dtype=bool), one, 0).astype(np.uint16)
    rng = np.random.default_rng(4)
    rnd = synth.round_f16_bits if dtype_in == "f16" else synth.round_bf16_bits
    X = rnd(rng.uniform(-1, 1, (n, n)))
    Z = np.zeros((n, n), np.uint16)
    # B = I, C = 0: D = A exactly; A = I: D = B^T (column-major storage)
    assert np.array_equal(oracle_mod.gemm_acc16(dtype_in, X, eye, Z), X)
    assert np.array_equal(oracle_mod.gemm_acc16(dtype_in, eye, X, None), X.T)
    # all ones, K = 64, C = 1: D = 65 (exact in both formats)
    ones = np.full((3, 64), one, np.uint16)
    D = oracle_mod.gemm_acc16(dtype_in, ones, ones, np.full((3, 3), one, np.uint16))
    want = oracle_mod.double_to_f16(65.0) if dtype_in == "f16" else oracle_mod.double_to_bf16(65.0)
    assert np.all(D == want)


# ------------------------------- c3b INT8/UINT8 signedness and clamp

@pytest.mark.parametrize("sa,sb", [(True, True), (True, False), (False, True), (False, False)])
def test_i8_ex_bruteforce_signedness(oracle_mod, sa, sb):
    rng = np.random.default_rng(int(sa) * 2 + int(sb))
    M, N, K = 7, 9, 33
    A = rng.integers(-128, 128, (M, K)).astype(np.int8)
    B = rng.integers(-128, 128, (N, K)).astype(np.int8)
    if not sa:
        A = A.view(np.uint8)
    if not sb:
        B = B.view(np.uint8)
    C = rng.integers(-(1 << 20), 1 << 20, (M, N)).astype(np.int32)
    D, ov = oracle_mod.gemm_i8_ex(A, B, C)
    assert ov == 0
    for i in range(M):
        for j in range(N):
            s = sum(int(A[i, k]) * int(B[j, k]) for k in range(K)) + int(C[i, j])
            assert int(D[i, j]) == s
    # signed x signed agrees with the plain INT8 oracle
    if sa and sb:
        assert np.array_equal(D, oracle_mod.gemm("i8", A, B, C))


def test_i8_ex_extremes_and_clamp(oracle_mod):
    M, N, K = 3, 4, 4096
    u = np.full((M, K), 255, np.uint8)
    v = np.full((N, K), 255, np.uint8)
    C = np.zeros((M, N), np.int32)
    D, ov = oracle_mod.gemm_i8_ex(u, v, C)
    assert ov == 0 and np.all(D == K * 255 * 255)     # 266,342,400 < 2^31
    # push past INT32: C near the top, positive products
    Ctop = np.full((M, N), 2 ** 31 - 1000, np.int32)
    D, ov = oracle_mod.gemm_i8_ex(u, v, Ctop)
    assert ov == M * N
    exact = 2 ** 31 - 1000 + K * 65025
    assert np.all(D == np.int32(np.int64(exact) - 2 ** 32))          # wraps
    D, ov = oracle_mod.gemm_i8_ex(u, v, Ctop, clamp=True)
    assert ov == M * N and np.all(D == 2 ** 31 - 1)                   # saturates
    # and below INT32 with a mixed-sign product
    neg = np.full((M, K), -128, np.int8)
    Cbot = np.full((M, N), -(2 ** 31) + 5, np.int32)
    D, ov = oracle_mod.gemm_i8_ex(neg, v, Cbot, clamp=True)
    assert np.all(D == -(2 ** 31))
    # no overflow: clamp changes nothing
    D1, _ = oracle_mod.gemm_i8_ex(neg, v, None)
    D2, _ = oracle_mod.gemm_i8_ex(neg, v, None, clamp=True)
    assert np.array_equal(D1, D2) and np.all(D1 == -128 * 255 * K)


# ------------------------------------------------ B lane-group pattern

def _golden_blgp():
    """{pattern: {dest quarter: source quarter}} from the lane-level moves
    transcribed in the golden file (16 lanes = one quarter = one entry of a
    group of four)."""
    out = {}
    with open(os.path.join(HERE, "golden", "blgp_lane_patterns.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            p = int(line[0])
            d0, d1 = map(int, line[1].split("-"))
            s0, s1 = map(int, line[2].split("-"))
            assert d1 - d0 == s1 - s0 and d0 % 16 == 0 and s0 % 16 == 0
            for off in range(0, d1 - d0 + 1, 16):
                out.setdefault(p, {})[(d0 + off) // 16] = (s0 + off) // 16
    return out


def test_blgp_patterns_follow_the_page(oracle_mod):
    table = _golden_blgp()
    assert sorted(table) == list(range(8))
    for p, m in table.items():
        assert sorted(m) == [0, 1, 2, 3], f"pattern {p} must cover all quarters"
        for q, src in m.items():
            assert oracle_mod.blgp_source(p, q) == src, (p, q)
    assert oracle_mod.blgp_source(8, 0) == -1


@pytest.mark.parametrize("blgp", range(8))
def test_batched_blgp_reads_the_mapped_b_tile(oracle_mod, blgp):
    """B tile t = (t+1) * I, A = I, C = 0: D_b = (srcB(b) + 1) * I, read off
    D for two groups of four entries (the group offset is checked too)."""
    table = _golden_blgp()[blgp]
    batch, n = 8, 16
    eye = np.eye(n, dtype=bool)
    one = 0x3F80
    A = np.broadcast_to(np.where(eye, one, 0).astype(np.uint16), (batch, n, n)).copy()
    B = np.zeros((batch, n, n), np.uint16)
    for t in range(batch):
        B[t] = np.where(eye, synth.round_bf16_bits(np.array([t + 1.0]))[0], 0)
    C = np.zeros((batch, n, n), np.float32)
    D = oracle_mod.gemm_batched("bf16", A, B, C, group=1, abid=0, blgp=blgp)
    for b in range(batch):
        src = (b // 4) * 4 + table[b % 4]
        assert np.array_equal(D[b], (src + 1) * np.eye(n, dtype=np.float32)), (blgp, b)


def test_batched_blgp_with_a_broadcast_and_rejections(oracle_mod):
    """cbsz/abid on A and blgp on B act independently: equal to a plain
    batch whose A and B tiles were gathered by the two source maps."""
    batch = 16
    bi = synth.batched_inputs("blgp_pin", "bf16", batch, M=24, N=40, K=32,
                              group=4, abid=2)
    D = oracle_mod.gemm_batched("bf16", bi.A, bi.B, bi.C, group=4, abid=2, blgp=3)
    srcA = [(b // 4) * 4 + 2 for b in range(batch)]
    srcB = [(b // 4) * 4 + (b + 1) % 4 for b in range(batch)]
    D2 = oracle_mod.gemm_batched("bf16", np.ascontiguousarray(bi.A[srcA]),
                                 np.ascontiguousarray(bi.B[srcB]), bi.C)
    assert np.array_equal(D, D2)
    with pytest.raises(ValueError):
        oracle_mod.gemm_batched("bf16", bi.A[:6], bi.B[:6], bi.C[:6], blgp=1)
    with pytest.raises(ValueError):
        oracle_mod.gemm_batched("bf16", bi.A, bi.B, bi.C, blgp=8)


@pytest.mark.parametrize("M,N,K", [(24, 40, 32), (1, 7, 3), (130, 9, 70)])
def test_batched_generic_shapes_are_independent_products(oracle_mod, M, N, K):
    """Any M x N x K: a batch without broadcast is the independent products
    of its entries (each checked against the single-problem oracle, itself
    pinned above by brute force)."""
    batch = 8
    bi = synth.batched_inputs(f"gen_pin_{M}_{N}_{K}", "bf16", batch, M=M, N=N, K=K,
                              group=1, abid=0)
    D = oracle_mod.gemm_batched("bf16", bi.A, bi.B, bi.C)
    for b in range(batch):
        assert np.array_equal(D[b], oracle_mod.gemm("bf16", bi.A[b], bi.B[b], bi.C[b]))


# ------------------- c5 batched INT8 / FP64 branches and row-major B tiles

def _brute_batched_int(A, B, C, b_layout, src_a, src_b):
    """Exact integer batched product in Python-sized integers (numpy int64
    with |sum| far below 2^63): entry b reads A[src_a[b]] and B[src_b[b]]."""
    D = []
    for b in range(A.shape[0]):
        a = A[src_a[b]].astype(np.int64)
        bt = B[src_b[b]].astype(np.int64)
        bm = bt.T if b_layout == "col" else bt  # K x N
        D.append(a @ bm + (0 if C is None else C[b].astype(np.int64)))
    return np.stack(D)


def _maps(batch, G, abid, blgp, table):
    src_a = [(b // G) * G + abid for b in range(batch)]
    src_b = [(b // 4) * 4 + table[b % 4] for b in range(batch)] if blgp else list(range(batch))
    return src_a, src_b


@pytest.mark.parametrize("b_layout", ["col", "row"])
@pytest.mark.parametrize("G,abid,blgp", [(1, 0, 0), (4, 1, 0), (2, 1, 3), (8, 5, 6), (4, 3, 1)])
def test_batched_i8_branch_bruteforce(oracle_mod, b_layout, G, abid, blgp):
    """The batched oracle's INT8 branch against exact integer arithmetic on
    every entry, with the A broadcast (cbsz/abid, "Common MFMA parameters",
    Shared parameters) and the B lane-group pattern (Dense MFMA parameters,
    blgp) gathered by the maps the page defines.  N != K and M != N, so a
    tile stride taken from the wrong extent, or counted in the wrong
    element size, reads another tile and fails."""
    batch, M, N, K = 16, 5, 7, 11
    rng = np.random.default_rng(100 + G * 10 + abid + blgp)
    A = rng.integers(-128, 128, (batch, M, K), dtype=np.int64).astype(np.int8)
    shape_b = (batch, N, K) if b_layout == "col" else (batch, K, N)
    B = rng.integers(-128, 128, shape_b, dtype=np.int64).astype(np.int8)
    C = rng.integers(-(1 << 20), 1 << 20, (batch, M, N), dtype=np.int64).astype(np.int32)
    table = _golden_blgp()[blgp]
    src_a, src_b = _maps(batch, G, abid, blgp, table)
    D = oracle_mod.gemm_batched("i8", A, B, C, group=G, abid=abid,
                                b_layout=b_layout, blgp=blgp)
    assert D.dtype == np.int32
    want = _brute_batched_int(A, B, C, b_layout, src_a, src_b)
    assert np.array_equal(D.astype(np.int64), want)
    # C = None reads as zero
    D0 = oracle_mod.gemm_batched("i8", A, B, None, group=G, abid=abid,
                                 b_layout=b_layout, blgp=blgp)
    assert np.array_equal(D0.astype(np.int64), want - C.astype(np.int64))


@pytest.mark.parametrize("b_layout", ["col", "row"])
@pytest.mark.parametrize("G,abid,blgp", [(1, 0, 0), (4, 1, 0), (2, 0, 2), (16, 9, 7)])
def test_batched_f64_branch_exact_on_integers(oracle_mod, b_layout, G, abid, blgp):
    """The FP64 branch on integer-valued doubles, whose sums are exact:
    the result must equal the integer brute force bit for bit, entry by
    entry, under every source map."""
    batch, M, N, K = 16, 6, 9, 13
    rng = np.random.default_rng(200 + G + abid + blgp)
    A = rng.integers(-1000, 1001, (batch, M, K)).astype(np.float64)
    shape_b = (batch, N, K) if b_layout == "col" else (batch, K, N)
    B = rng.integers(-1000, 1001, shape_b).astype(np.float64)
    C = rng.integers(-10 ** 6, 10 ** 6, (batch, M, N)).astype(np.float64)
    table = _golden_blgp()[blgp]
    src_a, src_b = _maps(batch, G, abid, blgp, table)
    D = oracle_mod.gemm_batched("f64", A, B, C, group=G, abid=abid,
                                b_layout=b_layout, blgp=blgp)
    assert D.dtype == np.float64
    want = _brute_batched_int(A.astype(np.int64), B.astype(np.int64),
                              C.astype(np.int64), b_layout, src_a, src_b)
    assert np.array_equal(D, want.astype(np.float64))


@pytest.mark.parametrize("dtype_in", ["i8", "f64"])
def test_batched_tagged_tiles_int8_and_f64(oracle_mod, dtype_in):
    """The page's worked example (cbsz = 2, abid = 1: block 1's A to blocks
    0, 2, 3 and block 5's to 4, 6, 7) read off tagged tiles in the INT8 and
    FP64 branches: A tile t = (t + 1) I, B = I, C = 0, so D_b = (src + 1) I.
    Non-square 16 x 16 x 16 tiles are not needed here; the rows and K are
    equal, so the tag also checks that nothing off the diagonal leaks in."""
    rows = _golden_broadcast()
    batch, n = 16, 16
    dt = np.int8 if dtype_in == "i8" else np.float64
    eye = np.eye(n, dtype=bool)
    A = np.zeros((batch, n, n), dt)
    for t in range(batch):
        A[t][eye] = t + 1
    B = np.broadcast_to(eye.astype(dt), (batch, n, n)).copy()
    C = np.zeros((batch, n, n), np.int32 if dtype_in == "i8" else np.float64)
    checked = 0
    for r in rows:
        if r[0] != "src":
            continue
        G, abid, block, source = map(int, r[1:])
        D = oracle_mod.gemm_batched(dtype_in, A, B, C, group=G, abid=abid)
        assert D[block, 0, 0] == source + 1 and D[block, n - 1, n - 1] == source + 1
        assert D[block, 0, 1] == 0 and D[block, 5, 4] == 0
        checked += 1
    assert checked >= 8


@pytest.mark.parametrize("dtype_in", ["bf16", "i8", "f64"])
def test_batched_row_major_b_equals_column_major(oracle_mod, dtype_in):
    """Row-major B tiles (batch, K, N) hold the same matrices as the
    column-major (batch, N, K) tiles transposed, so both layouts give the
    same D bit for bit (the oracle sums k in the same order); with K != N
    a tile stride computed from the wrong extent reads shifted data."""
    batch, M, N, K = 8, 7, 12, 20
    bi = synth.batched_inputs(f"rowb_pin_{dtype_in}", dtype_in, batch, M=M, N=N,
                              K=K, group=2, abid=1)
    Bt = np.ascontiguousarray(np.swapaxes(bi.B, 1, 2))  # (batch, K, N)
    for blgp in (0, 5):
        Dc = oracle_mod.gemm_batched(dtype_in, bi.A, bi.B, bi.C, group=2, abid=1,
                                     blgp=blgp)
        Dr = oracle_mod.gemm_batched(dtype_in, bi.A, Bt, bi.C, group=2, abid=1,
                                     b_layout="row", blgp=blgp)
        assert np.array_equal(Dc, Dr)
        # and each entry equals the single-problem oracle with row-major B
        # (pattern 5 sends quarter 1's B tile to the whole group of four)
        for b in (0, 3, batch - 1):
            src = (b // 2) * 2 + 1
            bsrc = (b // 4) * 4 + 1 if blgp == 5 else b
            single = oracle_mod.gemm(dtype_in, bi.A[src], Bt[bsrc], bi.C[b],
                                     b_layout="row")
            assert np.array_equal(Dr[b], single)
