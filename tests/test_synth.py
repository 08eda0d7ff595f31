"""The seeded input generator: determinism, ranges, and one-step rounding."""
from __future__ import annotations

import numpy as np
import pytest

from mixed_precision_dense_02_gb300 import synth


def _nearest_bf16_bruteforce(x: float) -> int:
    """Nearest bfloat16 to x by search over neighbouring patterns
    (ties to even mantissa), via float32 widening of candidates."""
    f = np.float32(x)
    base = int(np.array([f], np.float32).view(np.uint32)[0] >> 16)
    best = None
    for cand in (base - 1, base, base + 1, base + 2):
        if cand < 0 or cand > 0xFFFF:
            continue
        v = float(np.array([cand << 16], np.uint32).view(np.float32)[0])
        if not np.isfinite(v) or (v != 0 and np.sign(v) != np.sign(x)):
            continue
        d = abs(v - x)
        key = (d, cand & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return best[1]


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(11)
    xs = np.concatenate([rng.standard_normal(3000),
                         rng.uniform(-1, 1, 3000) * np.exp2(rng.integers(-40, 40, 3000))])
    got = synth.round_bf16_bits(xs)
    for x, g in zip(xs, got):
        assert int(g) == _nearest_bf16_bruteforce(float(x)), x


def test_bf16_rounding_ties():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    assert synth.round_bf16_bits(np.array([1.0 + 2 ** -8]))[0] == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even) -> up
    assert synth.round_bf16_bits(np.array([1.0 + 3 * 2 ** -8]))[0] == 0x3F82
    # just above the tie rounds up
    assert synth.round_bf16_bits(np.array([1.0 + 2 ** -8 + 2 ** -40]))[0] == 0x3F81
    assert synth.round_bf16_bits(np.array([-2.0]))[0] == 0xC000
    assert synth.round_bf16_bits(np.array([0.0]))[0] == 0


def test_f16_rounding_is_nearest_even():
    rng = np.random.default_rng(12)
    xs = rng.uniform(-1, 1, 5000)
    got = synth.round_f16_bits(xs).view(np.float16).astype(np.float64)
    up = np.nextafter(got.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(got.astype(np.float16), np.float16(-np.inf)).astype(np.float64)
    err = np.abs(got - xs)
    assert np.all(err <= np.abs(up - xs)) and np.all(err <= np.abs(dn - xs))
    assert synth.round_f16_bits(np.array([1.0 + 2 ** -11]))[0] == 0x3C00


def test_deterministic_and_streams_differ():
    a = synth.gemm_inputs("w", "bf16", 8, 8, 8)
    b = synth.gemm_inputs("w", "bf16", 8, 8, 8)
    assert np.array_equal(a.A, b.A) and np.array_equal(a.C, b.C)
    assert not np.array_equal(a.A, a.B.reshape(a.A.shape))
    c = synth.gemm_inputs("w2", "bf16", 8, 8, 8)
    assert not np.array_equal(a.A, c.A)
    d = synth.gemm_inputs("w", "bf16", 8, 8, 8, seed=1)
    assert not np.array_equal(a.A, d.A)


def test_ranges_and_moments():
    u = synth.uniform_pm1(0, 5, 200000)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    z = synth.normal(0, 6, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    i8 = synth.int8_uniform(0, 7, 100000)
    assert i8.min() == -128 and i8.max() == 127
    c = synth.int_uniform(0, 8, 100000, -(1 << 20), 1 << 20)
    assert c.min() >= -(1 << 20) and c.max() <= (1 << 20)
    small = synth.int_uniform(0, 9, 20000, -2, 2)
    assert set(np.unique(small)) == {-2, -1, 0, 1, 2}


@pytest.mark.parametrize("dtype_in", ["f16", "bf16", "i8", "f64"])
def test_gemm_input_shapes(dtype_in):
    g = synth.gemm_inputs("shape", dtype_in, 5, 7, 3)
    assert g.A.shape == (5, 3) and g.B.shape == (7, 3) and g.C.shape == (5, 7)
    g = synth.gemm_inputs("shape", dtype_in, 5, 7, 3, b_layout="row")
    assert g.B.shape == (3, 7)


def test_batched_algorithmic_bytes():
    bi = synth.batched_inputs("b", "bf16", 64, group=4, abid=1)
    assert bi.A.shape == (64, 16, 16) and bi.B.shape == (64, 16, 16)
    # A: 16 of 64 tiles read (512 B each); B 512 B, C and D 1 KiB per entry
    assert bi.algorithmic_bytes() == 16 * 512 + 64 * 512 + 2 * 64 * 1024
