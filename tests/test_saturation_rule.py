"""The rule by which the saturating 8-bit GEMM recovers clamp(S + C) from
S + C modulo 2^32 and the sign of C, when the exact product S lies in
(-2^30, 2^30) and C is any INT32.  S + C then lies in (-3 * 2^30, 3 * 2^30);
for C >= 0 it exceeds INT32_MAX exactly when the wrapped value is below
-2^30, for C < 0 it falls below INT32_MIN exactly when the wrapped value is
at least 2^30.  The check is exhaustive over the edges of both ranges and
random elsewhere; it is the arithmetic the kernel's emission relies on (the
kernel itself is compared with the oracle by the GPU tests)."""
from __future__ import annotations

import numpy as np

I32_MIN, I32_MAX = -(1 << 31), (1 << 31) - 1
B = 1 << 30


def _recover(S, C):
    T = S + C
    v = ((T + (1 << 32)) % (1 << 32)).astype(np.uint32).view(np.int32).astype(np.int64)
    neg = C < 0
    return np.where(~neg & (v < -B), I32_MAX, np.where(neg & (v >= B), I32_MIN, v))


def test_edges_exhaustive():
    s_edges = np.array([-B + 1, -B + 2, -B + 3, -2, -1, 0, 1, 2, B - 3, B - 2, B - 1],
                       np.int64)
    c_edges = []
    for base in (I32_MIN, -B - 1, -B, -1, 0, 1, B - 1, B, I32_MAX):
        c_edges.extend(base + d for d in range(-3, 4))
    c_edges = np.array([c for c in c_edges if I32_MIN <= c <= I32_MAX], np.int64)
    # C = target - S for targets at both ends of the INT32 range
    S, C = np.meshgrid(s_edges, c_edges)
    S, C = S.ravel(), C.ravel()
    for t in (I32_MAX - 1, I32_MAX, I32_MAX + 1, I32_MIN - 1, I32_MIN, I32_MIN + 1):
        c = t - s_edges
        ok = (c >= I32_MIN) & (c <= I32_MAX)
        S = np.concatenate([S, s_edges[ok]])
        C = np.concatenate([C, c[ok]])
    want = np.clip(S + C, I32_MIN, I32_MAX)
    assert np.array_equal(_recover(S, C), want)


def test_random_pairs():
    rng = np.random.default_rng(2024)
    S = rng.integers(-B + 1, B, 2_000_000)
    C = rng.integers(I32_MIN, I32_MAX, 2_000_000, endpoint=True)
    assert np.array_equal(_recover(S, C), np.clip(S + C, I32_MIN, I32_MAX))


def test_bound_is_needed():
    """At |S| = 2^30 + 1 the wrapped value no longer decides: two pairs with
    the same wrapped sum and the same sign of C have different clamps."""
    s1, c1 = B + 1, I32_MAX          # S + C = 3 * 2^30: saturates high
    s2, c2 = -B - 1, 1               # S + C = -2^30: in range
    # the same value modulo 2^32, and C >= 0 in both
    assert (s1 + c1) - (1 << 32) == s2 + c2 == -B
    assert np.clip(s1 + c1, I32_MIN, I32_MAX) != np.clip(s2 + c2, I32_MIN, I32_MAX)
