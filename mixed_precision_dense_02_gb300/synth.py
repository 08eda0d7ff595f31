"""Seeded synthetic inputs for the dense multiply-accumulate workloads.

This module only draws and encodes input values; it holds none of the
multiply-accumulate arithmetic.  Both the CUDA path's callers (tests, bench)
and the CPU oracle's callers take their inputs from here.

Random source: numpy's Philox-4x64 counter-based bit generator, keyed by
``(seed, stream)``; only its raw 64-bit words are used, and every transform
below is written out here so the values do not depend on numpy's
distribution code:

* uniform[-1, 1):   x = u53 * 2^-52 - 1          (u53 = top 53 bits, exact)
* N(0, 1):          Box-Muller, u1 in (0, 1], u2 in [0, 1):
                    r = sqrt(-2 ln u1), (r cos 2 pi u2, r sin 2 pi u2)
* int8 over [-128, 127] inclusive: one raw byte per value (exactly uniform)
* uint8 over [0, 255] inclusive: the same bytes read unsigned
* int32 over [-b, b] inclusive: rejection sampling on the smallest power-of-
  two range covering 2b + 1 values (exactly uniform)
* rounding to FP16 / BF16: round to nearest, ties to even, from the double.

Layouts follow the workloads: A is M x K row-major; B is stored column-major
(an N x K array, row j = column j of B) unless ``b_layout="row"`` (K x N);
C is M x N row-major.  16-bit float tensors are returned as ``uint16`` bit
patterns.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_TENSOR_IDS = {"A": 1, "B": 2, "C": 3}


def _bitgen(seed: int, stream: int) -> np.random.Philox:
    return np.random.Philox(key=np.array([seed, stream], dtype=np.uint64))


def stream_id(workload: str, tensor: str) -> int:
    """Stable 64-bit stream id for (workload name, tensor name)."""
    h = 1469598103934665603  # FNV-1a over the name, then the tensor id
    for ch in workload.encode():
        h = ((h ^ ch) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return ((h << 8) & 0xFFFFFFFFFFFFFFFF) | _TENSOR_IDS.get(tensor, 0)


def raw_u64(seed: int, stream: int, n: int) -> np.ndarray:
    return _bitgen(seed, stream).random_raw(int(n)).astype(np.uint64, copy=False)


def uniform_pm1(seed: int, stream: int, n: int) -> np.ndarray:
    """n doubles uniform on [-1, 1), each exactly u * 2^-52 - 1."""
    u = raw_u64(seed, stream, n) >> np.uint64(11)
    return u.astype(np.float64) * (2.0 ** -52) - 1.0


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """n doubles ~ N(0, 1) by the Box-Muller transform."""
    m = (int(n) + 1) // 2
    raw = raw_u64(seed, stream, 2 * m) >> np.uint64(11)
    u1 = (raw[0::2].astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = raw[1::2].astype(np.float64) * (2.0 ** -53)          # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * m, np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n]


def int8_uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """n int8 values uniform over the integers [-128, 127]."""
    words = (int(n) + 7) // 8
    return raw_u64(seed, stream, words).view(np.int8)[:n].copy()


def uint8_uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """n uint8 values uniform over the integers [0, 255]."""
    return int8_uniform(seed, stream, n).view(np.uint8)


def int_uniform(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n int64 values uniform over the integers [lo, hi] (rejection sampling)."""
    span = hi - lo + 1
    bits = int(span - 1).bit_length()
    mask = np.uint64((1 << bits) - 1)
    g = _bitgen(seed, stream)
    out = np.empty(0, np.int64)
    while out.size < n:
        need = int((n - out.size) * (1 << bits) / span * 1.05) + 64
        v = g.random_raw(need).astype(np.uint64) & mask
        v = v[v < np.uint64(span)].astype(np.int64) + lo
        out = np.concatenate([out, v])
    return out[:n]


def round_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round doubles to IEEE binary16 (nearest, ties to even); bit patterns."""
    return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def round_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite doubles to bfloat16 (nearest, ties to even); bit patterns.

    The double's significand is rounded to 8 bits with integer arithmetic on
    its bit pattern (so there is exactly one rounding), after which the value
    is exactly representable in float32 and its top 16 bits are the bf16.
    """
    x = np.asarray(x, np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("finite inputs only")
    b = x.view(np.uint64)
    drop = np.uint64(45)  # 52 - 7 fraction bits dropped
    half = np.uint64((1 << 44) - 1)
    lsb = (b >> drop) & np.uint64(1)
    b = (b + half + lsb) & ~np.uint64((1 << 45) - 1)
    f = b.view(np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class GemmInputs:
    dtype_in: str          # "f16" | "bf16" | "i8" | "f64" ("i8": A and B
                           # are int8 or uint8 arrays, see gemm_inputs)
    M: int
    N: int
    K: int
    A: np.ndarray          # M x K row-major
    B: np.ndarray          # stored: N x K (col) or K x N (row)
    C: np.ndarray          # M x N row-major
    b_layout: str = "col"

    @property
    def nbytes(self) -> int:
        return self.A.nbytes + self.B.nbytes + 2 * self.C.nbytes


def _floats(dist: str, seed: int, stream: int, n: int) -> np.ndarray:
    if dist == "uniform":
        return uniform_pm1(seed, stream, n)
    if dist == "normal":
        return normal(seed, stream, n)
    raise ValueError(dist)


def gemm_inputs(workload: str, dtype_in: str, M: int, N: int, K: int, *,
                dist: str = "normal", c_dist: str = "normal", seed: int = 0,
                b_layout: str = "col", c_int_bound: int = 1 << 20,
                c_int_range: tuple | None = None, acc16: bool = False,
                a_signed: bool = True, b_signed: bool = True) -> GemmInputs:
    """Inputs of one D = A*B + C problem.

    ``dist`` is the A/B distribution ("uniform" on [-1, 1) or "normal"),
    rounded to the input type; ``c_dist`` the C distribution (FP32/FP64:
    normal; INT32: uniform over [-c_int_bound, c_int_bound], or over the
    inclusive ``c_int_range`` when given).  With ``acc16`` (FP16/BF16 only)
    C is rounded to the input's 16-bit type.  For "i8", ``a_signed`` /
    ``b_signed`` False draw that operand as uint8 over [0, 255].
    """
    sA, sB, sC = (stream_id(workload, t) for t in "ABC")
    bshape = (N, K) if b_layout == "col" else (K, N)
    if dtype_in in ("f16", "bf16"):
        rnd = round_f16_bits if dtype_in == "f16" else round_bf16_bits
        A = rnd(_floats(dist, seed, sA, M * K)).reshape(M, K)
        B = rnd(_floats(dist, seed, sB, N * K)).reshape(bshape)
        C = _floats(c_dist, seed, sC, M * N)
        C = (rnd(C) if acc16 else C.astype(np.float32)).reshape(M, N)
    elif dtype_in == "i8":
        A = (int8_uniform if a_signed else uint8_uniform)(seed, sA, M * K).reshape(M, K)
        B = (int8_uniform if b_signed else uint8_uniform)(seed, sB, N * K).reshape(bshape)
        lo, hi = c_int_range if c_int_range else (-c_int_bound, c_int_bound)
        C = int_uniform(seed, sC, M * N, lo, hi).astype(np.int32).reshape(M, N)
    elif dtype_in == "f64":
        A = _floats(dist, seed, sA, M * K).reshape(M, K)
        B = _floats(dist, seed, sB, N * K).reshape(bshape)
        C = _floats(c_dist, seed, sC, M * N).reshape(M, N)
    else:
        raise ValueError(dtype_in)
    return GemmInputs(dtype_in, M, N, K, A, B, C, b_layout)


@dataclass
class BatchedInputs:
    dtype_in: str
    batch: int
    M: int
    N: int
    K: int
    group: int
    abid: int
    A: np.ndarray          # (batch, M, K); entry b reads tile (b//G)*G + abid
    B: np.ndarray          # (batch, N, K) column-major tiles
    C: np.ndarray          # (batch, M, N)
    blgp: int = 0          # B lane-group pattern (groups of four entries)

    def algorithmic_bytes(self) -> int:
        """A read once per group, the B tiles that are read once, C read
        once, D written once."""
        a_tile = self.M * self.K * self.A.itemsize
        b_tile = self.N * self.K * self.B.itemsize
        b_read = {0: 4, 1: 2, 2: 2, 3: 4}.get(self.blgp, 1)  # per group of 4
        n_b = self.batch if self.blgp == 0 else (self.batch // 4) * b_read
        return ((self.batch // self.group) * a_tile + n_b * b_tile
                + self.C.nbytes + self.C.nbytes)


def batched_inputs(workload: str, dtype_in: str, batch: int, M: int = 16,
                   N: int = 16, K: int = 16, *, group: int = 4, abid: int = 1,
                   dist: str = "uniform", seed: int = 0, blgp: int = 0,
                   acc16: bool = False) -> BatchedInputs:
    """Contiguous per-tile batched inputs (A allocated with ``batch`` tiles).
    With ``acc16`` (FP16/BF16) C is rounded to the input's 16-bit type."""
    sA, sB, sC = (stream_id(workload, t) for t in "ABC")
    if dtype_in in ("f16", "bf16"):
        rnd = round_f16_bits if dtype_in == "f16" else round_bf16_bits
        A = rnd(_floats(dist, seed, sA, batch * M * K)).reshape(batch, M, K)
        B = rnd(_floats(dist, seed, sB, batch * N * K)).reshape(batch, N, K)
        C = normal(seed, sC, batch * M * N)
        C = (rnd(C) if acc16 else C.astype(np.float32)).reshape(batch, M, N)
    elif dtype_in == "i8":
        A = int8_uniform(seed, sA, batch * M * K).reshape(batch, M, K)
        B = int8_uniform(seed, sB, batch * N * K).reshape(batch, N, K)
        C = int_uniform(seed, sC, batch * M * N, -(1 << 20), 1 << 20).astype(np.int32).reshape(batch, M, N)
    elif dtype_in == "f64":
        A = _floats(dist, seed, sA, batch * M * K).reshape(batch, M, K)
        B = _floats(dist, seed, sB, batch * N * K).reshape(batch, N, K)
        C = normal(seed, sC, batch * M * N).reshape(batch, M, N)
    else:
        raise ValueError(dtype_in)
    return BatchedInputs(dtype_in, batch, M, N, K, group, abid, A, B, C, blgp)


# The workloads, by what they are.
WORKLOADS = {
    "gemm_f16_256": dict(kind="gemm", dtype_in="f16", M=256, N=256, K=256,
                         dist="uniform"),
    "gemm_i8_4096": dict(kind="gemm", dtype_in="i8", M=4096, N=4096, K=4096),
    "batched_bf16_16x16x16_b262144_g4_abid1": dict(
        kind="batched", dtype_in="bf16", batch=262144, M=16, N=16, K=16,
        group=4, abid=1, dist="uniform"),
    "gemm_bf16_8192": dict(kind="gemm", dtype_in="bf16", M=8192, N=8192,
                           K=8192, dist="normal"),
    "gemm_f64_4096_rowB": dict(kind="gemm", dtype_in="f64", M=4096, N=4096,
                               K=4096, dist="normal", b_layout="row"),
    "gemm_bf16_skinny_16384x128x4096": dict(kind="gemm", dtype_in="bf16",
                                            M=16384, N=128, K=4096,
                                            dist="normal"),
    # BF16 -> BF16 accumulate (16-bit addend and result), large square shape
    "gemm_bf16_acc16_8192": dict(kind="gemm", dtype_in="bf16", M=8192, N=8192,
                                 K=8192, dist="normal", acc16=True),
    # batched 32 x 32 x 32 blocks (the warp-level streaming kernel), groups
    # of 4 with source 1
    "batched_bf16_32x32x32_b65536_g4_abid1": dict(
        kind="batched", dtype_in="bf16", batch=65536, M=32, N=32, K=32,
        group=4, abid=1, dist="uniform"),
    # batched 32 x 32 x 32 INT8 blocks (the integer streaming kernel),
    # groups of 4 with source 1
    "batched_i8_32x32x32_b65536_g4_abid1": dict(
        kind="batched", dtype_in="i8", batch=65536, M=32, N=32, K=32,
        group=4, abid=1),
    # batched 64 x 64 x 64 blocks (the CTA-cooperative tile kernel), groups
    # of 4 with source 1
    "batched_bf16_64x64x64_b16384_g4_abid1": dict(
        kind="batched", dtype_in="bf16", batch=16384, M=64, N=64, K=64,
        group=4, abid=1, dist="uniform"),
    # batched 128 x 128 x 128 tiles (larger blocks than the 16^3 form) with
    # the A block of each group of 4 broadcast from entry 1 of the group
    "batched_bf16_128x128x128_b8192_g4_abid1": dict(
        kind="batched", dtype_in="bf16", batch=8192, M=128, N=128, K=128,
        group=4, abid=1, dist="uniform"),
    # unsigned x unsigned 8-bit inputs with INT32 saturation; C spans the
    # whole INT32 range, so the outputs whose C lies within the product sum
    # of the top (about 1.6% of them) saturate
    "gemm_u8_4096_clamp": dict(kind="gemm", dtype_in="i8", M=4096, N=4096,
                               K=4096, a_signed=False, b_signed=False,
                               clamp=True,
                               c_int_range=(-(1 << 31), (1 << 31) - 1)),
    # few output tiles (64 of 128 x 128) over a deep K: the tiles' K steps
    # are split over every SM (stream-K)
    "gemm_bf16_deepk_1024x1024x32768": dict(kind="gemm", dtype_in="bf16",
                                            M=1024, N=1024, K=32768,
                                            dist="normal"),
}


def workload_gemm_inputs(name: str, seed: int = 0) -> GemmInputs:
    """The inputs of a named GEMM workload."""
    w = WORKLOADS[name]
    return gemm_inputs(name, w["dtype_in"], w["M"], w["N"], w["K"],
                       dist=w.get("dist", "normal"),
                       b_layout=w.get("b_layout", "col"), seed=seed,
                       acc16=w.get("acc16", False),
                       c_int_range=w.get("c_int_range"),
                       a_signed=w.get("a_signed", True),
                       b_signed=w.get("b_signed", True))
