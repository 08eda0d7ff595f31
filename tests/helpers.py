"""Shared test utilities: device upload, padded copies, tolerance checks.

Tolerances (floating point), elementwise against the CPU oracle:
  FP16/BF16 -> FP32:  |D - D_ref| <= 1e-3 * (|A||B|)_ij + 1e-6
  FP64:               |D - D_ref| <= 1e-12 * (|A||B|)_ij + 2^-52 * |D_ref|_ij
(the second FP64 term is the final rounding of the sum with C, which the
first term does not cover when |A||B| is tiny next to |C|).  INT8 -> INT32
is bit-exact.
"""
from __future__ import annotations

import numpy as np

import oracle

TOL = {"f16": (1e-3, 1e-6), "bf16": (1e-3, 1e-6), "f64": (1e-12, 0.0)}


def torch_dev():
    import torch
    return torch.device("cuda:0")


def to_dev(x: np.ndarray, dtype_in: str | None = None):
    """Upload a numpy array; 16-bit float bit patterns become f16/bf16."""
    import torch
    dev = torch_dev()
    if x.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev)
        return t.view(torch.bfloat16 if dtype_in == "bf16" else torch.float16)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def padded(x: np.ndarray, align_bytes: int = 16, extra: int = 0,
           fill: int = 0x5A) -> np.ndarray:
    """Copy of a 2-D array whose rows are padded to a 16-byte multiple
    (plus `extra` elements), padding filled with garbage."""
    rows, cols = x.shape
    per = align_bytes // x.itemsize
    ld = ((cols + per - 1) // per) * per + extra * per
    big = np.empty((rows, ld), x.dtype)
    big.view(np.uint8)[:] = fill
    big[:, :cols] = x
    return big[:, :cols]


def dev_padded(x: np.ndarray, dtype_in: str | None = None, extra: int = 0):
    """Device tensor view (rows, cols) with a padded leading dimension."""
    p = padded(x, extra=extra)
    base = to_dev(p.base if p.base is not None else p, dtype_in)
    return base[:, : x.shape[1]]


def check(dtype_in: str, got: np.ndarray, want: np.ndarray,
          absab: np.ndarray | None, what: str = "") -> None:
    if dtype_in == "i8":
        if not np.array_equal(got, want):
            bad = np.argwhere(got != want)
            idx = tuple(int(v) for v in bad[0])
            raise AssertionError(f"{what}: {len(bad)} INT32 mismatches, first "
                                 f"at {idx}: {got[idx]} vs {want[idx]}")
        return
    rel, ab0 = TOL[dtype_in]
    g = got.astype(np.float64)
    w = want.astype(np.float64)
    err = np.abs(g - w)
    bound = rel * absab + ab0
    if dtype_in == "f64":
        bound = bound + np.abs(w) * 2.0 ** -52
    bad = err > bound
    if np.any(bad) or not np.all(np.isfinite(g)):
        idx = np.argwhere(bad | ~np.isfinite(g))
        i = tuple(idx[0])
        raise AssertionError(
            f"{what}: {len(idx)} of {got.size} outside tolerance; first at {i}: "
            f"got {g[i]!r} want {w[i]!r} bound {bound[i]:.3e}; "
            f"max err/bound {np.max(err / np.maximum(bound, 1e-300)):.3f}")


def decode16(bits: np.ndarray, dtype_in: str) -> np.ndarray:
    bits = np.asarray(bits, np.uint16)
    if dtype_in == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def check16(dtype_in: str, got_bits, want_bits, absab, what: str = "") -> None:
    """16-bit accumulate: |D - D_ref| <= 1e-3 (|A||B|)_ij + 1e-6 + one ulp of
    the 16-bit result (2^-10 |D_ref| for FP16, 2^-7 for BF16): the GPU rounds
    its FP32 sum to 16 bits, the oracle its double sum."""
    g = decode16(got_bits, dtype_in)
    w = decode16(want_bits, dtype_in)
    ulp = 2.0 ** -10 if dtype_in == "f16" else 2.0 ** -7
    bound = 1e-3 * absab + 1e-6 + ulp * np.abs(w)
    err = np.abs(g - w)
    bad = (err > bound) | ~np.isfinite(g)
    if np.any(bad):
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError(f"{what}: {len(idx)} of {g.size} outside tolerance; "
                             f"first at {i}: got {g[i]!r} want {w[i]!r} bound {bound[i]:.3e}")


def oracle_ref(g, rows=None, cols=None):
    """Oracle D (and |A||B|) for GemmInputs g, optionally on a sub-block."""
    A, B, C = g.A, g.B, g.C
    if rows is not None:
        A = np.ascontiguousarray(A[rows])
        C = np.ascontiguousarray(C[rows])
    if cols is not None:
        if g.b_layout == "col":
            B = np.ascontiguousarray(B[cols])
        else:
            B = np.ascontiguousarray(B[:, cols])
        C = np.ascontiguousarray(C[:, cols])
    if g.dtype_in == "i8":
        return oracle.gemm("i8", A, B, C, b_layout=g.b_layout), None
    return oracle.gemm(g.dtype_in, A, B, C, b_layout=g.b_layout,
                       want_absab=True)


# ------------------------------------------------------------ guard bands
#
# compute-sanitizer is not available to these tests, so out-of-bounds
# stores are caught with canaries instead: every output is embedded in a
# larger device buffer whose bytes outside the output all hold CANARY, and
# after the call each of those bytes must still hold it (the padding
# columns between N and the leading dimension, a guard row above and below
# the matrix, a guard entry before and after a batch).  A store from a
# ragged TMA box, a predicated warp-level store or a tile half that
# overhangs its problem changes one of them.

CANARY = 0xA5


def _torch_dtype(np_dtype, dtype_in=None):
    import torch
    m = {np.dtype(np.float32): torch.float32, np.dtype(np.float64): torch.float64,
         np.dtype(np.int32): torch.int32, np.dtype(np.int8): torch.int8,
         np.dtype(np.uint8): torch.uint8}
    if np.dtype(np_dtype) == np.dtype(np.uint16):
        return torch.bfloat16 if dtype_in == "bf16" else torch.float16
    return m[np.dtype(np_dtype)]


def _check_canary(buf, inside, what):
    """buf: device tensor; inside: boolean numpy mask over buf's bytes
    (True where the call may write)."""
    import torch
    torch.cuda.synchronize()
    raw = buf.contiguous().view(torch.uint8).cpu().numpy().reshape(inside.shape)
    bad = (raw != CANARY) & ~inside
    if np.any(bad):
        idx = np.argwhere(bad)
        raise AssertionError(f"{what}: {len(idx)} guard bytes overwritten, first at "
                             f"byte index {tuple(int(v) for v in idx[0])} "
                             f"(value 0x{int(raw[tuple(idx[0])]):02X})")


class GuardedMatrix:
    """An M x N device matrix inside a canary-filled buffer: `lead` guard
    rows above, `tail` below, and the leading dimension rounded up to 16
    bytes plus `pad` more 16-byte chunks of padding columns.  `view` is the
    matrix (pass it as C or D); `init` (numpy, M x N) fills it."""

    def __init__(self, M, N, np_dtype, *, dtype_in=None, init=None, pad=1,
                 lead=1, tail=1):
        import torch
        self.M, self.N = M, N
        esize = np.dtype(np_dtype).itemsize
        per = 16 // esize
        self.ld = ((N + per - 1) // per) * per + pad * per
        self.lead, self.tail, self.esize = lead, tail, esize
        rows = M + lead + tail
        flat = torch.full((rows * self.ld * esize,), CANARY, dtype=torch.uint8,
                          device=torch_dev())
        self.buf = flat.view(_torch_dtype(np_dtype, dtype_in)).view(rows, self.ld)
        self.view = self.buf[lead:lead + M, :N]
        if init is not None:
            self.view.copy_(to_dev(np.ascontiguousarray(init), dtype_in))

    def verify(self, what="guard"):
        rows = self.M + self.lead + self.tail
        inside = np.zeros((rows, self.ld * self.esize), bool)
        inside[self.lead:self.lead + self.M, :self.N * self.esize] = True
        _check_canary(self.buf, inside, what)


class GuardedBatch:
    """`batch` contiguous M x N tiles (tile stride M * ld, ld >= N) inside a
    canary-filled buffer with `lead` guard tiles before and `tail` after.
    With ld == N, `view` is the contiguous (batch, M, N) tensor the batched
    binding takes; `ptr` and `ld` serve raw C-ABI calls with ld > N."""

    def __init__(self, batch, M, N, np_dtype, *, dtype_in=None, init=None,
                 pad_cols=0, lead=1, tail=1):
        import torch
        self.batch, self.M, self.N = batch, M, N
        esize = np.dtype(np_dtype).itemsize
        self.esize = esize
        self.ld = N + pad_cols
        self.lead, self.tail = lead, tail
        tiles = batch + lead + tail
        flat = torch.full((tiles * M * self.ld * esize,), CANARY, dtype=torch.uint8,
                          device=torch_dev())
        self.buf = flat.view(_torch_dtype(np_dtype, dtype_in)).view(tiles, M, self.ld)
        self.tiles = self.buf[lead:lead + batch]          # (batch, M, ld)
        self.view = self.tiles if pad_cols == 0 else None
        self.ptr = self.tiles.data_ptr()
        if init is not None:
            self.tiles[:, :, :N].copy_(to_dev(np.ascontiguousarray(init), dtype_in))

    def result(self):
        """The (batch, M, N) outputs as a host array (16-bit floats as bits)."""
        import torch
        t = self.tiles[:, :, :self.N]
        if t.dtype in (torch.float16, torch.bfloat16):
            return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return t.contiguous().cpu().numpy()

    def verify(self, what="guard"):
        tiles = self.batch + self.lead + self.tail
        inside = np.zeros((tiles, self.M, self.ld * self.esize), bool)
        inside[self.lead:self.lead + self.batch, :, :self.N * self.esize] = True
        _check_canary(self.buf, inside, what)
