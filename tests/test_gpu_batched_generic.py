"""Parity of the batched products of any M x N x K (mma_gemm_batched_ex)
with the CPU oracle: A-block broadcast (cbsz/abid of "Common MFMA
parameters", section "Shared parameters") and the B lane-group pattern
(blgp, section "Dense MFMA parameters", read at matrix level) on every
dtype pair.

Shapes span one and several tiles per entry, ragged M/N/K edges inside each
entry (the tensor maps' batch coordinate keeps a tile's overhang from
reading the next entry), the CTA-pair path (M > 128 with enough work), and
16 x 16 x 16 tiles on the HBM-streaming kernel with every blgp pattern.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from mixed_precision_dense_02_gb300 import binding, synth

from helpers import TOL, GuardedBatch, check, check16, to_dev

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


OUT_NP = {"f16": np.float32, "bf16": np.float32, "i8": np.int32, "f64": np.float64}


def run(bi, *, use_c=True, acc=None):
    """The batched call with D inside a guard band (a canary tile before
    and after the batch); 16-bit results come back as bit patterns."""
    out16 = acc == "same" or (use_c and bi.C.dtype == np.uint16)
    Gd = GuardedBatch(bi.batch, bi.M, bi.N, np.uint16 if out16 else OUT_NP[bi.dtype_in],
                      dtype_in=bi.dtype_in)
    binding.gemm_batched(to_dev(bi.A, bi.dtype_in), to_dev(bi.B, bi.dtype_in),
                         to_dev(bi.C, bi.dtype_in) if use_c else None, Gd.view,
                         group=bi.group, abid=bi.abid, blgp=bi.blgp, acc=acc)
    Gd.verify(f"batched {bi.dtype_in} {bi.M}x{bi.N}x{bi.K} x{bi.batch} D guard")
    return Gd.result()


def absab(bi):
    """(|A| |B|) per output, the scale of the floating-point tolerance."""
    if bi.dtype_in in ("f16", "bf16"):
        a, b = bi.A & 0x7FFF, bi.B & 0x7FFF
    else:
        a, b = np.abs(bi.A), np.abs(bi.B)
    return oracle.gemm_batched(bi.dtype_in, a, b, None, group=bi.group,
                               abid=bi.abid, blgp=bi.blgp).astype(np.float64)


def want(bi, use_c=True):
    return oracle.gemm_batched(bi.dtype_in, bi.A, bi.B, bi.C if use_c else None,
                               group=bi.group, abid=bi.abid, blgp=bi.blgp)


# (M, N, K): K a multiple of 8 (16-bit rows of 16 bytes), N of 4 (FP32 rows)
SHAPES = [(24, 40, 32), (128, 128, 64), (130, 200, 136), (64, 264, 520),
          (1, 8, 8), (200, 4, 1000)]
GROUPS = [(1, 0, 0), (4, 1, 0), (2, 1, 3), (16, 15, 5), (8, 3, 1), (4, 2, 7)]


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("G,abid,blgp", GROUPS)
def test_generic_f16_bf16(dtype_in, M, N, K, G, abid, blgp):
    bi = synth.batched_inputs(f"bg_{M}_{N}_{K}", dtype_in, 16, M=M, N=N, K=K,
                              group=G, abid=abid, blgp=blgp)
    check(dtype_in, run(bi), want(bi), absab(bi),
          f"{dtype_in} {M}x{N}x{K} G={G} abid={abid} blgp={blgp}")


def test_generic_no_c_and_pair_path():
    """C = None, and entries with M > 128, more than 2^30 multiply-adds and
    at least one 256 x 256 pair tile per CTA pair (the CTA-pair kernel):
    80 entries of 256 x 256 x 256."""
    bi = synth.batched_inputs("bg_pair", "bf16", 80, M=256, N=256, K=256,
                              group=4, abid=3, blgp=3)
    check("bf16", run(bi, use_c=False), want(bi, use_c=False), absab(bi),
          "bf16 256^3 x 80, pair path, no C")
    # ragged M (300 = 256 + 44) on pairs: 100 entries, 2^30 multiply-adds
    bi = synth.batched_inputs("bg_pair_r", "f16", 100, M=300, N=136, K=264,
                              group=2, abid=0, blgp=6)
    check("f16", run(bi), want(bi), absab(bi), "f16 300x136x264 x 100, ragged pair")


@pytest.mark.parametrize("M,N,K,G,abid,blgp", [(24, 40, 32, 4, 1, 0),
                                               (130, 200, 1040, 2, 1, 3),
                                               (256, 128, 2048, 4, 0, 4)])
def test_generic_i8_exact(M, N, K, G, abid, blgp):
    bi = synth.batched_inputs(f"bg_i8_{M}", "i8", 16, M=M, N=N, K=K, group=G,
                              abid=abid, blgp=blgp)
    check("i8", run(bi), want(bi), None, f"i8 {M}x{N}x{K} G={G} blgp={blgp}")


@pytest.mark.parametrize("M,N,K,G,abid,blgp", [(24, 40, 32, 4, 1, 0),
                                               (130, 66, 70, 2, 1, 3),
                                               (64, 64, 64, 16, 7, 5)])
def test_generic_f64(M, N, K, G, abid, blgp):
    bi = synth.batched_inputs(f"bg_f64_{M}", "f64", 16, M=M, N=N, K=K, group=G,
                              abid=abid, blgp=blgp)
    got, w = run(bi), want(bi)
    ab = absab(bi)
    check("f64", got, w, ab, f"f64 {M}x{N}x{K}")


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,G,abid,blgp", [(24, 40, 32, 4, 1, 2),
                                               (136, 264, 200, 8, 6, 3)])
def test_generic_16bit_accumulate(dtype_in, M, N, K, G, abid, blgp):
    """FP16->FP16 / BF16->BF16: each entry against the single-problem
    16-bit-accumulate oracle on the tiles the source maps select."""
    bi = synth.batched_inputs(f"bg_h_{M}", dtype_in, 16, M=M, N=N, K=K,
                              group=G, abid=abid, blgp=blgp, acc16=True)
    got = run(bi, acc="same")
    for b in range(bi.batch):
        sa = (b // G) * G + abid
        sb = (b // 4) * 4 + oracle.blgp_source(blgp, b % 4)
        w, ab = oracle.gemm_acc16(dtype_in, bi.A[sa], bi.B[sb], bi.C[b],
                                  want_absab=True)
        check16(dtype_in, got[b], w, ab, f"{dtype_in}->16 entry {b}")


@pytest.mark.parametrize("blgp", range(8))
def test_16x16x16_every_blgp(blgp):
    """16^3 tiles take the HBM-streaming kernel; every lane-group pattern,
    with an A broadcast at the same time."""
    bi = synth.batched_inputs(f"b16_blgp_{blgp}", "bf16", 1024, group=4, abid=2,
                              blgp=blgp)
    check("bf16", run(bi), want(bi), absab(bi), f"16^3 blgp={blgp}")


@pytest.mark.parametrize("path", ["stream", "tcgen05"])
def test_blgp_identifies_source_tiles(path):
    """B tile t = (t+1) I, A = I, C = 0: D_b = (bsrc(b)+1) I, read off D,
    for the rotation pattern (3) on both batched kernels."""
    import torch
    n = 16 if path == "stream" else 24
    batch = 8
    eye = np.eye(n, dtype=bool)
    A = np.broadcast_to(np.where(eye, np.uint16(0x3F80), np.uint16(0)),
                        (batch, n, n)).copy()
    B = np.zeros((batch, n, n), np.uint16)
    for t in range(batch):
        B[t] = np.where(eye, synth.round_bf16_bits(np.array([t + 1.0]))[0], 0)
    D = binding.gemm_batched(to_dev(A, "bf16"), to_dev(B, "bf16"), None, blgp=3)
    torch.cuda.synchronize()
    D = D.cpu().numpy()
    for b in range(batch):
        src = (b // 4) * 4 + (b + 1) % 4
        assert np.array_equal(D[b], (src + 1) * np.eye(n, dtype=np.float32)), b


def test_k_zero_and_empty():
    import torch
    bi = synth.batched_inputs("bg_k0", "bf16", 8, M=24, N=40, K=8, group=2, abid=1)
    dev = torch.device("cuda:0")
    A = torch.zeros((8, 24, 0), dtype=torch.bfloat16, device=dev)
    B = torch.zeros((8, 40, 0), dtype=torch.bfloat16, device=dev)
    C = to_dev(bi.C)
    D = binding.gemm_batched(A, B, C, group=2, abid=1)
    torch.cuda.synchronize()
    assert torch.equal(D, C)


@pytest.mark.parametrize("name", ["batched_bf16_128x128x128_b8192_g4_abid1",
                                  "batched_bf16_64x64x64_b16384_g4_abid1",
                                  "batched_bf16_32x32x32_b65536_g4_abid1",
                                  "batched_i8_32x32x32_b65536_g4_abid1"])
def test_full_size_generic_batched_workload(name):
    """The batched workloads of 128^3 BF16 blocks (tensor-memory GEMM), 64^3
    BF16 blocks (CTA-cooperative tile kernel), 32^3 BF16 blocks (warp-level
    streaming kernel) and 32^3 INT8 blocks (integer streaming kernel),
    groups of 4 (source 1): sampled entries (and the
    last) against the oracle on those entries' tiles; BF16 outputs finite,
    INT8 bit-exact."""
    import torch
    w = synth.WORKLOADS[name]
    dt = w["dtype_in"]
    bi = synth.batched_inputs(name, dt, w["batch"], M=w["M"], N=w["N"],
                              K=w["K"], group=w["group"], abid=w["abid"],
                              dist=w.get("dist", "uniform"))
    D = binding.gemm_batched(to_dev(bi.A, dt), to_dev(bi.B, dt),
                             to_dev(bi.C), group=bi.group, abid=bi.abid)
    torch.cuda.synchronize()
    if dt != "i8":
        assert bool(torch.isfinite(D).all())
    rng = np.random.default_rng(99)
    ents = np.unique(np.append(rng.choice(bi.batch, 63, replace=False), bi.batch - 1))
    src = (ents // bi.group) * bi.group + bi.abid
    A, B, C = (np.ascontiguousarray(x) for x in (bi.A[src], bi.B[ents], bi.C[ents]))
    want = oracle.gemm_batched(dt, A, B, C)
    got = D[torch.from_numpy(ents).cuda()].cpu().numpy()
    if dt == "i8":
        check("i8", got, want, None, name)
        return
    ab = oracle.gemm_batched(dt, A & 0x7FFF, B & 0x7FFF, None).astype(np.float64)
    check(dt, got, want, ab, name)


# Dense blocks with M, N, K multiples of 16 and at most 96 * 96 * 64
# multiply-adds take the warp-level streaming kernel (32 x 32 warp tiles
# when M and N are multiples of 32, else 16 x 16; K in 32-deep chunks plus
# a tail); (128, 128, 128) just beyond the limit takes the tensor-memory
# GEMM.
STREAM_SHAPES = [(32, 32, 32), (64, 64, 64), (16, 48, 80), (96, 64, 96),
                 (64, 64, 144), (48, 16, 16), (32, 96, 16), (128, 128, 128)]


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", STREAM_SHAPES)
@pytest.mark.parametrize("G,abid,blgp", [(1, 0, 0), (4, 1, 3), (8, 6, 5)])
def test_streaming_kernel_shapes(dtype_in, M, N, K, G, abid, blgp):
    bi = synth.batched_inputs(f"bs_{M}_{N}_{K}", dtype_in, 64, M=M, N=N, K=K,
                              group=G, abid=abid, blgp=blgp)
    check(dtype_in, run(bi), want(bi), absab(bi),
          f"{dtype_in} {M}x{N}x{K} G={G} blgp={blgp}")


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(32, 32, 32), (16, 48, 80), (64, 64, 144)])
def test_streaming_kernel_16bit_and_no_c(dtype_in, M, N, K):
    bi = synth.batched_inputs(f"bs_h_{M}", dtype_in, 32, M=M, N=N, K=K,
                              group=2, abid=1, blgp=2, acc16=True)
    got = run(bi, acc="same")
    for b in range(bi.batch):
        sa = (b // 2) * 2 + 1
        sb = (b // 4) * 4 + oracle.blgp_source(2, b % 4)
        w, ab = oracle.gemm_acc16(dtype_in, bi.A[sa], bi.B[sb], bi.C[b],
                                  want_absab=True)
        check16(dtype_in, got[b], w, ab, f"{dtype_in}->16 {M}x{N}x{K} entry {b}")
    bf = synth.batched_inputs(f"bs_n_{M}", dtype_in, 32, M=M, N=N, K=K,
                              group=4, abid=0, blgp=7)
    check(dtype_in, run(bf, use_c=False), want(bf, use_c=False), absab(bf),
          f"{dtype_in} {M}x{N}x{K} no C")


# INT8 blocks up to 128^3 multiply-adds take the integer streaming kernel
I8_STREAM_SHAPES = [(16, 16, 16), (32, 32, 32), (64, 64, 64), (16, 48, 80),
                    (96, 64, 96), (32, 96, 48), (128, 128, 128)]


@pytest.mark.parametrize("M,N,K", I8_STREAM_SHAPES)
@pytest.mark.parametrize("G,abid,blgp", [(1, 0, 0), (4, 1, 3), (16, 5, 6)])
def test_streaming_kernel_int8_exact(M, N, K, G, abid, blgp):
    """Small and mid-size INT8 blocks on the integer warp-level kernel (K a
    multiple of 16: the last 32-deep step of K = 16, 48, 80 is half empty
    and reads as zero), bit-exact."""
    bi = synth.batched_inputs(f"bs_i8_{M}_{N}_{K}", "i8", 64, M=M, N=N, K=K,
                              group=G, abid=abid, blgp=blgp)
    check("i8", run(bi), want(bi), None, f"i8 {M}x{N}x{K} G={G} blgp={blgp}")
    check("i8", run(bi, use_c=False), want(bi, use_c=False), None,
          f"i8 {M}x{N}x{K} no C")


def test_streaming_kernel_int8_wraps_like_int32():
    """Every product 127 * 127 with C at the top of INT32: D wraps modulo
    2^32 exactly as an INT32 accumulator does (closed form)."""
    import torch
    batch, M, N, K = 8, 32, 32, 64
    A = np.full((batch, M, K), 127, np.int8)
    B = np.full((batch, N, K), 127, np.int8)
    C = np.full((batch, M, N), 2 ** 31 - 100, np.int32)
    D = binding.gemm_batched(to_dev(A), to_dev(B), to_dev(C), group=2, abid=1)
    torch.cuda.synchronize()
    exact = 2 ** 31 - 100 + K * 127 * 127
    assert np.all(D.cpu().numpy() == np.int32(exact - 2 ** 32))


# FP16/BF16 blocks with M, N, K multiples of 64 and at most 2^20
# multiply-adds take the CTA-cooperative kernel (64 x 64 CTA tiles, operands
# staged once per tile through a cp.async ring crossing tile boundaries)
TILE_SHAPES = [(64, 64, 64), (128, 64, 128), (64, 128, 64), (128, 128, 64),
               (64, 64, 256), (64, 192, 64)]


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", TILE_SHAPES)
@pytest.mark.parametrize("G,abid,blgp", [(1, 0, 0), (4, 3, 3), (16, 9, 4)])
def test_cooperative_tile_kernel(dtype_in, M, N, K, G, abid, blgp):
    bi = synth.batched_inputs(f"bt_{M}_{N}_{K}", dtype_in, 48, M=M, N=N, K=K,
                              group=G, abid=abid, blgp=blgp)
    check(dtype_in, run(bi), want(bi), absab(bi),
          f"{dtype_in} {M}x{N}x{K} G={G} blgp={blgp}")


@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("K", [64, 128])   # C staged in shared memory / read directly
def test_cooperative_tile_kernel_16bit_and_no_c(dtype_in, K):
    M, N = 64, 128
    bi = synth.batched_inputs(f"bt_h{K}", dtype_in, 32, M=M, N=N, K=K, group=2,
                              abid=1, blgp=1, acc16=True)
    got = run(bi, acc="same")
    for b in range(bi.batch):
        sa = (b // 2) * 2 + 1
        sb = (b // 4) * 4 + oracle.blgp_source(1, b % 4)
        w, ab = oracle.gemm_acc16(dtype_in, bi.A[sa], bi.B[sb], bi.C[b],
                                  want_absab=True)
        check16(dtype_in, got[b], w, ab, f"{dtype_in}->16 tile entry {b}")
    bf = synth.batched_inputs(f"bt_n{K}", dtype_in, 40, M=M, N=N, K=K, group=4,
                              abid=0, blgp=5)
    check(dtype_in, run(bf, use_c=False), want(bf, use_c=False), absab(bf),
          f"{dtype_in} tile kernel no C")


_FORCED_TILE_SCRIPT = """
import sys, numpy as np, torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + '/tests']
from mixed_precision_dense_02_gb300 import binding, synth
from helpers import to_dev
binding.load()
out = {}
for (M, N, K, dt) in [(128, 128, 128, 'bf16'), (256, 256, 64, 'f16'),
                      (128, 128, 256, 'bf16')]:
    bi = synth.batched_inputs(f'btf_{M}_{N}_{K}', dt, 24, M=M, N=N, K=K,
                              group=4, abid=2, blgp=6)
    D = binding.gemm_batched(to_dev(bi.A, dt), to_dev(bi.B, dt), to_dev(bi.C),
                             group=4, abid=2, blgp=6)
    torch.cuda.synchronize()
    out[f'{M}_{N}_{K}_{dt}'] = D.cpu().numpy()
binding.device_status()
np.savez(sys.argv[2], **out)
"""


def test_cooperative_tile_kernel_forced_on_larger_blocks(tmp_path):
    """MMA_GB300_BATCHED=tile sends blocks above the routing threshold (128^3,
    256 x 256 x 64, 128 x 128 x 256) to the CTA-cooperative kernel; run in a
    child process (the override is read once per process) and compared
    with the oracle here."""
    import os
    import pathlib
    import subprocess
    import sys
    root = str(pathlib.Path(__file__).resolve().parents[1])
    out = tmp_path / "forced_tile.npz"
    env = dict(os.environ, MMA_GB300_BATCHED="tile")
    r = subprocess.run([sys.executable, "-c", _FORCED_TILE_SCRIPT, root, str(out)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = np.load(out)
    for (M, N, K, dt) in [(128, 128, 128, "bf16"), (256, 256, 64, "f16"),
                          (128, 128, 256, "bf16")]:
        bi = synth.batched_inputs(f"btf_{M}_{N}_{K}", dt, 24, M=M, N=N, K=K,
                                  group=4, abid=2, blgp=6)
        check(dt, got[f"{M}_{N}_{K}_{dt}"], want(bi), absab(bi),
              f"forced tile {dt} {M}x{N}x{K}")


# C and D the same buffer (in place): every batched kernel reads an
# output's addend before it writes that output
INPLACE_CASES = [
    ("bf16", 16, 16, 16, 64),     # 16^3 streaming kernel
    ("bf16", 32, 32, 32, 64),     # warp-level streaming kernel
    ("f16", 64, 64, 64, 32),      # CTA-cooperative tile kernel, C staged
    ("bf16", 64, 128, 128, 32),   # CTA-cooperative tile kernel, C direct
    ("bf16", 128, 128, 128, 16),  # tensor-memory GEMM
    ("i8", 32, 32, 32, 64),       # integer streaming kernel
    ("i8", 160, 96, 64, 8),       # INT8 on the tensor-memory GEMM
    ("f64", 24, 40, 16, 8),       # FP64 DMMA tiles
]


@pytest.mark.parametrize("dtype_in,M,N,K,batch", INPLACE_CASES)
def test_batched_in_place(dtype_in, M, N, K, batch):
    import torch
    bi = synth.batched_inputs(f"bip_{M}_{N}_{K}", dtype_in, batch, M=M, N=N,
                              K=K, group=4, abid=3, blgp=2)
    Gc = GuardedBatch(batch, M, N, OUT_NP[dtype_in], init=bi.C)
    C = Gc.view
    D = binding.gemm_batched(to_dev(bi.A, dtype_in), to_dev(bi.B, dtype_in), C,
                             C, group=4, abid=3, blgp=2)
    Gc.verify(f"{dtype_in} {M}x{N}x{K} in place guard")
    assert D.data_ptr() == C.data_ptr()
    check(dtype_in, Gc.result(), want(bi), absab(bi) if dtype_in != "i8" else None,
          f"{dtype_in} {M}x{N}x{K} in place")


@pytest.mark.parametrize("in_place", [False, True])
def test_batched_i8_tensor_memory_long_k(in_place):
    """Batched INT8 on the tensor-memory GEMM with three 1024-deep chunks
    per tile, where C joins the INT32 sums during the chunk phase through
    the entry's own tensor-map coordinate; broadcast and B pattern on."""
    import torch
    bi = synth.batched_inputs("bi8_long_k", "i8", 8, M=144, N=96, K=3072,
                              group=4, abid=3, blgp=2)
    C = to_dev(bi.C)
    D = binding.gemm_batched(to_dev(bi.A, "i8"), to_dev(bi.B, "i8"), C,
                             C if in_place else None, group=4, abid=3, blgp=2)
    torch.cuda.synchronize()
    check("i8", D.cpu().numpy(), want(bi), None, f"batched i8 long K in_place={in_place}")


# Batched outputs with padding columns (ldc = ldd > N, tile stride M * ld)
# through the raw C ABI, inside guard bands: nothing may be written to the
# padding columns of any tile, nor before the first or after the last tile.
PADDED_LD_CASES = [
    ("bf16", 16, 16, 16, 64, 4),
    ("bf16", 32, 32, 32, 64, 4),
    ("f16", 64, 64, 64, 32, 8),
    ("bf16", 64, 128, 128, 16, 4),
    ("bf16", 128, 128, 128, 16, 4),
    ("bf16", 100, 72, 40, 12, 4),
    ("i8", 32, 32, 32, 64, 4),
    ("i8", 160, 96, 64, 8, 4),
    ("f64", 24, 40, 16, 8, 2),
]


@pytest.mark.parametrize("dtype_in,M,N,K,batch,pad", PADDED_LD_CASES)
def test_batched_padded_ld_guard(dtype_in, M, N, K, batch, pad):
    import torch
    bi = synth.batched_inputs(f"bpld_{dtype_in}_{M}_{N}_{K}", dtype_in, batch, M=M,
                              N=N, K=K, group=2, abid=1, blgp=7)
    codes = {"f16": (binding.MMA_F16, binding.MMA_F32),
             "bf16": (binding.MMA_BF16, binding.MMA_F32),
             "i8": (binding.MMA_I8, binding.MMA_I32),
             "f64": (binding.MMA_F64, binding.MMA_F64)}[dtype_in]
    out_dt = OUT_NP[dtype_in]
    Gc = GuardedBatch(batch, M, N, out_dt, init=bi.C, pad_cols=pad)
    Gd = GuardedBatch(batch, M, N, out_dt, pad_cols=pad)
    A, B = to_dev(bi.A, dtype_in), to_dev(bi.B, dtype_in)
    st = binding.mma_gemm_batched_ex(codes[0], codes[1], M, N, K, A.data_ptr(), K,
                                     B.data_ptr(), K, Gc.ptr, Gc.ld, Gd.ptr, Gd.ld,
                                     batch, 2, 1, 7,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.STATUS.get(st, st)
    Gd.verify(f"batched {dtype_in} {M}x{N}x{K} padded ldd guard")
    Gc.verify(f"batched {dtype_in} {M}x{N}x{K} padded ldc (input) guard")
    check(dtype_in, Gd.result(), want(bi), absab(bi) if dtype_in != "i8" else None,
          f"batched {dtype_in} {M}x{N}x{K} padded ld")


# IEEE special values through each batched kernel: a NaN in the broadcast A
# tile of the first group, an infinity in one entry's B met by zeros,
# positives and negatives of its A column (NaN, +inf, -inf outputs), and a
# NaN and an infinity in another entry's C.  NaN positions and infinity
# signs must match the oracle; finite outputs keep the tolerance.
_SPECIAL_BITS = {"f16": (0x7E00, 0x7C00, 0x3C00), "bf16": (0x7FC0, 0x7F80, 0x3F80)}


@pytest.mark.parametrize("dtype_in,M,N,K,batch", [
    ("bf16", 16, 16, 16, 64),      # streaming 16^3 kernel
    ("bf16", 32, 32, 32, 64),      # warp-level kernel
    ("f16", 64, 64, 64, 48),       # CTA-cooperative kernel
    ("bf16", 128, 128, 128, 16),   # tensor-memory kernel
    ("f64", 32, 32, 32, 32),       # FP64 batched
])
def test_batched_special_values(dtype_in, M, N, K, batch):
    bi = synth.batched_inputs(f"bsv_{dtype_in}_{M}", dtype_in, batch, M=M, N=N, K=K,
                              group=4, abid=1)
    A, B, C = bi.A.copy(), bi.B.copy(), bi.C.copy()
    if dtype_in == "f64":
        nan, inf, one = np.nan, np.inf, 1.0
        neg = lambda v: -v
    else:
        nan, inf, one = _SPECIAL_BITS[dtype_in]
        neg = lambda v: v | 0x8000
    A[1, 3, 5] = nan                 # group 0 reads A tile 1: row 3 NaN in entries 0..3
    B[6, 2, 0] = inf                 # entry 6, column 2, k = 0
    A[5, 0:M:3, 0] = 0               # entry 6 reads A tile 5: NaN rows
    A[5, 1:M:3, 0] = one             # +inf rows
    A[5, 2:M:3, 0] = neg(one)        # -inf rows
    C[9, 4, 7] = np.nan
    C[9, 5, 8] = np.inf
    bs = synth.BatchedInputs(dtype_in, batch, M, N, K, 4, 1, A, B, C, 0)
    w = want(bs)
    got = run(bs)
    assert np.array_equal(np.isnan(got), np.isnan(w)), "NaN positions differ"
    inf_w = np.isinf(w)
    assert np.array_equal(np.isinf(got), inf_w), "infinity positions differ"
    assert np.array_equal(np.sign(got[inf_w]), np.sign(w[inf_w])), "infinity signs differ"
    assert np.isnan(w[0:4, 3]).all() and np.isnan(w[6, 0:M:3, 2]).all()
    assert (w[6, 1:M:3, 2] == np.inf).all() and (w[6, 2:M:3, 2] == -np.inf).all()
    ab = absab(bs)
    fin = np.isfinite(w) & np.isfinite(ab)
    rel, ab0 = TOL[dtype_in]
    err = np.abs(got[fin].astype(np.float64) - w[fin].astype(np.float64))
    bound = rel * ab[fin] + ab0
    if dtype_in == "f64":
        bound = bound + np.abs(w[fin]) * 2.0 ** -52
    assert (err <= bound).all(), f"finite outputs off by up to {err.max()}"
