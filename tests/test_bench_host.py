"""Host-side logic of bench.py on CPU: the multi-rank path over gloo
(world size 2), the reference arm's JSON line, and the clock summary."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    d = bench.Dist(want_cuda=False)
    d.barrier()
    m = d.max(1.0 + rank)           # each rank's own "time"
    v = bench.whole_job(10.0, 4, d.world, m)
    d.close()
    q.put((rank, m, v))


def test_two_rank_max_and_whole_job_over_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the max time (2.0) and the whole-job value 10*4*2/2
    assert out == [(0, 2.0, 40.0), (1, 2.0, 40.0)]


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"),
                          "--impl", "reference", "--steps", "1", "--warmup", "0",
                          "--workload", "gemm_f16_256"],
                         capture_output=True, text=True, timeout=300, check=True)
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert rec["unit"] == "TFLOP/s" and rec["warmup"] >= 3
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_non_zero_rank_is_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    # rank 1 alone: its process group cannot form, so run the rank logic
    # directly instead of the whole program
    args = type("A", (), dict(steps=1, warmup=0, workload="gemm_f16_256", gpus=2))
    d = type("D", (), dict(rank=1, world=2))
    assert bench.run_reference(args, d) == 0
    del env


def test_clock_summary_window_and_reasons():
    c = bench.ClockSampler(0)
    row = lambda mhz, pc: ["0", str(mhz), "2070", "900", "0x0", "Not Active",
                           "Not Active", "Not Active", pc]
    c.samples = [(1.0, row(800, "Not Active")), (10.0, row(1800, "Active")),
                 (11.0, row(1900, "Not Active")), (30.0, row(700, "Not Active"))]
    s = c.summary(9.9, 11.1)
    assert s["sm_mhz"] == 1850 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2


def test_workload_meta_algorithmic_figures():
    w = bench.workload_meta("batched_bf16_16x16x16_b262144_g4_abid1")
    assert w["algorithmic_bytes"] == 704643072
    assert w["ops"] == 262144 * 2 * 16 ** 3
    w = bench.workload_meta("gemm_i8_4096")
    assert w["ops"] == 2 * 4096 ** 3 and w["unit"] == "TOP/s"
    assert w["algorithmic_bytes"] == 2 * 4096 ** 2 + 2 * 4 * 4096 ** 2


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    """The traffic figures are keyed by the code of a kernel source: a
    comment or whitespace edit keeps the key, a code edit changes it."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = tmp_path / "k.cu"
    f.write_text("// kernel\n__global__ void k(int* p) { p[0] = 1; }\n")
    h0 = bench.source_sha("k.cu")
    f.write_text("/* another\n   comment */ __global__  void k(int* p)\n"
                 "{  // store\n  p[0] = 1;\n}\n")
    assert bench.source_sha("k.cu") == h0
    f.write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.source_sha("k.cu") != h0
    assert bench.source_sha("missing.cu") is None


def test_traffic_keys_name_existing_workloads():
    from mixed_precision_dense_02_gb300 import synth
    assert set(bench.NCU_TRAFFIC) <= set(synth.WORKLOADS)
    for rec in bench.NCU_TRAFFIC.values():
        assert len(rec["sha"]) == 16
        assert rec["bytes"] > 0


def _cxx_constant(rel, name):
    """Value of `constexpr ... name = <integer expression>;` in a library
    source: literals, int64_t(...) casts, *, << only."""
    import ast
    import re
    with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
        m = re.search(r"constexpr\s+\w+\s+" + name + r"\s*=\s*([^;]+);", f.read())
    assert m, f"{name} not found in {rel}"
    expr = re.sub(r"int64_t\(([^()]*)\)", r"(\1)", m.group(1))

    def ev(node):
        if isinstance(node, ast.Expression):
            return ev(node.body)
        if isinstance(node, ast.Constant) and isinstance(node.value, (int, float)):
            return node.value
        if isinstance(node, ast.BinOp) and isinstance(node.op, (ast.Mult, ast.LShift)):
            a, b = ev(node.left), ev(node.right)
            return a * b if isinstance(node.op, ast.Mult) else a << b
        raise AssertionError(f"unexpected expression {expr!r}")

    return ev(ast.parse(expr.strip(), mode="eval"))


def test_bench_kernel_attribution_follows_the_library_routing():
    """bench.py attributes each workload's traffic figure to the source
    file of the kernel the library picks; its thresholds must be the
    library's own."""
    csrc = "mixed_precision_dense_02_gb300/csrc/"
    tile_max = _cxx_constant(csrc + "batched_tile.cu", "kTileMaxMacs")
    mma_max = _cxx_constant(csrc + "batched_mma.cu", "kMaxBlockMacs")
    mma_max_i8 = _cxx_constant(csrc + "batched_mma.cu", "kMaxBlockMacsI8")
    i8_min = _cxx_constant(csrc + "api.cu", "kI8TensorCoreMinWork")

    def src(dt, M, N, K, kind="batched"):
        return bench.kernel_source({"kind": kind, "dtype_in": dt, "M": M,
                                    "N": N, "K": K}).rsplit("/", 1)[-1]

    assert tile_max == 1 << 20 and src("bf16", 128, 64, 128) == "batched_tile.cu"
    assert src("bf16", 128, 128, 128) == "gemm_tc.cu"            # 2^21 > tile_max
    assert mma_max == 96 * 96 * 64 and src("bf16", 96, 96, 64) == "batched_mma.cu"
    assert src("bf16", 96, 96, 80) == "gemm_tc.cu"               # above mma_max
    assert mma_max_i8 == 128 ** 3 and src("i8", 128, 128, 128) == "batched_mma.cu"
    assert src("i8", 144, 128, 128) == "gemm_tc.cu"
    assert src("bf16", 16, 16, 16) == "batched16.cu"
    assert i8_min == 2.0 ** 24
    small = {"kind": "gemm", "dtype_in": "i8", "M": 256, "N": 256, "K": 255}
    big = dict(small, K=256)
    assert bench.kernel_source(small).endswith("gemm_i8.cu")
    assert bench.kernel_source(big).endswith("gemm_tc.cu")
    # stream-K: the rule of gemm_sk_fits (few tiles, deep K)
    with open(os.path.join(ROOT, csrc + "gemm_sk.cu"), encoding="utf-8") as f:
        src = f.read()
    assert "2 * tiles < num_sms && nk >= 8 && tiles * nk >= 2 * int64_t(num_sms)" in src
    assert "(4 * tiles <= num_sms || nk >= 128)" in src
    deep = {"kind": "gemm", "dtype_in": "bf16", "M": 1024, "N": 1024, "K": 32768}
    assert bench.kernel_source(deep).endswith("gemm_sk.cu")
    skinny = dict(deep, M=16384, N=128, K=4096)           # 128 tiles >= 76
    assert bench.kernel_source(skinny).endswith("gemm_tc.cu")
    assert bench.kernel_source(dict(deep, acc16=True)).endswith("gemm_tc.cu")


def test_saturating_early_c_rule_in_the_library():
    """The saturating 8-bit path adds C during the chunk phase only on
    224-wide CTA-pair tiles with three or more 1024-deep chunks and
    K * max|a| * max|b| < 2^30; the GPU tests aim their shapes with a mirror
    of this rule, so it is pinned here against the library source."""
    path = os.path.join(ROOT, "mixed_precision_dense_02_gb300", "csrc", "gemm_tc.cu")
    with open(path, encoding="utf-8") as f:
        src = f.read()
    assert "const double amax = a_signed ? 128.0 : 255.0;" in src
    assert "const double bmax = b_signed ? 128.0 : 255.0;" in src
    assert "if (cl == 2 && bn == 224 && K > 2 * kI8ChunkK &&" in src
    assert "double(K) * amax * bmax < 1073741824.0)" in src
    assert "constexpr int kI8ChunkK = 1024;" in src
    # the mode's shared-memory sign words fit beside the 224-wide pair
    # layout (six stages, two staging blocks per warp) but not the 256-wide
    stage224 = 128 * 64 * 2 + 112 * 64 * 2
    stage256 = 128 * 64 * 2 + 128 * 64 * 2
    staging, bars, slack = 8 * 2 * 32 * 16 * 4, (2 * 6 + 5 + 2 * 8) * 8 + 16, 1024
    sign = 8 * 32 * 4 * 4
    assert 6 * stage224 + staging + bars + slack + sign <= 232448
    assert 6 * stage256 + staging + bars + slack + sign > 232448
