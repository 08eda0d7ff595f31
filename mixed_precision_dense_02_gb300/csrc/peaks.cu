// Issue-rate probes of the pipes the library computes on: the measured
// form of "peak throughput = operations per instruction / cycles per
// instruction x clock" ("CDNA2 dense MFMA builtins", section "Instruction
// throughput").  Each probe keeps one pipe of every SM busy with
// independent back-to-back instructions on register or shared-memory
// operands (no DRAM traffic), so the operations of one launch divided by
// its duration is that pipe's rate at the clock the launch ran at.
//   MMA_PEAK_TC_F16  tcgen05.mma kind::f16 (BF16 in, FP32 accumulate),
//                    M = 128, N = 256, K = 16 from shared memory into
//                    tensor memory, one issuing thread per SM
//   MMA_PEAK_DMMA    mma.sync m8n8k4 FP64 (the FP64 GEMM's instruction)
//   MMA_PEAK_IMMA    mma.sync m16n8k32 s8 -> s32 (the small-INT8 kernel's)
//   MMA_PEAK_DFMA    scalar FP64 fused multiply-add
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace mmagb {

// results the probes fold their accumulators into, so no work is dropped
__device__ unsigned long long g_peak_sink;

namespace {

constexpr int kTcThreads = 128;
constexpr int kTcN = 256;
constexpr int kTcABytes = 128 * 64 * 2;   // 128 rows x 64 K (one swizzle row)
constexpr int kTcBBytes = kTcN * 64 * 2;  // 256 rows x 64 K
// more shared memory than two CTAs could share, so that the grid of one CTA
// per SM really lands one on every SM (48 KB of it are used)
constexpr int kTcSmem = 120 * 1024;
static_assert(kTcABytes + kTcBBytes + 64 + 1024 <= kTcSmem, "probe tiles fit");

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_probe_kernel(long long iters, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + kTcABytes + kTcBBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  // operands: small BF16 values of both signs (the swizzle only permutes
  // 16-byte chunks, so any fill is a valid operand tile)
  uint32_t* w = reinterpret_cast<uint32_t*>(smem);
  for (int i = threadIdx.x; i < (kTcABytes + kTcBBytes) / 4; i += kTcThreads) {
    const uint32_t lo = 0x3F80u | ((i * 7u) & 0x7Fu) | ((i & 1u) << 15);
    const uint32_t hi = 0x3F00u | ((i * 13u) & 0x7Fu) | ((i & 2u) << 14);
    w[i] = lo | (hi << 16);
  }
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  fence_proxy_async_smem();
  if (threadIdx.x < 32) {
    tmem_alloc(tmem_slot, kTcN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x < 32 && elect_one()) {
    constexpr uint32_t idesc = idesc_f16_f32(true, 128, kTcN);
    const uint32_t sa = smem_u32(smem);
    const uint64_t da = sw128_kmajor_desc(sa);
    const uint64_t db = sw128_kmajor_desc(sa + kTcABytes);
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_f16(tmem, da + uint64_t(2 * k), db + uint64_t(2 * k), idesc,
                 (i | k) ? 1u : 0u);
    }
    umma_commit(done);
    (void)mbar_wait(done, 0, reinterpret_cast<volatile int*>(abort_flag), status);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(tmem, r);
    tmem_ld_wait();
    if (r[0] == 0x7FC00001u) atomicAdd(&g_peak_sink, 1ull);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcN);
  }
}

constexpr int kWarpThreads = 256;
constexpr int kChains = 8;  // independent accumulators per thread

__global__ void __launch_bounds__(kWarpThreads)
    dmma_probe_kernel(long long iters) {
  double d[kChains][2];
  double a = 1.0 + threadIdx.x * 1e-9, b = 1.0 - threadIdx.x * 1e-9;
#pragma unroll
  for (int c = 0; c < kChains; ++c) d[c][0] = d[c][1] = c * 0.5;
  for (long long i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) mma_f64_884(d[c], a, b);
  }
  double s = 0.0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += d[c][0] + d[c][1];
  if (s == 1.2345e-300) atomicAdd(&g_peak_sink, 1ull);
}

__global__ void __launch_bounds__(kWarpThreads)
    imma_probe_kernel(long long iters) {
  int d[kChains][4] = {};
  const uint32_t x = 0x01FF02FEu ^ threadIdx.x;
  const uint32_t a[4] = {x, x * 3u, x * 5u, x * 7u};
  const uint32_t b[2] = {x * 11u, x * 13u};
  for (long long i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) mma_s8_16832(d[c], a, b);
  }
  int s = 0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += d[c][0] ^ d[c][1] ^ d[c][2] ^ d[c][3];
  if (s == 0x12345) atomicAdd(&g_peak_sink, 1ull);
}

__global__ void __launch_bounds__(kWarpThreads)
    dfma_probe_kernel(long long iters) {
  double d[kChains];
  const double a = 1.0 + threadIdx.x * 1e-12, b = 1e-3;
#pragma unroll
  for (int c = 0; c < kChains; ++c) d[c] = c;
  for (long long i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) d[c] = fma(d[c], a, b);
  }
  double s = 0.0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += d[c];
  if (s == 1.2345e-300) atomicAdd(&g_peak_sink, 1ull);
}

}  // namespace
}  // namespace mmagb

using namespace mmagb;

extern "C" mma_status_t mma_peak_probe(int kind, int64_t iterations,
                                       double* ops_per_launch, void* stream) {
  if (iterations < 1 || iterations > (int64_t(1) << 40) || !ops_per_launch)
    return MMA_ERR_INVALID_ARG;
  Ctx ctx{};
  if (!current_ctx(stream, &ctx)) return MMA_ERR_NO_DEVICE;
  attach_profile(ctx);
  const double it = double(iterations);
  // warp-level probes: two 256-thread blocks per SM
  const unsigned blocks = unsigned(ctx.num_sms) * 2u;
  const double warps = double(blocks) * (kWarpThreads / 32);
  switch (kind) {
    case MMA_PEAK_TC_F16: {
      // at most about a second of MMAs at the lowest clocks, well inside
      // the probe's bounded completion wait
      if (iterations > (int64_t(1) << 21)) return MMA_ERR_INVALID_ARG;
      static PerContext<bool> attr;
      bool ok = false;
      if (!attr.get(ctx, &ok, [](bool* v) {
            *v = cudaFuncSetAttribute(tc_probe_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kTcSmem) == cudaSuccess;
            if (!*v) cudaGetLastError();
            return *v;
          }))
        return MMA_ERR_LAUNCH;
      *ops_per_launch = double(ctx.num_sms) * it * 4.0 * 2.0 * 128.0 * kTcN * 16.0;
      ctx.mark_start();
      tc_probe_kernel<<<ctx.num_sms, kTcThreads, kTcSmem, ctx.stream>>>(
          iterations, ctx.status);
      ctx.mark_stop();
      break;
    }
    case MMA_PEAK_DMMA:
      *ops_per_launch = warps * it * kChains * 2.0 * 8 * 8 * 4;
      ctx.mark_start();
      dmma_probe_kernel<<<blocks, kWarpThreads, 0, ctx.stream>>>(iterations);
      ctx.mark_stop();
      break;
    case MMA_PEAK_IMMA:
      *ops_per_launch = warps * it * kChains * 2.0 * 16 * 8 * 32;
      ctx.mark_start();
      imma_probe_kernel<<<blocks, kWarpThreads, 0, ctx.stream>>>(iterations);
      ctx.mark_stop();
      break;
    case MMA_PEAK_DFMA:
      *ops_per_launch = double(blocks) * kWarpThreads * it * kChains * 2.0;
      ctx.mark_start();
      dfma_probe_kernel<<<blocks, kWarpThreads, 0, ctx.stream>>>(iterations);
      ctx.mark_stop();
      break;
    default:
      return MMA_ERR_INVALID_ARG;
  }
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}
