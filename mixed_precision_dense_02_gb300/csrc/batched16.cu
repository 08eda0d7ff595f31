// Batched 16x16x16 FP16/BF16 -> FP32 multiply-accumulate with A-block
// broadcast:  D_b = A_{src(b)} * B_{bsrc(b)} + C_b,  src(b) = (b / G) * G +
// abid, bsrc(b) = (b / 4) * 4 + (quarter read under lane-group pattern blgp;
// page "Common MFMA parameters", section "Dense MFMA parameters", read at
// matrix level with the four entries of a group as the four 16-lane
// quarters of the B operand; blgp = 0 gives bsrc(b) = b).
//
// Semantics: page "Common MFMA parameters", section "Shared parameters"
// (cbsz broadcasts the A values of block abid of each group of G = 2^cbsz
// neighbouring blocks to the others), with batch entries in the role of the
// independent blocks of "CDNA2 dense MFMA builtins", section "Accumulator
// layout".  Storage is contiguous per tile: A/B tiles of 256 elements (B
// column-major, i.e. its transpose row-major), C/D tiles of 256 floats.
//
// At 3 flop per byte this path is bound by HBM bandwidth, not by the tensor
// cores, so the kernel is shaped around memory traffic:
//   * one warp handles a unit of 4 consecutive entries; every load and
//     store of the unit is issued before any is consumed (about 6 KB in
//     flight per warp), with streaming (evict-first) cache hints;
//   * the A tile of a group is read once per unit (once per group for
//     G >= 4, the algorithmic minimum);
//   * operands are loaded straight into mma.sync fragments with 8-byte
//     accesses that cover whole 32-byte sectors.  To make that possible the
//     K index is permuted identically in A and B: fragment slots
//     {2t, 2t+1, 2t+8, 2t+9} of lane (g, t) hold physical k = 4t .. 4t+3,
//     which leaves the sum over k unchanged.
//   * two m16n8k16 MMAs per entry with C as the initial accumulator.
#include "kernels.h"
#include "ptx.cuh"

namespace mmagb {
namespace {

constexpr int kThreads = 256;

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  if constexpr (BF16)
    mma_bf16_16816(d, a, b);
  else
    mma_f16_16816(d, a, b);
}

template <int G, bool BF16>
__global__ void __launch_bounds__(kThreads)
    batched16_kernel(const uint16_t* __restrict__ A,
                     const uint16_t* __restrict__ B,
                     const float* __restrict__ C, float* __restrict__ D,
                     int64_t batch, int abid, int blgp) {
  constexpr int NA = G >= 4 ? 1 : 4 / G;  // distinct A tiles per unit
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t4 = (lane & 3) * 4;   // physical k offset of this lane
  const int t2 = (lane & 3) * 2;   // output column offset of this lane
  const int64_t warp0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  const int64_t units = (batch + 3) >> 2;

  for (int64_t u = warp0; u < units; u += nwarps) {
    const int64_t b0 = u * 4;
    uint32_t a[NA][4];
#pragma unroll
    for (int i = 0; i < NA; ++i) {
      const int64_t first = b0 + int64_t(i) * (G >= 4 ? 0 : G);
      a[i][0] = a[i][1] = a[i][2] = a[i][3] = 0u;
      if (first < batch) {
        const uint16_t* at = A + ((first / G) * G + abid) * 256;
        const uint2 lo = __ldcs(reinterpret_cast<const uint2*>(at + g * 16 + t4));
        const uint2 hi = __ldcs(reinterpret_cast<const uint2*>(at + (g + 8) * 16 + t4));
        a[i][0] = lo.x;
        a[i][1] = hi.x;
        a[i][2] = lo.y;
        a[i][3] = hi.y;
      }
    }
    uint2 bf[4][2];
    float2 cf[4][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t b = b0 + e;
      if (b < batch) {
        // quarter e of the group of four whose first entry is b0: the
        // quarter it reads under pattern blgp (a unit is one such group)
        const int qs = blgp == 0   ? e
                       : blgp == 1 ? (e & 1)
                       : blgp == 2 ? (2 | (e & 1))
                       : blgp == 3 ? ((e + 1) & 3)
                                   : blgp - 4;
        const uint16_t* bt = B + (b0 + qs) * 256;
        bf[e][0] = __ldcs(reinterpret_cast<const uint2*>(bt + g * 16 + t4));
        bf[e][1] = __ldcs(reinterpret_cast<const uint2*>(bt + (g + 8) * 16 + t4));
        const float* ct = C ? C + b * 256 : nullptr;
        if (ct) {
          cf[e][0] = __ldcs(reinterpret_cast<const float2*>(ct + g * 16 + t2));
          cf[e][1] = __ldcs(reinterpret_cast<const float2*>(ct + (g + 8) * 16 + t2));
          cf[e][2] = __ldcs(reinterpret_cast<const float2*>(ct + g * 16 + 8 + t2));
          cf[e][3] = __ldcs(reinterpret_cast<const float2*>(ct + (g + 8) * 16 + 8 + t2));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) cf[e][j] = make_float2(0.f, 0.f);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t b = b0 + e;
      if (b < batch) {
        const int ai = G >= 4 ? 0 : e / G;
        float d0[4] = {cf[e][0].x, cf[e][0].y, cf[e][1].x, cf[e][1].y};
        float d1[4] = {cf[e][2].x, cf[e][2].y, cf[e][3].x, cf[e][3].y};
        const uint32_t bn0[2] = {bf[e][0].x, bf[e][0].y};
        const uint32_t bn1[2] = {bf[e][1].x, bf[e][1].y};
        mma16816<BF16>(d0, a[ai], bn0);
        mma16816<BF16>(d1, a[ai], bn1);
        float* dt = D + b * 256;
        __stcs(reinterpret_cast<float2*>(dt + g * 16 + t2), make_float2(d0[0], d0[1]));
        __stcs(reinterpret_cast<float2*>(dt + (g + 8) * 16 + t2), make_float2(d0[2], d0[3]));
        __stcs(reinterpret_cast<float2*>(dt + g * 16 + 8 + t2), make_float2(d1[0], d1[1]));
        __stcs(reinterpret_cast<float2*>(dt + (g + 8) * 16 + 8 + t2), make_float2(d1[2], d1[3]));
      }
    }
  }
}

template <int G, bool BF16>
mma_status_t run(const Ctx& ctx, int64_t batch, int abid, int blgp,
                 const void* A, const void* B, const float* C, float* D) {
  const int64_t units = (batch + 3) / 4;
  const int64_t warps_per_block = kThreads / 32;
  int64_t blocks = (units + warps_per_block - 1) / warps_per_block;
  const int64_t cap = int64_t(ctx.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  ctx.mark_start();
  batched16_kernel<G, BF16><<<int(blocks), kThreads, 0, ctx.stream>>>(
      static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), C, D,
      batch, abid, blgp);
  ctx.mark_stop();
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

template <bool BF16>
mma_status_t dispatch_group(const Ctx& ctx, int64_t batch, int group, int abid,
                            int blgp, const void* A, const void* B,
                            const float* C, float* D) {
  switch (group) {
    case 1: return run<1, BF16>(ctx, batch, abid, blgp, A, B, C, D);
    case 2: return run<2, BF16>(ctx, batch, abid, blgp, A, B, C, D);
    case 4: return run<4, BF16>(ctx, batch, abid, blgp, A, B, C, D);
    case 8: return run<8, BF16>(ctx, batch, abid, blgp, A, B, C, D);
    case 16: return run<16, BF16>(ctx, batch, abid, blgp, A, B, C, D);
    default: return MMA_ERR_INVALID_ARG;
  }
}

}  // namespace

mma_status_t launch_batched16(const Ctx& ctx, bool bf16, int64_t batch,
                              int group, int abid, int blgp, const void* A,
                              const void* B, const float* C, float* D) {
  return bf16 ? dispatch_group<true>(ctx, batch, group, abid, blgp, A, B, C, D)
              : dispatch_group<false>(ctx, batch, group, abid, blgp, A, B, C,
                                      D);
}

}  // namespace mmagb
