// Batched FP16/BF16 products of small and mid-size blocks, streamed from HBM:
//
//     D_b = A_{srcA(b)} * B_{srcB(b)} + C_b,
//     srcA(b) = (b / G) * G + abid                  (cbsz/abid broadcast)
//     srcB(b) = (b / 4) * 4 + P[blgp][b % 4]        (B lane-group pattern)
//
// Semantics: page "Common MFMA parameters", sections "Shared parameters"
// (cbsz, abid) and "Dense MFMA parameters" (blgp, read at matrix level: the
// four entries of a group of four play the four 16-lane quarters of the B
// operand), with batch entries in the role of the independent blocks of
// "CDNA2 dense MFMA builtins", section "Accumulator layout".  Tiles are
// contiguous: A M x K and C, D M x N row-major, B column-major (N rows of
// K), tile t of each at t times its size.
//
// Blocks of up to a few hundred rows move about one byte per flop or less,
// so the path is bound by HBM bandwidth, and the tensor-memory GEMM's
// per-tile pipeline latency (one mostly padded 128-row tile per entry)
// would dominate.  This kernel is shaped around memory traffic instead,
// like the 16 x 16 x 16 kernel:
//   * a warp computes one WM x WN tile of one entry (32 x 32, or 16 x 16
//     when the block is not a multiple of 32) and walks the units of all
//     entries with a warp-stride loop;
//   * C goes straight into the FP32 accumulators, and every operand
//     fragment of a 32-deep K chunk is loaded before its MMAs, so each warp
//     keeps about 8 KB in flight (two 256-thread blocks per SM: more
//     resident warps with fewer registers each, or deeper chunks, measured
//     slower);
//   * operand fragments are read straight from global memory with 8-byte
//     accesses that cover whole 32-byte sectors: the K index is permuted
//     identically in A and B (fragment slots {2t, 2t+1, 2t+8, 2t+9} of
//     lane (g, t) hold physical k = 4t .. 4t+3), which leaves each sum over
//     k unchanged;
//   * m16n8k16 MMAs accumulate in FP32; D is stored with streaming hints,
//     as FP32 or rounded once to the 16-bit input type (16-bit accumulate).
#include "kernels.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <type_traits>

namespace mmagb {
namespace {

constexpr int kThreads = 256;

// The quarter whose B data quarter q receives under lane-group pattern p
// (0 none moved; 1 lanes 0-31 copied to 32-63; 2 lanes 32-63 copied to
// 0-31; 3 rotated down by 16 lanes; 4..7 quarter p - 4 copied to all).
__device__ __forceinline__ int blgp_quarter(int p, int q) {
  return p == 0 ? q : p == 1 ? (q & 1) : p == 2 ? (2 | (q & 1))
                                      : p == 3 ? ((q + 1) & 3) : p - 4;
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  if constexpr (BF16)
    mma_bf16_16816(d, a, b);
  else
    mma_f16_16816(d, a, b);
}

template <bool BF16>
__device__ __forceinline__ float2 half2_to_f32x2(uint32_t v) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  } else {
    const __half2 h = *reinterpret_cast<const __half2*>(&v);
    return __half22float2(h);
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t f32x2_to_half2(float lo, float hi) {
  if constexpr (BF16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}

// MT m16 tiles x NT n8 tiles per warp; OUT16: C and D of the 16-bit input
// type (else FP32).
template <int MT, int NT, bool BF16, bool OUT16>
__global__ void __launch_bounds__(kThreads, 2)
    batched_mma_kernel(const uint16_t* __restrict__ A,
                       const uint16_t* __restrict__ B,
                       const void* __restrict__ Cv, void* __restrict__ Dv,
                       int M, int N, int K, int64_t batch, int group, int abid,
                       int blgp) {
  constexpr int WM = 16 * MT, WN = 8 * NT;
  constexpr int KS = 2;  // k16 steps per chunk: all their loads in flight
  using CT = typename std::conditional<OUT16, uint16_t, float>::type;
  const CT* C = static_cast<const CT*>(Cv);
  CT* D = static_cast<CT*>(Dv);
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int tiles_n = N / WN;
  const int64_t per_entry = int64_t(M / WM) * tiles_n;
  const int64_t units = batch * per_entry;
  const int64_t warp0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;

  for (int64_t u = warp0; u < units; u += nwarps) {
    const int64_t b = u / per_entry;
    const int r = int(u - b * per_entry);
    const int tm = r / tiles_n, tn = r - tm * tiles_n;
    const int64_t za = (b / group) * group + abid;
    const int64_t zb = (b & ~int64_t(3)) + blgp_quarter(blgp, int(b & 3));
    const uint16_t* At = A + (za * M + tm * WM) * int64_t(K);
    const uint16_t* Bt = B + (zb * N + tn * WN) * int64_t(K);
    const int64_t c0 = (b * M + tm * WM) * int64_t(N) + tn * WN;

    // accumulators start from C: rows g and g + 8 of each m16 tile,
    // columns 2t, 2t + 1 of each n8 tile
    float acc[MT][NT][4];
#pragma unroll
    for (int mi = 0; mi < MT; ++mi)
#pragma unroll
      for (int ni = 0; ni < NT; ++ni) {
        const int64_t o0 = c0 + int64_t(mi * 16 + g) * N + ni * 8 + 2 * t;
        const int64_t o1 = o0 + int64_t(8) * N;
        if (C != nullptr) {
          if constexpr (OUT16) {
            const float2 v0 = half2_to_f32x2<BF16>(
                __ldcs(reinterpret_cast<const unsigned int*>(C + o0)));
            const float2 v1 = half2_to_f32x2<BF16>(
                __ldcs(reinterpret_cast<const unsigned int*>(C + o1)));
            acc[mi][ni][0] = v0.x; acc[mi][ni][1] = v0.y;
            acc[mi][ni][2] = v1.x; acc[mi][ni][3] = v1.y;
          } else {
            const float2 v0 = __ldcs(reinterpret_cast<const float2*>(C + o0));
            const float2 v1 = __ldcs(reinterpret_cast<const float2*>(C + o1));
            acc[mi][ni][0] = v0.x; acc[mi][ni][1] = v0.y;
            acc[mi][ni][2] = v1.x; acc[mi][ni][3] = v1.y;
          }
        } else {
          acc[mi][ni][0] = acc[mi][ni][1] = acc[mi][ni][2] = acc[mi][ni][3] = 0.f;
        }
      }

    for (int k0 = 0; k0 < K; k0 += 16 * KS) {
      // every fragment of the chunk first (physical k = 4t .. 4t+3 of each
      // k16 step, one 8-byte load per row)
      uint2 af[KS][MT][2];
      uint2 bf[KS][NT];
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int kk = k0 + s * 16 + 4 * t;
        if (kk < K) {
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            af[s][mi][0] = __ldg(reinterpret_cast<const uint2*>(
                At + int64_t(mi * 16 + g) * K + kk));
            af[s][mi][1] = __ldg(reinterpret_cast<const uint2*>(
                At + int64_t(mi * 16 + g + 8) * K + kk));
          }
#pragma unroll
          for (int ni = 0; ni < NT; ++ni)
            bf[s][ni] = __ldg(reinterpret_cast<const uint2*>(
                Bt + int64_t(ni * 8 + g) * K + kk));
        }
      }
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        if (k0 + s * 16 < K) {
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            const uint32_t a[4] = {af[s][mi][0].x, af[s][mi][1].x,
                                   af[s][mi][0].y, af[s][mi][1].y};
#pragma unroll
            for (int ni = 0; ni < NT; ++ni) {
              const uint32_t bb[2] = {bf[s][ni].x, bf[s][ni].y};
              mma16816<BF16>(acc[mi][ni], a, bb);
            }
          }
        }
      }
    }

#pragma unroll
    for (int mi = 0; mi < MT; ++mi)
#pragma unroll
      for (int ni = 0; ni < NT; ++ni) {
        const int64_t o0 = c0 + int64_t(mi * 16 + g) * N + ni * 8 + 2 * t;
        const int64_t o1 = o0 + int64_t(8) * N;
        if constexpr (OUT16) {
          __stcs(reinterpret_cast<unsigned int*>(D + o0),
                 f32x2_to_half2<BF16>(acc[mi][ni][0], acc[mi][ni][1]));
          __stcs(reinterpret_cast<unsigned int*>(D + o1),
                 f32x2_to_half2<BF16>(acc[mi][ni][2], acc[mi][ni][3]));
        } else {
          __stcs(reinterpret_cast<float2*>(D + o0),
                 make_float2(acc[mi][ni][0], acc[mi][ni][1]));
          __stcs(reinterpret_cast<float2*>(D + o1),
                 make_float2(acc[mi][ni][2], acc[mi][ni][3]));
        }
      }
  }
}

// INT8 -> INT32 (exact; the INT32 accumulators wrap like the INT8 GEMM's):
// the same structure with m16n8k32 integer MMAs.  A lane's fragment bytes
// for one 32-deep K step are the 8 contiguous physical k = 8t .. 8t+7 of a
// row (one 8-byte load): the low word takes the fragment's k = 4t .. 4t+3,
// the high word k = 16+4t .. 16+4t+3, identically in A and B.  K beyond the
// block (K a multiple of 8) reads as zero.
template <int MT, int NT, int KS>
__global__ void __launch_bounds__(kThreads, 2)
    batched_i8_kernel(const int8_t* __restrict__ A, const int8_t* __restrict__ B,
                      const int32_t* __restrict__ C, int32_t* __restrict__ D,
                      int M, int N, int K, int64_t batch, int group, int abid,
                      int blgp) {
  // KS: k32 steps per chunk, all their loads in flight
  constexpr int WM = 16 * MT, WN = 8 * NT;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int tiles_n = N / WN;
  const int64_t per_entry = int64_t(M / WM) * tiles_n;
  const int64_t units = batch * per_entry;
  const int64_t warp0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;

  for (int64_t u = warp0; u < units; u += nwarps) {
    const int64_t b = u / per_entry;
    const int r = int(u - b * per_entry);
    const int tm = r / tiles_n, tn = r - tm * tiles_n;
    const int64_t za = (b / group) * group + abid;
    const int64_t zb = (b & ~int64_t(3)) + blgp_quarter(blgp, int(b & 3));
    const int8_t* At = A + (za * M + tm * WM) * int64_t(K);
    const int8_t* Bt = B + (zb * N + tn * WN) * int64_t(K);
    const int64_t c0 = (b * M + tm * WM) * int64_t(N) + tn * WN;

    int acc[MT][NT][4];
#pragma unroll
    for (int mi = 0; mi < MT; ++mi)
#pragma unroll
      for (int ni = 0; ni < NT; ++ni) {
        const int64_t o0 = c0 + int64_t(mi * 16 + g) * N + ni * 8 + 2 * t;
        const int64_t o1 = o0 + int64_t(8) * N;
        if (C != nullptr) {
          const int2 v0 = __ldcs(reinterpret_cast<const int2*>(C + o0));
          const int2 v1 = __ldcs(reinterpret_cast<const int2*>(C + o1));
          acc[mi][ni][0] = v0.x; acc[mi][ni][1] = v0.y;
          acc[mi][ni][2] = v1.x; acc[mi][ni][3] = v1.y;
        } else {
          acc[mi][ni][0] = acc[mi][ni][1] = acc[mi][ni][2] = acc[mi][ni][3] = 0;
        }
      }

    for (int k0 = 0; k0 < K; k0 += 32 * KS) {
      uint2 af[KS][MT][2];
      uint2 bf[KS][NT];
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int kk = k0 + s * 32 + 8 * t;
        const bool in = kk < K;
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
          af[s][mi][0] = in ? __ldg(reinterpret_cast<const uint2*>(
                                  At + int64_t(mi * 16 + g) * K + kk))
                            : make_uint2(0u, 0u);
          af[s][mi][1] = in ? __ldg(reinterpret_cast<const uint2*>(
                                  At + int64_t(mi * 16 + g + 8) * K + kk))
                            : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int ni = 0; ni < NT; ++ni)
          bf[s][ni] = in ? __ldg(reinterpret_cast<const uint2*>(
                               Bt + int64_t(ni * 8 + g) * K + kk))
                         : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        if (k0 + s * 32 < K) {
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            const uint32_t a[4] = {af[s][mi][0].x, af[s][mi][1].x,
                                   af[s][mi][0].y, af[s][mi][1].y};
#pragma unroll
            for (int ni = 0; ni < NT; ++ni) {
              const uint32_t bb[2] = {bf[s][ni].x, bf[s][ni].y};
              mma_s8_16832(acc[mi][ni], a, bb);
            }
          }
        }
      }
    }

#pragma unroll
    for (int mi = 0; mi < MT; ++mi)
#pragma unroll
      for (int ni = 0; ni < NT; ++ni) {
        const int64_t o0 = c0 + int64_t(mi * 16 + g) * N + ni * 8 + 2 * t;
        const int64_t o1 = o0 + int64_t(8) * N;
        __stcs(reinterpret_cast<int2*>(D + o0), make_int2(acc[mi][ni][0], acc[mi][ni][1]));
        __stcs(reinterpret_cast<int2*>(D + o1), make_int2(acc[mi][ni][2], acc[mi][ni][3]));
      }
  }
}

template <int MT, int NT>
mma_status_t run_i8(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                    const void* A, const void* B, const void* C, void* D,
                    int64_t batch, int group, int abid, int blgp) {
  const int64_t units = batch * (M / (16 * MT)) * (N / (8 * NT));
  int64_t blocks = (units + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = int64_t(ctx.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  ctx.mark_start();
  // one 32-deep step per chunk when K fits it (no predicated-off second
  // step): 65536 x 32^3 105.6 -> 98.2 us
  auto kern = K <= 32 ? batched_i8_kernel<MT, NT, 1> : batched_i8_kernel<MT, NT, 2>;
  kern<<<int(blocks), kThreads, 0, ctx.stream>>>(
      static_cast<const int8_t*>(A), static_cast<const int8_t*>(B),
      static_cast<const int32_t*>(C), static_cast<int32_t*>(D), int(M),
      int(N), int(K), batch, group, abid, blgp);
  ctx.mark_stop();
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

template <int MT, int NT, bool BF16, bool OUT16>
mma_status_t run(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                 const void* A, const void* B, const void* C, void* D,
                 int64_t batch, int group, int abid, int blgp) {
  const int64_t units = batch * (M / (16 * MT)) * (N / (8 * NT));
  const int64_t warps_per_block = kThreads / 32;
  int64_t blocks = (units + warps_per_block - 1) / warps_per_block;
  const int64_t cap = int64_t(ctx.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  ctx.mark_start();
  batched_mma_kernel<MT, NT, BF16, OUT16><<<int(blocks), kThreads, 0, ctx.stream>>>(
      static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), C, D,
      int(M), int(N), int(K), batch, group, abid, blgp);
  ctx.mark_stop();
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

template <bool BF16, bool OUT16>
mma_status_t pick(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                  const void* A, const void* B, const void* C, void* D,
                  int64_t batch, int group, int abid, int blgp) {
  if (M % 32 == 0 && N % 32 == 0)
    return run<2, 4, BF16, OUT16>(ctx, M, N, K, A, B, C, D, batch, group, abid,
                                  blgp);
  return run<1, 2, BF16, OUT16>(ctx, M, N, K, A, B, C, D, batch, group, abid,
                                blgp);
}

}  // namespace

// Shapes this kernel takes: dense tiles (leading dimensions equal to the
// row lengths), M, N and K multiples of 16, and blocks of at most
// kMaxBlockMacs multiply-adds.  Measured in % of the copy bandwidth, this
// kernel against the tensor-memory GEMM: 32^3 93 against 7, 64^3 73 against
// 29, 96 x 96 x 64 65 against 58, 128^3 54 against 88 (larger blocks carry
// enough work per tile for the tensor-memory GEMM; here each warp re-reads
// the A and B rows its neighbours share).  INT8 blocks go through BF16
// copies on the tensor-memory side, so the integer kernel keeps them up to
// kMaxBlockMacsI8: 16^3 59 against 1, 32^3 86 against 6, 64^3 73 against
// 20, 128^3 56 against 49.  MMA_GB300_BATCHED (mma or tc) overrides the
// size rule, for tuning.
constexpr int64_t kMaxBlockMacs = int64_t(96) * 96 * 64;
constexpr int64_t kMaxBlockMacsI8 = int64_t(128) * 128 * 128;

bool batched_mma_fits(int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int64_t ldc, int64_t ldd, bool has_c,
                      bool i8) {
  static const int forced = [] {
    const char* e = getenv("MMA_GB300_BATCHED");
    if (!e) return 0;
    if (e[0] == 'm') return 1;
    if (e[0] == 't') return -1;
    return 0;
  }();
  const bool shape_ok = M % 16 == 0 && N % 16 == 0 && K % 16 == 0 && M > 0 &&
                        N > 0 && K > 0 && lda == K && ldb == K && ldd == N &&
                        (!has_c || ldc == N) && M < (int64_t(1) << 24) &&
                        N < (int64_t(1) << 24) && K < (int64_t(1) << 24);
  if (!shape_ok || forced < 0) return false;
  return forced > 0 || M * N * K <= (i8 ? kMaxBlockMacsI8 : kMaxBlockMacs);
}

mma_status_t launch_batched_i8_mma(const Ctx& ctx, int64_t M, int64_t N,
                                   int64_t K, const void* A, const void* B,
                                   const void* C, void* D, int64_t batch,
                                   int group, int abid, int blgp) {
  if (M % 32 == 0 && N % 32 == 0)
    return run_i8<2, 4>(ctx, M, N, K, A, B, C, D, batch, group, abid, blgp);
  return run_i8<1, 2>(ctx, M, N, K, A, B, C, D, batch, group, abid, blgp);
}

mma_status_t launch_batched_mma(const Ctx& ctx, bool bf16, bool out16,
                                int64_t M, int64_t N, int64_t K, const void* A,
                                const void* B, const void* C, void* D,
                                int64_t batch, int group, int abid, int blgp) {
  if (bf16)
    return out16 ? pick<true, true>(ctx, M, N, K, A, B, C, D, batch, group,
                                    abid, blgp)
                 : pick<true, false>(ctx, M, N, K, A, B, C, D, batch, group,
                                     abid, blgp);
  return out16 ? pick<false, true>(ctx, M, N, K, A, B, C, D, batch, group,
                                   abid, blgp)
               : pick<false, false>(ctx, M, N, K, A, B, C, D, batch, group,
                                    abid, blgp);
}

}  // namespace mmagb
