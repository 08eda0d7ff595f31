// Batched FP16/BF16 products of mid-size blocks (M and N multiples of 64,
// K a multiple of 64), streamed from HBM by cooperating warps:
//
//     D_b = A_{srcA(b)} * B_{srcB(b)} + C_b,
//     srcA(b) = (b / G) * G + abid                  (cbsz/abid broadcast)
//     srcB(b) = (b / 4) * 4 + P[blgp][b % 4]        (B lane-group pattern)
//
// Semantics as in batched_mma.cu: page "Common MFMA parameters", sections
// "Shared parameters" (cbsz, abid) and "Dense MFMA parameters" (blgp, read
// at matrix level), batch entries in the role of the independent blocks of
// "CDNA2 dense MFMA builtins", section "Accumulator layout"; contiguous
// tiles (A M x K and C, D M x N row-major, B column-major).
//
// The warp-level streaming kernel loads each operand row once per warp
// tile that uses it (twice or more for blocks of 64 and up), and keeps only
// one unit's loads in flight per warp.  Here a CTA of four warps computes a
// 64 x 64 tile of an entry:
//   * the CTA's units (tile, 64-deep K chunk) form one sequence; a
//     STAGES-deep ring of shared-memory stages (A 64 x 64 and B 64 x 64
//     16-bit values, rows padded to 144 bytes, and for K = 64 the tile's
//     64 x 64 C, rows padded by 8 elements) is filled by cp.async
//     STAGES - 1 chunks ahead, across tile boundaries, so every input byte
//     is read from global memory once and the next tiles' operands (and
//     addends) are in flight while the current one is computed;
//   * each warp computes a 32 x 32 quarter with m16n8k16 MMAs, fragments
//     read by ldmatrix (conflict-free with the padded rows; B stored N x K
//     gives the column-major B fragment directly);
//   * C goes into the FP32 accumulators at a tile's first chunk (from the
//     stage for K = 64, else straight from global memory), D leaves by streaming stores after its last, as FP32 or
//     rounded once to the 16-bit input type.
#include "kernels.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <type_traits>

namespace mmagb {
namespace {

constexpr int kTileThreads = 128;
constexpr int TM = 64, TN = 64, TK = 64;
constexpr int LDS = TK + 8;  // padded operand row, 16-bit elements (144 B)
constexpr int CLD = TN + 8;  // padded C row, elements (288 B FP32, 144 B 16-bit)
constexpr int STAGES = 3;
constexpr int kOperandBytes = (TM + TN) * LDS * 2;
// STAGE_C: C also passes through the ring (tiles of one K chunk, where the
// addend is most of the input and its latency would otherwise be exposed at
// every tile); otherwise C is read straight into the accumulators, which
// keeps the stages small and four CTAs resident per SM for deeper K.
template <bool OUT16, bool STAGE_C>
__host__ __device__ constexpr int stage_bytes() {
  return kOperandBytes + (STAGE_C ? TM * CLD * (OUT16 ? 2 : 4) : 0);
}
template <bool OUT16, bool STAGE_C>
__host__ __device__ constexpr int smem_bytes() {
  return STAGES * stage_bytes<OUT16, STAGE_C>();
}

__device__ __forceinline__ int blgp_quarter_t(int p, int q) {
  return p == 0 ? q : p == 1 ? (q & 1) : p == 2 ? (2 | (q & 1))
                                      : p == 3 ? ((q + 1) & 3) : p - 4;
}

// ldmatrix of four 8 x 8 16-bit matrices (ordered after the shared-memory
// writes by the caller's barrier).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(saddr)
      : "memory");
}

template <bool BF16>
__device__ __forceinline__ void mma_t(float (&d)[4], const uint32_t (&a)[4],
                                      uint32_t b0, uint32_t b1) {
  const uint32_t b[2] = {b0, b1};
  if constexpr (BF16)
    mma_bf16_16816(d, a, b);
  else
    mma_f16_16816(d, a, b);
}

template <bool BF16>
__device__ __forceinline__ float2 h2_to_f2(uint32_t v) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  } else {
    const __half2 h = *reinterpret_cast<const __half2*>(&v);
    return __half22float2(h);
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  if constexpr (BF16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}

template <bool BF16, bool OUT16, bool STAGE_C>
__global__ void __launch_bounds__(kTileThreads)
    batched_tile_kernel(const uint16_t* __restrict__ A,
                        const uint16_t* __restrict__ B,
                        const void* __restrict__ Cv, void* __restrict__ Dv,
                        int M, int N, int K, int64_t batch, int group, int abid,
                        int blgp) {
  extern __shared__ __align__(16) uint8_t smem[];
  using CT = typename std::conditional<OUT16, uint16_t, float>::type;
  constexpr int kStage = stage_bytes<OUT16, STAGE_C>();
  constexpr int kCChunksPerRow = TN * int(sizeof(CT)) / 16;
  constexpr int kCElemsPerChunk = 16 / int(sizeof(CT));
  const CT* C = static_cast<const CT*>(Cv);
  CT* D = static_cast<CT*>(Dv);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;
  const int tiles_n = N / TN;
  const int64_t per_entry = int64_t(M / TM) * tiles_n;
  const int64_t units = batch * per_entry;
  const int KT = K / TK;
  // this CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int64_t my_tiles =
      units > blockIdx.x ? (units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t items = my_tiles * KT;

  // entry and tile coordinates of item `it` (tile index within this CTA,
  // K chunk)
  auto tile_of = [&](int64_t it, int64_t& b, int& tm, int& tn) {
    const int64_t u = blockIdx.x + (it / KT) * gridDim.x;
    b = u / per_entry;
    const int r = int(u - b * per_entry);
    tm = r / tiles_n;
    tn = r - tm * tiles_n;
  };
  // one stage: the A and B chunks of item `it` and, at a tile's first
  // chunk, the tile's C, all by cp.async
  auto load_item = [&](int64_t it, int stage) {
    int64_t b;
    int tm, tn;
    tile_of(it, b, tm, tn);
    const int kci = int(it % KT);
    const int kc = kci * TK;
    const int64_t za = (b / group) * group + abid;
    const int64_t zb = (b & ~int64_t(3)) + blgp_quarter_t(blgp, int(b & 3));
    const uint16_t* At = A + (za * M + tm * TM) * int64_t(K) + kc;
    const uint16_t* Bt = B + (zb * N + tn * TN) * int64_t(K) + kc;
    uint16_t* sA = reinterpret_cast<uint16_t*>(smem + stage * kStage);
    uint16_t* sB = sA + TM * LDS;
    // 64 rows x 8 chunks of 16 bytes for each operand: 4 + 4 per thread
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * kTileThreads;
      const int row = idx >> 3, ch = (idx & 7) * 8;
      cp_async_16(smem_u32(sA + row * LDS + ch), At + int64_t(row) * K + ch);
      cp_async_16(smem_u32(sB + row * LDS + ch), Bt + int64_t(row) * K + ch);
    }
    if (STAGE_C && kci == 0 && C != nullptr) {
      CT* sC = reinterpret_cast<CT*>(smem + stage * kStage + kOperandBytes);
      const CT* Ct = C + (b * M + tm * TM) * int64_t(N) + tn * TN;
#pragma unroll
      for (int i = 0; i < TM * kCChunksPerRow / kTileThreads; ++i) {
        const int idx = tid + i * kTileThreads;
        const int row = idx / kCChunksPerRow;
        const int ch = (idx % kCChunksPerRow) * kCElemsPerChunk;
        cp_async_16(smem_u32(sC + row * CLD + ch), Ct + int64_t(row) * N + ch);
      }
    }
  };

  // prologue: the first STAGES - 1 items
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < items) load_item(s, s);
    cp_async_commit();
  }

  float acc[2][4][4];
  for (int64_t it = 0; it < items; ++it) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();  // item `it` landed; the stage refilled below is free
    {
      const int64_t nx = it + STAGES - 1;
      if (nx < items) load_item(nx, int(nx % STAGES));
      cp_async_commit();
    }
    int64_t b;
    int tm, tn;
    tile_of(it, b, tm, tn);
    const int kci = int(it % KT);
    const int stage = int(it % STAGES);
    const uint16_t* sA = reinterpret_cast<const uint16_t*>(smem + stage * kStage);
    const uint16_t* sB = sA + TM * LDS;
    if (kci == 0) {
      // accumulators start from C (rows g, g + 8; columns 2t, 2t + 1 of
      // each 16 x 8 piece): from the stage, whose padded rows keep the
      // reads conflict-free, or straight from global memory
      const CT* sC = reinterpret_cast<const CT*>(smem + stage * kStage + kOperandBytes);
      const int64_t g0 = (b * M + tm * TM + wm) * int64_t(N) + tn * TN + wn;
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const int o0 = (wm + mi * 16 + g) * CLD + wn + ni * 8 + 2 * t;
          const int o1 = o0 + 8 * CLD;
          const int64_t q0 = g0 + int64_t(mi * 16 + g) * N + ni * 8 + 2 * t;
          const int64_t q1 = q0 + int64_t(8) * N;
          if (C == nullptr) {
            acc[mi][ni][0] = acc[mi][ni][1] = acc[mi][ni][2] = acc[mi][ni][3] = 0.f;
          } else if constexpr (!STAGE_C && OUT16) {
            const float2 v0 = h2_to_f2<BF16>(__ldcs(reinterpret_cast<const unsigned int*>(C + q0)));
            const float2 v1 = h2_to_f2<BF16>(__ldcs(reinterpret_cast<const unsigned int*>(C + q1)));
            acc[mi][ni][0] = v0.x; acc[mi][ni][1] = v0.y;
            acc[mi][ni][2] = v1.x; acc[mi][ni][3] = v1.y;
          } else if constexpr (!STAGE_C) {
            const float2 v0 = __ldcs(reinterpret_cast<const float2*>(C + q0));
            const float2 v1 = __ldcs(reinterpret_cast<const float2*>(C + q1));
            acc[mi][ni][0] = v0.x; acc[mi][ni][1] = v0.y;
            acc[mi][ni][2] = v1.x; acc[mi][ni][3] = v1.y;
          } else if constexpr (OUT16) {
            const float2 v0 = h2_to_f2<BF16>(*reinterpret_cast<const uint32_t*>(sC + o0));
            const float2 v1 = h2_to_f2<BF16>(*reinterpret_cast<const uint32_t*>(sC + o1));
            acc[mi][ni][0] = v0.x; acc[mi][ni][1] = v0.y;
            acc[mi][ni][2] = v1.x; acc[mi][ni][3] = v1.y;
          } else {
            const float2 v0 = *reinterpret_cast<const float2*>(sC + o0);
            const float2 v1 = *reinterpret_cast<const float2*>(sC + o1);
            acc[mi][ni][0] = v0.x; acc[mi][ni][1] = v0.y;
            acc[mi][ni][2] = v1.x; acc[mi][ni][3] = v1.y;
          }
        }
    }
#pragma unroll
    for (int kk = 0; kk < TK; kk += 16) {
      uint32_t af[2][4], bfr[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int row = wm + mi * 16 + (lane & 15);
        const int col = kk + (lane >> 4) * 8;
        ldsm_x4(af[mi], smem_u32(sA + row * LDS + col));
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        // n8 tiles 2nj and 2nj + 1: (n 0-7, k 0-7), (n 0-7, k 8-15),
        // (n 8-15, k 0-7), (n 8-15, k 8-15)
        const int row = wn + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int col = kk + ((lane >> 3) & 1) * 8;
        ldsm_x4(bfr[nj], smem_u32(sB + row * LDS + col));
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
          mma_t<BF16>(acc[mi][ni], af[mi], bfr[ni >> 1][(ni & 1) * 2],
                      bfr[ni >> 1][(ni & 1) * 2 + 1]);
    }
    if (kci == KT - 1) {
      const int64_t c0 = (b * M + tm * TM + wm) * int64_t(N) + tn * TN + wn;
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const int64_t o0 = c0 + int64_t(mi * 16 + g) * N + ni * 8 + 2 * t;
          const int64_t o1 = o0 + int64_t(8) * N;
          if constexpr (OUT16) {
            __stcs(reinterpret_cast<unsigned int*>(D + o0),
                   f2_to_h2<BF16>(acc[mi][ni][0], acc[mi][ni][1]));
            __stcs(reinterpret_cast<unsigned int*>(D + o1),
                   f2_to_h2<BF16>(acc[mi][ni][2], acc[mi][ni][3]));
          } else {
            __stcs(reinterpret_cast<float2*>(D + o0),
                   make_float2(acc[mi][ni][0], acc[mi][ni][1]));
            __stcs(reinterpret_cast<float2*>(D + o1),
                   make_float2(acc[mi][ni][2], acc[mi][ni][3]));
          }
        }
    }
  }
  cp_async_wait<0>();  // no copy outlives the CTA
}

}  // namespace

// Shapes this kernel takes: dense tiles, M and N multiples of 64, K a
// multiple of 64, and blocks of at most kTileMaxMacs multiply-adds.  On a
// GB300 (BF16, groups of 4) this kernel reached 78 / 68 / 70 % of the copy
// bandwidth at 64^3 / 128x64x128 / 64x64x256 against 72 / 55 / 53 % for the
// warp-level streaming kernel and 28 / 57 / 46 % for the tensor-memory GEMM;
// from 128^3 up (67 % against 83 %) the tensor-memory GEMM wins, so larger
// blocks go there.  MMA_GB300_BATCHED=tile forces this kernel for every
// fitting shape, =mma or =tc never, for tuning.
constexpr int64_t kTileMaxMacs = int64_t(1) << 20;

bool batched_tile_fits(int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldc, int64_t ldd, bool has_c) {
  static const int forced = [] {
    const char* e = getenv("MMA_GB300_BATCHED");
    if (!e) return 0;
    if (e[0] == 'm' || (e[0] == 't' && e[1] == 'c')) return -1;
    if (e[0] == 't') return 1;  // "tile"
    return 0;
  }();
  const bool shape_ok = M % TM == 0 && N % TN == 0 && K % TK == 0 && M > 0 &&
                        N > 0 && K > 0 && lda == K && ldb == K && ldd == N &&
                        (!has_c || ldc == N) && M < (int64_t(1) << 24) &&
                        N < (int64_t(1) << 24) && K < (int64_t(1) << 24);
  if (!shape_ok || forced < 0) return false;
  return forced > 0 || M * N * K <= kTileMaxMacs;
}

namespace {

template <bool BF16, bool OUT16, bool STAGE_C>
mma_status_t run_tile(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                      const void* A, const void* B, const void* C, void* D,
                      int64_t batch, int group, int abid, int blgp) {
  auto kern = batched_tile_kernel<BF16, OUT16, STAGE_C>;
  // shared-memory limit and resident CTAs per SM, once per context
  static PerContext<int> occupancy;
  int per_sm = 0;
  if (!occupancy.get(ctx, &per_sm, [&](int* v) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes<OUT16, STAGE_C>()) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                v, kern, kTileThreads, smem_bytes<OUT16, STAGE_C>()) != cudaSuccess ||
            *v < 1) {
          cudaGetLastError();
          return false;
        }
        return true;
      }))
    return MMA_ERR_LAUNCH;
  const int64_t units = batch * (M / TM) * (N / TN);
  int64_t blocks = int64_t(ctx.num_sms) * per_sm;
  if (blocks > units) blocks = units;
  ctx.mark_start();
  kern<<<int(blocks), kTileThreads, smem_bytes<OUT16, STAGE_C>(), ctx.stream>>>(
      static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), C, D,
      int(M), int(N), int(K), batch, group, abid, blgp);
  ctx.mark_stop();
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

}  // namespace

mma_status_t launch_batched_tile(const Ctx& ctx, bool bf16, bool out16,
                                 int64_t M, int64_t N, int64_t K,
                                 const void* A, const void* B, const void* C,
                                 void* D, int64_t batch, int group, int abid,
                                 int blgp) {
  using Fn = mma_status_t (*)(const Ctx&, int64_t, int64_t, int64_t,
                              const void*, const void*, const void*, void*,
                              int64_t, int, int, int);
  static const Fn table[8] = {
      run_tile<false, false, false>, run_tile<false, false, true>,
      run_tile<false, true, false>,  run_tile<false, true, true>,
      run_tile<true, false, false>,  run_tile<true, false, true>,
      run_tile<true, true, false>,   run_tile<true, true, true>};
  const bool stage_c = K == TK;
  return table[(bf16 ? 4 : 0) + (out16 ? 2 : 0) + (stage_c ? 1 : 0)](
      ctx, M, N, K, A, B, C, D, batch, group, abid, blgp);
}

}  // namespace mmagb
