// tcgen05 GEMM, D = A * B + C, A M x K row-major, B column-major (N rows of
// K), C/D M x N row-major: FP16/BF16 inputs with FP32 accumulation, and
// INT8 inputs with exact INT32 accumulation.
//
// The operation is the K-looped matrix multiply-accumulate of the page
// "CDNA2 dense MFMA builtins" (section "Naming convention": each step adds
// one K-panel's contribution to the M x N tile) with the FP16/BF16 -> FP32
// pairs of its "Builtin reference"; the tiled-kernel structure (block tile,
// K loop over staged panels, bounds-predicated store) is the one of
// "RDNA3 dense WMMA builtins", section "Using WMMA builtins as a compute
// policy", rebuilt for sm_103a:
//   * persistent CTAs (one per SM), tiles visited in M-grouped order so the
//     A and B panels in flight stay resident in L2;
//   * warp 0 drives TMA: 128x64 A and BNx64 B boxes, 128-byte swizzled,
//     into a STAGES-deep shared-memory ring guarded by mbarriers;
//   * warp 1 issues tcgen05.mma (M=128, N=BN, K=16) from one thread into a
//     double-buffered FP32 accumulator in tensor memory;
//   * warps 2..9 (two per tensor-memory lane quarter, one per column half)
//     drain the accumulator with tcgen05.ld, add C and store D with 16-byte
//     vector accesses, overlapping the next tile's MMAs.
// The same kernel carries the exact INT8 -> INT32 product on the BF16
// tensor pipe (sm_103a has no integer kind of tcgen05.mma): int8 operands
// are widened to BF16 (exact), K is split into chunks short enough that
// every FP32 partial sum is an exactly representable integer, and the
// epilogue sums the chunks in INT32 (see Epi::I32EXACT).
// Ragged M/N/K edges: TMA zero-fills out-of-bounds box elements (so they
// add nothing to the sum) and the epilogue predicates its stores.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace mmagb {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 x 2 bytes = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int kEpiWarps = 8;  // two per tensor-memory lane quarter
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kGroupM = 16;

// Epilogue modes:
//   F32      D = acc + C in FP32 (FP16/BF16 inputs)
//   I32EXACT the inputs are int8 values carried exactly in BF16; K is cut
//            into chunks whose partial sums stay below 2^24 in magnitude, so
//            each chunk's FP32 accumulator holds an exact integer; the
//            epilogue converts every chunk to INT32, sums the chunks, adds
//            the INT32 C and stores INT32 D (wrapping modulo 2^32).
enum class Epi { F32, I32EXACT };

// Chunk depth of the exact INT8 mode: |a*b| <= 2^14, so 1024 products keep
// every partial sum within 2^24, the range where FP32 represents all
// integers.
constexpr int kI8ChunkK = 1024;

template <int BN, int STAGES>
struct Layout {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int TOTAL = BAR_OFFSET + NUM_BARS * 8 + 16;
  static constexpr int ALLOC = TOTAL + 1024;  // room to align the base
  static constexpr uint32_t TMEM_COLS = 2 * BN;
};

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n,
                                            int& mb, int& nb) {
  const int per_group = kGroupM * num_n;
  const int g = t / per_group;
  const int first_m = g * kGroupM;
  const int gm = min(num_m - first_m, kGroupM);
  const int r = t - g * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

// Wait without giving up on the abort flag (used only while draining).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity,
                                                unsigned* status) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      return;
    }
  }
}

template <int BN, int STAGES, bool BF16, Epi EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const void* __restrict__ Cv, int64_t ldc,
                   void* __restrict__ Dv, int64_t ldd, int M, int N, int K,
                   int kb_per_chunk, unsigned* status) {
  using L = Layout<BN, STAGES>;
  constexpr int HALF = BN / 2;  // columns per epilogue warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFFSET);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int num_kb = (K + BK - 1) / BK;
  const int kpc = EPI == Epi::F32 ? num_kb : kb_per_chunk;
  const int chunks = (num_kb + kpc - 1) / kpc;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiThreads);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, num_m, num_n, mb, nb);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * L::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], L::STAGE_BYTES);
          tma_load_2d(&tmA, &full[stage], sa, kb * BK, mb * BM);
          tma_load_2d(&tmB, &full[stage], sa + L::A_BYTES, kb * BK, nb * BN);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every load still in flight land before the CTA exits.
        for (int s = 0; s < STAGES; ++s) {
          const uint32_t fills = issued / STAGES + (uint32_t(s) < issued % STAGES);
          if (fills) mbar_wait_drain(&full[s], (fills - 1) & 1u, status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_f16_f32(BF16, BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int ch = 0; ch < chunks && ok; ++ch) {
          if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
          const int kb0 = ch * kpc;
          const int kb1 = min(num_kb, kb0 + kpc);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * L::STAGE_BYTES);
            const uint64_t da = sw128_kmajor_desc(sa);
            const uint64_t db = sw128_kmajor_desc(sa + L::A_BYTES);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
              // advance 16 elements (32 bytes) along K inside the swizzle row
              umma_f16(d_tmem, da + uint64_t(2 * k), db + uint64_t(2 * k),
                       idesc, (kb != kb0 || k != 0) ? 1u : 0u);
            }
            umma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(&tfull[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      // Every MMA issued above completes before tensor memory is released.
      umma_commit(done);
      mbar_wait_drain(done, 0, status);
    }
  } else {
    // ------------------------------------------------ epilogue warps
    const int ew = warp - 2;           // 0 .. 7
    const int q = warp & 3;            // tensor-memory lane quarter
    const int h = ew >> 2;             // column half of the tile
    const int lane = threadIdx.x & 31;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, num_m, num_n, mb, nb);
      const int row = mb * BM + q * 32 + lane;
      const int colh = nb * BN + h * HALF;  // first column of this half
      [[maybe_unused]] uint32_t iacc[EPI == Epi::I32EXACT ? HALF : 1];
      if constexpr (EPI == Epi::I32EXACT) {
#pragma unroll
        for (int j = 0; j < HALF; ++j) iacc[j] = 0u;
      }
      for (int ch = 0; ch < chunks; ++ch) {
        ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + uint32_t(acc * BN + h * HALF) +
                               (uint32_t(q * 32) << 16);
        if constexpr (EPI == Epi::F32) {
          const float* C = static_cast<const float*>(Cv);
          float* D = static_cast<float*>(Dv);
#pragma unroll 1
          for (int c = 0; c < HALF / 32; ++c) {
            const int col0 = colh + c * 32;
            if (col0 >= N) break;
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + uint32_t(c * 32), r);
            tmem_ld_wait();
            if (row < M) {
              float* drow = D + int64_t(row) * ldd + col0;
              const float* crow = C ? C + int64_t(row) * ldc + col0 : nullptr;
              if (col0 + 32 <= N) {
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                  float4 cv = make_float4(0.f, 0.f, 0.f, 0.f);
                  if (crow) cv = __ldg(reinterpret_cast<const float4*>(crow) + v);
                  float4 o;
                  o.x = __uint_as_float(r[4 * v + 0]) + cv.x;
                  o.y = __uint_as_float(r[4 * v + 1]) + cv.y;
                  o.z = __uint_as_float(r[4 * v + 2]) + cv.z;
                  o.w = __uint_as_float(r[4 * v + 3]) + cv.w;
                  reinterpret_cast<float4*>(drow)[v] = o;
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  if (col0 + j < N)
                    drow[j] = __uint_as_float(r[j]) + (crow ? crow[j] : 0.f);
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < HALF / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + uint32_t(c * 32), r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              iacc[c * 32 + j] += uint32_t(__float2int_rn(__uint_as_float(r[j])));
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if constexpr (EPI == Epi::I32EXACT) {
        if (ok && row < M) {
          const int32_t* C = static_cast<const int32_t*>(Cv);
          int32_t* D = static_cast<int32_t*>(Dv);
          int32_t* drow = D + int64_t(row) * ldd + colh;
          const int32_t* crow = C ? C + int64_t(row) * ldc + colh : nullptr;
          if (colh + HALF <= N) {
#pragma unroll
            for (int v = 0; v < HALF / 4; ++v) {
              int4 cv = make_int4(0, 0, 0, 0);
              if (crow) cv = __ldg(reinterpret_cast<const int4*>(crow) + v);
              int4 o;
              o.x = int32_t(iacc[4 * v + 0] + uint32_t(cv.x));
              o.y = int32_t(iacc[4 * v + 1] + uint32_t(cv.y));
              o.z = int32_t(iacc[4 * v + 2] + uint32_t(cv.z));
              o.w = int32_t(iacc[4 * v + 3] + uint32_t(cv.w));
              reinterpret_cast<int4*>(drow)[v] = o;
            }
          } else {
#pragma unroll
            for (int j = 0; j < HALF; ++j) {
              if (colh + j < N)
                drow[j] = int32_t(iacc[j] + uint32_t(crow ? crow[j] : 0));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// int8 -> bfloat16 (exact: every int8 value has at most 8 significant bits).
// One flat index over 16-byte chunks of the rows of A then of B.
__global__ void __launch_bounds__(256)
    i8_to_bf16_kernel(const int8_t* __restrict__ A, int64_t lda, int M,
                      const int8_t* __restrict__ B, int64_t ldb, int N, int K,
                      uint16_t* __restrict__ W, int64_t ldw) {
  const int64_t cpr = (K + 15) / 16;  // chunks per row
  const int64_t total = int64_t(M + N) * cpr;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / cpr;
    const int c = int(i - r * cpr) * 16;
    const int8_t* src = r < M ? A + r * lda + c : B + (r - M) * ldb + c;
    uint16_t* dst = W + r * ldw + c;
    if (c + 16 <= K) {
      const int4 v = __ldcs(reinterpret_cast<const int4*>(src));
      const uint32_t w[4] = {uint32_t(v.x), uint32_t(v.y), uint32_t(v.z),
                             uint32_t(v.w)};
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int lo = int(int8_t((w[j >> 1] >> (16 * (j & 1))) & 0xFF));
        const int hi = int(int8_t((w[j >> 1] >> (16 * (j & 1) + 8)) & 0xFF));
        o[j] = (__float_as_uint(float(lo)) >> 16) |
               (__float_as_uint(float(hi)) & 0xFFFF0000u);
      }
      reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
      reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      for (int j = 0; c + j < K; ++j)
        dst[j] = uint16_t(__float_as_uint(float(src[j])) >> 16);
    }
  }
}

// ----------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D K-major operand: inner dim K (contiguous), outer dim rows, box
// 64 x box_rows, 128-byte swizzle, zero fill out of bounds.
bool make_kmajor_map(CUtensorMap* map, const void* base, int64_t K,
                     int64_t rows, int64_t ld_elems, int box_rows, bool bf16) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(ld_elems) * 2};
  cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map,
                   bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int STAGES, bool BF16, Epi EPI>
mma_status_t run(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                 const void* A, int64_t lda, const void* B, int64_t ldb,
                 const void* C, int64_t ldc, void* D, int64_t ldd) {
  using L = Layout<BN, STAGES>;
  CUtensorMap ta, tb;
  if (!make_kmajor_map(&ta, A, K, M, lda, BM, BF16) ||
      !make_kmajor_map(&tb, B, K, N, ldb, BN, BF16))
    return MMA_ERR_LAUNCH;
  auto kern = gemm_tc_kernel<BN, STAGES, BF16, EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           L::ALLOC) != cudaSuccess)
    return MMA_ERR_LAUNCH;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = int(tiles < ctx.num_sms ? tiles : ctx.num_sms);
  ctx.mark_start();
  kern<<<grid, kThreads, L::ALLOC, ctx.stream>>>(ta, tb, C, ldc, D, ldd,
                                                 int(M), int(N), int(K),
                                                 kI8ChunkK / BK, ctx.status);
  ctx.mark_stop();
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

// Wide tiles when there are enough of them to fill the chip, else narrow.
bool use_wide(const Ctx& ctx, int64_t M, int64_t N) {
  const int64_t wide_tiles = ((M + BM - 1) / BM) * ((N + 255) / 256);
  return N > 128 && wide_tiles >= ctx.num_sms;
}

}  // namespace

mma_status_t launch_gemm_tc_f16(const Ctx& ctx, bool bf16, int64_t M,
                                int64_t N, int64_t K, const void* A,
                                int64_t lda, const void* B, int64_t ldb,
                                const float* C, int64_t ldc, float* D,
                                int64_t ldd) {
  const bool wide = use_wide(ctx, M, N);
  if (bf16)
    return wide ? run<256, 4, true, Epi::F32>(ctx, M, N, K, A, lda, B, ldb, C, ldc, D, ldd)
                : run<128, 6, true, Epi::F32>(ctx, M, N, K, A, lda, B, ldb, C, ldc, D, ldd);
  return wide ? run<256, 4, false, Epi::F32>(ctx, M, N, K, A, lda, B, ldb, C, ldc, D, ldd)
              : run<128, 6, false, Epi::F32>(ctx, M, N, K, A, lda, B, ldb, C, ldc, D, ldd);
}

size_t gemm_i8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int64_t ldw = (K + 7) / 8 * 8;
  return size_t(M + N) * size_t(ldw) * 2;
}

mma_status_t launch_gemm_i8_tc(const Ctx& ctx, int64_t M, int64_t N,
                               int64_t K, const int8_t* A, int64_t lda,
                               const int8_t* B, int64_t ldb, const int32_t* C,
                               int64_t ldc, int32_t* D, int64_t ldd,
                               void* workspace) {
  const int64_t ldw = (K + 7) / 8 * 8;
  uint16_t* W = static_cast<uint16_t*>(workspace);
  const int64_t chunks = (M + N) * ((K + 15) / 16);
  int64_t blocks = (chunks + 255) / 256;
  if (blocks > int64_t(ctx.num_sms) * 16) blocks = int64_t(ctx.num_sms) * 16;
  i8_to_bf16_kernel<<<int(blocks), 256, 0, ctx.stream>>>(
      A, lda, int(M), B, ldb, int(N), int(K), W, ldw);
  if (cudaGetLastError() != cudaSuccess) return MMA_ERR_LAUNCH;
  const uint16_t* Aw = W;
  const uint16_t* Bw = W + M * ldw;
  return use_wide(ctx, M, N)
             ? run<256, 4, true, Epi::I32EXACT>(ctx, M, N, K, Aw, ldw, Bw, ldw,
                                                C, ldc, D, ldd)
             : run<128, 6, true, Epi::I32EXACT>(ctx, M, N, K, Aw, ldw, Bw, ldw,
                                                C, ldc, D, ldd);
}

}  // namespace mmagb
