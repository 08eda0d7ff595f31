// INT8 GEMM with INT32 accumulation on the warp-level integer tensor path
// (mma.sync m16n8k32 .s8.s8.s32):
//   D = A * B + C,  A M x K row-major int8, B column-major (N rows of K)
//   int8, C/D M x N row-major int32.
//
// Page "CDNA2 dense MFMA builtins", section "Builtin reference", INT32-
// accumulate builtins (signed 8-bit inputs, INT32 accumulator), and
// "RDNA3 dense WMMA builtins", section "Builtin reference" (the iu8 builtin
// returns srcA x srcB + srcC; a_neg/b_neg select signed inputs).  The
// integer sum is exact; INT32 results wrap modulo 2^32 like the hardware
// accumulator (no clamp).
//
// sm_103a has no integer kind of tcgen05.mma, so this kernel uses the
// warp-synchronous IMMA instruction: block tile 128 x 128, K panel 64
// bytes, 8 warps of 64 x 32, a 4-stage cp.async ring, 16-byte rows chunks
// XOR-swizzled in shared memory so ldmatrix reads are conflict-free.
#include "kernels.h"
#include "ptx.cuh"

namespace mmagb {
namespace {

constexpr int TM = 128, TN = 128, TK = 64;
constexpr int STAGES = 4;
constexpr int kThreads = 256;
constexpr int TILE_BYTES = TM * TK;  // A and B tiles are both 128 x 64 bytes

// byte offset of (row, 16-byte chunk) inside a 64-byte-row tile
__device__ __forceinline__ int swz(int row, int chunk) {
  return row * TK + ((chunk ^ ((row >> 1) & 3)) << 4);
}

__global__ void __launch_bounds__(kThreads)
    gemm_i8_imma_kernel(const int8_t* __restrict__ A, int64_t lda,
                        const int8_t* __restrict__ B, int64_t ldb,
                        const int32_t* __restrict__ C, int64_t ldc,
                        int32_t* __restrict__ D, int64_t ldd, int M, int N,
                        int K) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = (warp >> 2) * 64, wn = (warp & 3) * 32;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int num_k = (K + TK - 1) / TK;
  const uint32_t sbase = smem_u32(smem);

  auto load_stage = [&](int stage, int kt) {
    const uint32_t sa = sbase + stage * 2 * TILE_BYTES;
    const uint32_t sb = sa + TILE_BYTES;
    const int k0 = kt * TK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int id = tid + i * kThreads;  // 0..511
      const int r = id >> 2, c = id & 3;
      const int gk = k0 + c * 16;
      const int kb = K - gk;
      const int bytes = kb >= 16 ? 16 : (kb > 0 ? kb : 0);
      {
        const int gm = m0 + r;
        const int nb = gm < M ? bytes : 0;
        const int8_t* src = nb ? A + int64_t(gm) * lda + gk : A;
        cp_async_16_zfill(sa + swz(r, c), src, nb);
      }
      {
        const int gn = n0 + r;
        const int nb = gn < N ? bytes : 0;
        const int8_t* src = nb ? B + int64_t(gn) * ldb + gk : B;
        cp_async_16_zfill(sb + swz(r, c), src, nb);
      }
    }
  };

  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[i][j][v] = 0;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < num_k) load_stage(s, s);
    cp_async_commit();
  }

  const int q = lane >> 3, rr = lane & 7;
  for (int kt = 0; kt < num_k; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {
      const int nk = kt + STAGES - 1;
      if (nk < num_k) load_stage(nk % STAGES, nk);
      cp_async_commit();
    }
    const uint32_t sa = sbase + (kt % STAGES) * 2 * TILE_BYTES;
    const uint32_t sb = sa + TILE_BYTES;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t af[4][4], bfr[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // matrices: rows +0/+8 (q&1), k bytes +0/+16 (q>>1)
        const int row = wm + i * 16 + (q & 1) * 8 + rr;
        ldmatrix_x4(af[i], sa + swz(row, ks * 2 + (q >> 1)));
      }
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        // matrices: n-tile j / j+1 (q>>1), k bytes +0/+16 (q&1)
        const int row = wn + (j + (q >> 1)) * 8 + rr;
        uint32_t r4[4];
        ldmatrix_x4(r4, sb + swz(row, ks * 2 + (q & 1)));
        bfr[j][0] = r4[0];
        bfr[j][1] = r4[1];
        bfr[j + 1][0] = r4[2];
        bfr[j + 1][1] = r4[3];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_s8_16832(acc[i][j], af[i], bfr[j]);
    }
  }
  cp_async_wait<0>();

  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = m0 + wm + i * 16 + g + h * 8;
      if (r >= M) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = n0 + wn + j * 8 + 2 * t;
        const int v0 = acc[i][j][2 * h], v1 = acc[i][j][2 * h + 1];
        if (c + 1 < N) {
          int2 cv = make_int2(0, 0);
          if (C) cv = *reinterpret_cast<const int2*>(C + int64_t(r) * ldc + c);
          int2 o;
          o.x = int(unsigned(v0) + unsigned(cv.x));
          o.y = int(unsigned(v1) + unsigned(cv.y));
          *reinterpret_cast<int2*>(D + int64_t(r) * ldd + c) = o;
        } else if (c < N) {
          const int cv = C ? C[int64_t(r) * ldc + c] : 0;
          D[int64_t(r) * ldd + c] = int(unsigned(v0) + unsigned(cv));
        }
      }
    }
  }
}

}  // namespace

mma_status_t launch_gemm_i8_imma(const Ctx& ctx, int64_t M, int64_t N,
                                 int64_t K, const int8_t* A, int64_t lda,
                                 const int8_t* B, int64_t ldb,
                                 const int32_t* C, int64_t ldc, int32_t* D,
                                 int64_t ldd) {
  const int64_t gx = (N + TN - 1) / TN, gy = (M + TM - 1) / TM;
  if (gy > 65535) return MMA_ERR_UNSUPPORTED;
  constexpr int smem = STAGES * 2 * TILE_BYTES;
  if (cudaFuncSetAttribute(gemm_i8_imma_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return MMA_ERR_LAUNCH;
  ctx.mark_start();
  gemm_i8_imma_kernel<<<dim3(unsigned(gx), unsigned(gy)), kThreads, smem,
                        ctx.stream>>>(A, lda, B, ldb, C, ldc, D, ldd, int(M),
                                      int(N), int(K));
  ctx.mark_stop();
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

}  // namespace mmagb
