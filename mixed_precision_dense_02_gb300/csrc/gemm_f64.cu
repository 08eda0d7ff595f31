// FP64 GEMM on the double-precision tensor path (mma.sync m8n8k4 DMMA):
//   D = A * B + C, all FP64, A row-major, B column- or row-major.
//
// Page "CDNA2 dense MFMA builtins", section "Builtin reference", FP64-
// accumulate builtins: FP64 inputs accumulate in FP64 with IEEE round-to-
// nearest-even (no round-toward-zero partial products).  DMMA accumulates
// each product with a fused multiply-add in FP64, which satisfies that.
//
// Block tile 64 x 64, K step 16, four warps each owning a 32 x 32 sub-tile
// (4 x 4 fragments of 8 x 8).  Operand tiles are staged through shared
// memory with register double buffering: the next K panel is fetched from
// global memory while the current one feeds the DMMAs.
#include "kernels.h"
#include "ptx.cuh"

namespace mmagb {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;
constexpr int kThreads = 128;
constexpr int LDS = TK + 4;  // padded row (doubles) of the shared tiles

// One 64 x 64 tile of D = A * B + C (block tile (blockIdx.y, blockIdx.x)).
template <bool B_ROW>
__device__ __forceinline__ void gemm_f64_tile(
    const double* __restrict__ A, int64_t lda, const double* __restrict__ B,
    int64_t ldb, const double* __restrict__ C, int64_t ldc,
    double* __restrict__ D, int64_t ldd, int M, int N, int K) {
  __shared__ double As[TM * LDS];
  __shared__ double Bs[TN * LDS];  // Bs[n][k]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;

  double acc[4][4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = 0.0;

  // Each thread fetches 8 elements of each operand tile per K panel.
  double ra[8], rb[8];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // A: 64 rows x 16 k; thread covers row tid/2, k (tid%2)*8 + i
      const int r = tid >> 1, k = (tid & 1) * 8 + i;
      const int gm = m0 + r, gk = k0 + k;
      ra[i] = (gm < M && gk < K) ? __ldg(A + int64_t(gm) * lda + gk) : 0.0;
    }
    if constexpr (!B_ROW) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int n = tid >> 1, k = (tid & 1) * 8 + i;
        const int gn = n0 + n, gk = k0 + k;
        rb[i] = (gn < N && gk < K) ? __ldg(B + int64_t(gn) * ldb + gk) : 0.0;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // row-major B: 16 k-rows of 64 n; thread covers n = tid%64,
        // k = (tid/64)*8 + i (coalesced along n)
        const int n = tid & 63, k = (tid >> 6) * 8 + i;
        const int gn = n0 + n, gk = k0 + k;
        rb[i] = (gn < N && gk < K) ? __ldg(B + int64_t(gk) * ldb + gn) : 0.0;
      }
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      As[(tid >> 1) * LDS + (tid & 1) * 8 + i] = ra[i];
      if constexpr (!B_ROW)
        Bs[(tid >> 1) * LDS + (tid & 1) * 8 + i] = rb[i];
      else
        Bs[(tid & 63) * LDS + (tid >> 6) * 8 + i] = rb[i];
    }
  };

  const int num_k = (K + TK - 1) / TK;
  if (num_k > 0) fetch(0);
  for (int kt = 0; kt < num_k; ++kt) {
    __syncthreads();
    stash();
    __syncthreads();
    if (kt + 1 < num_k) fetch((kt + 1) * TK);
#pragma unroll
    for (int kk = 0; kk < TK; kk += 4) {
      double af[4], bfr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) af[i] = As[(wm + i * 8 + g) * LDS + kk + t];
#pragma unroll
      for (int j = 0; j < 4; ++j) bfr[j] = Bs[(wn + j * 8 + g) * LDS + kk + t];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_f64_884(acc[i][j], af[i], bfr[j]);
    }
  }

  // fragment (i, j): rows wm + 8i + g, columns wn + 8j + 2t, +1
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + wm + i * 8 + g;
    if (r >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + wn + j * 8 + 2 * t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (c + h < N) {
          const double cv = C ? C[int64_t(r) * ldc + c + h] : 0.0;
          D[int64_t(r) * ldd + c + h] = acc[i][j][h] + cv;
        }
      }
    }
  }
}

// Grid z walks the batch entries (one problem: batch = 1).  Entry b reads
// the A tile (b / group) * group + abid and the B tile of lane-group
// pattern blgp (see launch_gemm_f64_batched); tiles are contiguous, tile t
// of A at A + t*M*lda, of B at B + t*(B_ROW ? K : N)*ldb, of C and D at
// t*M*ldc and t*M*ldd.
template <bool B_ROW>
__global__ void __launch_bounds__(kThreads)
    gemm_f64_kernel(const double* __restrict__ A, int64_t lda,
                    const double* __restrict__ B, int64_t ldb,
                    const double* __restrict__ C, int64_t ldc,
                    double* __restrict__ D, int64_t ldd, int M, int N, int K,
                    int batch, int group, int abid, int blgp) {
  const int64_t b_tile = int64_t(B_ROW ? K : N) * ldb;
  for (int b = blockIdx.z; b < batch; b += gridDim.z) {
    const int za = (b / group) * group + abid;
    const int q = b & 3;
    const int zb = (b & ~3) + (blgp == 0   ? q
                               : blgp == 1 ? (q & 1)
                               : blgp == 2 ? (2 | (q & 1))
                               : blgp == 3 ? ((q + 1) & 3)
                                           : blgp - 4);
    gemm_f64_tile<B_ROW>(A + int64_t(za) * M * lda, lda, B + zb * b_tile, ldb,
                         C ? C + int64_t(b) * M * ldc : nullptr, ldc,
                         D + int64_t(b) * M * ldd, ldd, M, N, K);
    __syncthreads();  // the shared tiles are reused by the next entry
  }
}

}  // namespace

mma_status_t launch_gemm_f64(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                             const double* A, int64_t lda, const double* B,
                             int64_t ldb, bool b_row_major, const double* C,
                             int64_t ldc, double* D, int64_t ldd) {
  const int64_t gx = (N + TN - 1) / TN, gy = (M + TM - 1) / TM;
  if (gy > 65535) return MMA_ERR_UNSUPPORTED;
  const dim3 grid{unsigned(gx), unsigned(gy), 1u};
  ctx.mark_start();
  if (b_row_major)
    gemm_f64_kernel<true><<<grid, kThreads, 0, ctx.stream>>>(
        A, lda, B, ldb, C, ldc, D, ldd, int(M), int(N), int(K), 1, 1, 0, 0);
  else
    gemm_f64_kernel<false><<<grid, kThreads, 0, ctx.stream>>>(
        A, lda, B, ldb, C, ldc, D, ldd, int(M), int(N), int(K), 1, 1, 0, 0);
  ctx.mark_stop();
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

// Batched FP64 (column-major B tiles): grid z covers the entries.
mma_status_t launch_gemm_f64_batched(const Ctx& ctx, int64_t M, int64_t N,
                                     int64_t K, const double* A, int64_t lda,
                                     const double* B, int64_t ldb,
                                     const double* C, int64_t ldc, double* D,
                                     int64_t ldd, int64_t batch, int group,
                                     int abid, int blgp) {
  const int64_t gx = (N + TN - 1) / TN, gy = (M + TM - 1) / TM;
  if (gy > 65535 || batch > int64_t(INT32_MAX)) return MMA_ERR_UNSUPPORTED;
  const int64_t gz = batch < 65535 ? batch : 65535;
  const dim3 grid{unsigned(gx), unsigned(gy), unsigned(gz)};
  ctx.mark_start();
  gemm_f64_kernel<false><<<grid, kThreads, 0, ctx.stream>>>(
      A, lda, B, ldb, C, ldc, D, ldd, int(M), int(N), int(K), int(batch),
      group, abid, blgp);
  ctx.mark_stop();
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

}  // namespace mmagb
