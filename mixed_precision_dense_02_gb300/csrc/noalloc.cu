// mma_gemm_i8_noalloc: the exact INT8 -> INT32 GEMM on the tensor pipe
// without any device allocation.
//
// mma_gemm runs large INT8 products on the BF16 tensor pipe, which needs
// scratch space for BF16 copies of A and B; it gets that space by growing a
// library-owned buffer with cudaMalloc.  Some callers cannot let a library
// do that: a program whose own pool allocator has already reserved the
// device memory it may use (a cudaMalloc behind its back either fails or
// eats into memory the pool was promised), and a latency-bound service that
// forbids allocation after start-up, because cudaMalloc and cudaFree can
// block and synchronise the whole device at an unpredictable moment.  This
// entry point serves them: its scratch is a fixed array in the library's
// own device image, sized once (MMA_NOALLOC_SCRATCH_BYTES) and held by every
// GPU that loads the library until the process exits.
//
// Set-up: the first call on each device (with that device current) looks
// the array's device address up with cudaGetSymbolAddress and caches it
// for the device's context (a context that replaces it, after
// cudaDeviceReset, looks it up again); make that first call before any
// stream capture begins.  Every call on a
// device shares the one array and leaves its contents behind; nothing in it
// has to start at zero, because each call rewrites every scratch element it
// later reads.  Two calls whose work overlaps on the GPU (different
// streams, no ordering between them) race on the array: order them.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

// The scratch array.  In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[MMA_NOALLOC_SCRATCH_BYTES];

namespace mmagb {
namespace {

PerContext<void*> g_scratch;

// Device address of the scratch array in the context of `ctx` (whose device
// is current), or null if the lookup fails.
void* scratch_address(const Ctx& ctx) {
  void* ptr = nullptr;
  if (!g_scratch.get(ctx, &ptr, [](void** v) {
        if (cudaGetSymbolAddress(v, g_noalloc_scratch) != cudaSuccess) {
          cudaGetLastError();
          return false;
        }
        return *v != nullptr;
      }))
    return nullptr;
  return ptr;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace
}  // namespace mmagb

using namespace mmagb;

extern "C" mma_status_t mma_gemm_i8_noalloc(int64_t M, int64_t N, int64_t K,
                                            const void* A, int64_t lda,
                                            const void* B, int64_t ldb,
                                            const void* C, int64_t ldc,
                                            void* D, int64_t ldd,
                                            void* stream) {
  constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return MMA_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MMA_OK;
  if (D == nullptr || ldd < N) return MMA_ERR_INVALID_ARG;
  if (C != nullptr && ldc < N) return MMA_ERR_INVALID_ARG;
  if (C != nullptr && C == D && ldc != ldd) return MMA_ERR_INVALID_ARG;
  if (K > 0) {
    if (A == nullptr || B == nullptr || lda < K || ldb < K)
      return MMA_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || (lda & 15) || (ldb & 15))
      return MMA_ERR_MISALIGNED;
  }
  if (!aligned16(D) || ((ldd * 4) & 15)) return MMA_ERR_MISALIGNED;
  if (C != nullptr && (!aligned16(C) || ((ldc * 4) & 15)))
    return MMA_ERR_MISALIGNED;
  // Problems whose BF16 copies of A and B do not fit the fixed scratch.
  const double need = double(M + N) * double((K + 7) / 8 * 8) * 2.0;
  if (K > 0 && need > double(MMA_NOALLOC_SCRATCH_BYTES))
    return MMA_ERR_UNSUPPORTED;

  Ctx ctx{};
  if (!current_ctx(stream, &ctx)) return MMA_ERR_NO_DEVICE;
  attach_profile(ctx);
  if (K == 0) return launch_copy_c(ctx, M, N, 4, C, ldc, D, ldd);
  void* scratch = scratch_address(ctx);
  if (scratch == nullptr) return MMA_ERR_LAUNCH;
  return launch_gemm_i8_tc(ctx, M, N, K, static_cast<const int8_t*>(A), lda,
                           static_cast<const int8_t*>(B), ldb,
                           static_cast<const int32_t*>(C), ldc,
                           static_cast<int32_t*>(D), ldd, scratch,
                           /*b_row_major=*/false, /*a_signed=*/true,
                           /*b_signed=*/true, /*clamp=*/false);
}
