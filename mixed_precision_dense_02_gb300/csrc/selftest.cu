// mma_selftest_wait_timeout, mma_selftest_gemm_abort: the failure-detection
// path of the pipeline kernels, exercised on purpose without faulting or
// hanging the GPU.
//
// Every wait of the tcgen05 pipeline (TMA stage, accumulator hand-off, C
// block) is mbar_wait from ptx.cuh: bounded by a time limit, after which it
// raises the CTA's abort flag, records MMA_ERR_TIMEOUT in the library's
// device status word and returns false, so the kernel drains and exits and
// the context stays usable.  This kernel runs that same wait on an mbarrier
// that no thread ever arrives on, with a short caller-chosen limit, so the
// wait runs out exactly as a stuck pipeline's would.  The second runs the
// tcgen05 GEMM kernel itself, single CTAs or a CTA pair, with its producer
// told to issue no loads and its waits limited to limit_ns: the MMA
// issuer's first stage wait runs out with no copy or MMA in flight, and
// the kernel's own abort path (abort flag, drain, tensor-memory release,
// cluster exit) runs for real.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace mmagb {
namespace {

__global__ void wait_timeout_kernel(unsigned* status,
                                    unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival, which never comes
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // returns false after limit_ns, having recorded the timeout
    (void)mbar_wait(&bar, 0u, &abort_flag, status, limit_ns);
  }
  __syncthreads();
}

}  // namespace
}  // namespace mmagb

using namespace mmagb;

extern "C" mma_status_t mma_selftest_wait_timeout(int64_t limit_ns,
                                                  void* stream) {
  // 1 us .. 10 s
  if (limit_ns < 1000 || limit_ns > 10000000000ll) return MMA_ERR_INVALID_ARG;
  Ctx ctx{};
  if (!current_ctx(stream, &ctx)) return MMA_ERR_NO_DEVICE;
  wait_timeout_kernel<<<1, 32, 0, ctx.stream>>>(
      ctx.status, static_cast<unsigned long long>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

extern "C" mma_status_t mma_selftest_gemm_abort(int cluster, int64_t limit_ns,
                                                const void* A, const void* B,
                                                void* D, void* stream) {
  if (cluster != 1 && cluster != 2) return MMA_ERR_INVALID_ARG;
  if (limit_ns < 1000000 || limit_ns > 10000000000ll) return MMA_ERR_INVALID_ARG;
  if (!A || !B || !D) return MMA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(D)) & 15u)
    return MMA_ERR_MISALIGNED;
  Ctx ctx{};
  if (!current_ctx(stream, &ctx)) return MMA_ERR_NO_DEVICE;
  return launch_gemm_tc_abort_selftest(ctx, cluster, limit_ns, A, B, D);
}
