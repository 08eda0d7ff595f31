// C ABI of the library (declared in include/mma_gb300.h): argument
// validation, per-device set-up and dispatch to the kernels.  Nothing here
// computes any part of D = A * B + C; every arithmetic step runs on the GPU.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"

namespace mmagb {

// Device-side status word: bounded pipeline waits OR their error bits in.
__device__ unsigned g_mma_status;

namespace {

struct DeviceInfo {
  bool ready = false;
  bool usable = false;
  int num_sms = 0;
  unsigned* status = nullptr;
  uint64_t gen = 0;  // context the fields above were set up in
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Profiling ring: while active, each call records one event pair around its
// dominant kernel.  Events are created once and reused.
constexpr int kProfMax = 4096;
struct Profile {
  bool active = false;
  int device = -1;
  int count = 0;
  cudaEvent_t ev[2 * kProfMax] = {};
  bool created = false;
  uint64_t gen = 0;  // context the events belong to
};
Profile g_prof;
std::mutex g_prof_mu;

// INT8 scratch: one buffer per device for the BF16 copies of A and B,
// allocated on the first INT8 call that needs it and grown (never shrunk)
// when a larger problem arrives; kept until the process exits.  An event
// records the last call that used it, and a call on another stream waits
// for that event first, so concurrent calls never share it in flight.
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  cudaEvent_t done = nullptr;
  uint64_t gen = 0;  // context the buffer and event belong to
};
Workspace g_ws[kMaxDevices];
std::mutex g_ws_mu;

// Stream-K hand-off flags: one small buffer per device (zeroed when
// allocated) and the sequence number of the last stream-K call; calls use
// the flags in the order the scratch buffer's event imposes on them.
struct StreamKFlags {
  unsigned* ptr = nullptr;
  size_t count = 0;
  unsigned seq = 0;
  uint64_t gen = 0;
};
StreamKFlags g_skf[kMaxDevices];

// Identifier of the calling thread's current CUDA context plus one (0 when
// no context is current yet).  Without the driver's context-id call every
// context reads as 1, and state is then set up once per device.
uint64_t current_context_gen() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  });
  if (!get_cur || !get_id) return 1;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 1;
  return uint64_t(id) + 1;
}

// Per-device set-up, once per context, with that device current: SM count,
// the architecture check and the device address of the status word.  A
// replaced context (cudaDeviceReset) is set up again.
const DeviceInfo* device_info(int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  *dev_out = dev;
  uint64_t gen = current_context_gen();
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready || (gen != 0 && gen != d.gen)) {
    d = DeviceInfo{};
    d.ready = true;
    int major = 0, minor = 0, sms = 0;
    void* p = nullptr;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor,
                               dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor,
                               dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ==
            cudaSuccess &&
        major == 10 && minor == 3 &&
        cudaGetSymbolAddress(&p, g_mma_status) == cudaSuccess) {
      d.usable = true;
      d.num_sms = sms;
      d.status = static_cast<unsigned*>(p);
    } else {
      cudaGetLastError();
    }
    // the symbol lookup made the device's primary context current
    if (gen == 0) gen = current_context_gen();
    d.gen = gen != 0 ? gen : 1;
  }
  return d.usable ? &d : nullptr;
}

Ctx make_ctx(void* stream, int dev, const DeviceInfo* info) {
  return Ctx{static_cast<cudaStream_t>(stream), dev, info->num_sms,
             info->status, info->gen};
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool ld_ok(int64_t ld, int64_t elem) { return ((ld * elem) & 15) == 0; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

__global__ void copy_c_kernel(const uint8_t* __restrict__ C, int64_t ldc_b,
                              uint8_t* __restrict__ D, int64_t ldd_b,
                              int64_t M, int64_t N, int elem) {
  const int64_t total = M * N;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / N, c = i % N;
    if (elem == 8) {
      const uint64_t v =
          C ? *reinterpret_cast<const uint64_t*>(C + r * ldc_b + c * 8) : 0ull;
      *reinterpret_cast<uint64_t*>(D + r * ldd_b + c * 8) = v;
    } else if (elem == 2) {
      const uint16_t v =
          C ? *reinterpret_cast<const uint16_t*>(C + r * ldc_b + c * 2) : 0u;
      *reinterpret_cast<uint16_t*>(D + r * ldd_b + c * 2) = v;
    } else {
      const uint32_t v =
          C ? *reinterpret_cast<const uint32_t*>(C + r * ldc_b + c * 4) : 0u;
      *reinterpret_cast<uint32_t*>(D + r * ldd_b + c * 4) = v;
    }
  }
}

}  // namespace

bool current_ctx(void* stream, Ctx* out) {
  int dev = -1;
  const DeviceInfo* info = device_info(&dev);
  if (!info) return false;
  *out = make_ctx(stream, dev, info);
  return true;
}

void attach_profile(Ctx& ctx) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof.active || g_prof.device != ctx.device || g_prof.gen != ctx.gen ||
      g_prof.count >= kProfMax)
    return;
  ctx.prof_start = g_prof.ev[2 * g_prof.count];
  ctx.prof_stop = g_prof.ev[2 * g_prof.count + 1];
  ++g_prof.count;
}

mma_status_t launch_copy_c(const Ctx& ctx, int64_t M, int64_t N,
                           int elem_bytes, const void* C, int64_t ldc, void* D,
                           int64_t ldd) {
  int64_t blocks = (M * N + 255) / 256;
  if (blocks > int64_t(ctx.num_sms) * 16) blocks = int64_t(ctx.num_sms) * 16;
  copy_c_kernel<<<int(blocks), 256, 0, ctx.stream>>>(
      static_cast<const uint8_t*>(C), ldc * elem_bytes,
      static_cast<uint8_t*>(D), ldd * elem_bytes, M, N, elem_bytes);
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

}  // namespace mmagb

using namespace mmagb;

namespace {

// Problems at least this large (M*N*K) take the tcgen05 exact-INT8 path;
// smaller ones stay on the IMMA kernel, which needs no scratch.
constexpr double kI8TensorCoreMinWork = 16777216.0;  // 2^24

// Run `enqueue(workspace)` with at least `need` bytes of the device's
// scratch buffer, growing it if needed, ordered after the buffer's previous
// user (an event) and marking this stream as its new user.
template <class F>
mma_status_t with_workspace(const Ctx& ctx, size_t need, F&& enqueue) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Workspace& w = g_ws[ctx.device];
  if (w.gen != ctx.gen) {
    // set up in a context that has since been replaced: its buffer and
    // event went with it
    w = Workspace{};
    w.gen = ctx.gen;
  }
  if (!w.done &&
      cudaEventCreateWithFlags(&w.done, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    w.done = nullptr;
    return MMA_ERR_LAUNCH;
  }
  if (w.bytes < need) {
    if (w.ptr) {
      if (cudaEventSynchronize(w.done) != cudaSuccess) return MMA_ERR_LAUNCH;
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    const size_t grain = size_t(64) << 20;
    const size_t bytes = (need + grain - 1) / grain * grain;
    if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) {
      cudaGetLastError();
      w.ptr = nullptr;
      return MMA_ERR_NO_MEMORY;
    }
    w.bytes = bytes;
  }
  if (cudaStreamWaitEvent(ctx.stream, w.done, 0) != cudaSuccess)
    return MMA_ERR_LAUNCH;
  const mma_status_t st = enqueue(w.ptr);
  if (cudaEventRecord(w.done, ctx.stream) != cudaSuccess) return MMA_ERR_LAUNCH;
  return st;
}

}  // namespace

namespace {

// Enqueue a stream-K GEMM: partial sums in the scratch buffer, hand-off
// flags with a fresh sequence number.  Runs under the scratch buffer's lock
// (inside with_workspace), which also orders the flags' users.
mma_status_t enqueue_stream_k(const Ctx& ctx, bool bf16, int64_t M, int64_t N,
                              int64_t K, const void* A, int64_t lda,
                              const void* B, int64_t ldb, const void* C,
                              int64_t ldc, void* D, int64_t ldd, void* ws) {
  StreamKFlags& f = g_skf[ctx.device];
  if (f.gen != ctx.gen) f = StreamKFlags{};  // set up in a replaced context
  const size_t need = gemm_sk_flag_count(ctx.num_sms);
  if (f.ptr == nullptr || f.count < need) {
    if (f.ptr) cudaFree(f.ptr);
    f = StreamKFlags{};
    void* p = nullptr;
    if (cudaMalloc(&p, need * sizeof(unsigned)) != cudaSuccess) {
      cudaGetLastError();
      return MMA_ERR_NO_MEMORY;
    }
    if (cudaMemset(p, 0, need * sizeof(unsigned)) != cudaSuccess) {
      cudaFree(p);
      cudaGetLastError();
      return MMA_ERR_LAUNCH;
    }
    f.ptr = static_cast<unsigned*>(p);
    f.count = need;
    f.gen = ctx.gen;
  }
  // nonzero and different from every value still in the flags; after 2^32
  // calls the flags are cleared again before the numbers repeat
  if (++f.seq == 0) {
    if (cudaMemsetAsync(f.ptr, 0, f.count * sizeof(unsigned), ctx.stream) !=
        cudaSuccess)
      return MMA_ERR_LAUNCH;
    f.seq = 1;
  }
  return launch_gemm_sk(ctx, bf16, M, N, K, A, lda, B, ldb,
                        static_cast<const float*>(C), ldc,
                        static_cast<float*>(D), ldd, static_cast<float*>(ws),
                        f.ptr, f.seq);
}

// Element sizes of a supported (dtype_in, dtype_acc) pair, or false.
bool pair_sizes(int in, int acc, int64_t* in_b, int64_t* acc_b) {
  if ((in == MMA_F16 || in == MMA_BF16) && acc == MMA_F32) {
    *in_b = 2;
    *acc_b = 4;
    return true;
  }
  if ((in == MMA_F16 || in == MMA_BF16) && acc == in) {  // 16-bit accumulate
    *in_b = 2;
    *acc_b = 2;
    return true;
  }
  if (in == MMA_I8 && acc == MMA_I32) {
    *in_b = 1;
    *acc_b = 4;
    return true;
  }
  if (in == MMA_F64 && acc == MMA_F64) {
    *in_b = 8;
    *acc_b = 8;
    return true;
  }
  return false;
}

}  // namespace

namespace {

// Argument checks shared by the dense entry points (element sizes eb of A
// and B, ea of C and D).  Returns MMA_OK when the call should go ahead.
mma_status_t check_dense_args(int64_t eb, int64_t ea, int layout_b, int64_t M,
                              int64_t N, int64_t K, const void* A, int64_t lda,
                              const void* B, int64_t ldb, const void* C,
                              int64_t ldc, const void* D, int64_t ldd) {
  if (layout_b != MMA_COL_MAJOR && layout_b != MMA_ROW_MAJOR)
    return MMA_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return MMA_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MMA_OK;
  const bool b_row = layout_b == MMA_ROW_MAJOR;
  if (D == nullptr || ldd < N) return MMA_ERR_INVALID_ARG;
  if (C != nullptr && ldc < N) return MMA_ERR_INVALID_ARG;
  if (C != nullptr && C == D && ldc != ldd) return MMA_ERR_INVALID_ARG;
  if (K > 0) {
    if (A == nullptr || B == nullptr) return MMA_ERR_INVALID_ARG;
    if (lda < K || ldb < (b_row ? N : K)) return MMA_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !ld_ok(lda, eb) || !ld_ok(ldb, eb))
      return MMA_ERR_MISALIGNED;
  }
  if (!aligned16(D) || !ld_ok(ldd, ea)) return MMA_ERR_MISALIGNED;
  if (C != nullptr && (!aligned16(C) || !ld_ok(ldc, ea)))
    return MMA_ERR_MISALIGNED;
  return MMA_OK;
}

}  // namespace

extern "C" mma_status_t mma_gemm_ex(int dtype_in, int dtype_acc, int64_t M,
                                    int64_t N, int64_t K, const void* A,
                                    int64_t lda, const void* B, int64_t ldb,
                                    int layout_b, const void* C, int64_t ldc,
                                    void* D, int64_t ldd, void* stream) {
  int64_t eb = 0, ea = 0;
  if (!pair_sizes(dtype_in, dtype_acc, &eb, &ea)) return MMA_ERR_UNSUPPORTED;
  const mma_status_t chk = check_dense_args(eb, ea, layout_b, M, N, K, A, lda,
                                            B, ldb, C, ldc, D, ldd);
  if (chk != MMA_OK || M == 0 || N == 0) return chk;
  const bool b_row = layout_b == MMA_ROW_MAJOR;
  int dev = -1;
  const DeviceInfo* info = device_info(&dev);
  if (!info) return MMA_ERR_NO_DEVICE;
  Ctx ctx = make_ctx(stream, dev, info);
  attach_profile(ctx);

  if (K == 0) return launch_copy_c(ctx, M, N, int(ea), C, ldc, D, ldd);
  switch (dtype_in) {
    case MMA_F16:
    case MMA_BF16: {
      const bool bf16 = dtype_in == MMA_BF16;
      const bool out16 = dtype_acc != MMA_F32;
      // fewer output tiles than SMs: K split across every SM (stream-K)
      if (!b_row && !out16 && gemm_sk_fits(ctx.num_sms, M, N, K))
        return with_workspace(ctx, gemm_sk_workspace_bytes(ctx.num_sms),
                              [&](void* ws) {
                                return enqueue_stream_k(ctx, bf16, M, N, K, A,
                                                        lda, B, ldb, C, ldc, D,
                                                        ldd, ws);
                              });
      if (!b_row)
        return launch_gemm_tc_f16(ctx, bf16, out16, M, N, K, A, lda, B, ldb, C,
                                  ldc, D, ldd);
      return with_workspace(ctx, gemm_tc_rowb_workspace_bytes(N, K),
                            [&](void* ws) {
                              return launch_gemm_tc_f16_rowb(
                                  ctx, bf16, out16, M, N, K, A, lda, B, ldb, C,
                                  ldc, D, ldd, ws);
                            });
    }
    case MMA_I8: {
      const int8_t* A8 = static_cast<const int8_t*>(A);
      const int8_t* B8 = static_cast<const int8_t*>(B);
      const int32_t* Ci = static_cast<const int32_t*>(C);
      int32_t* Di = static_cast<int32_t*>(D);
      // Large problems, and every row-major B, take the tensor-pipe path.
      if (b_row || double(M) * double(N) * double(K) >= kI8TensorCoreMinWork)
        return with_workspace(ctx, gemm_i8_tc_workspace_bytes(M, N, K),
                              [&](void* ws) {
                                return launch_gemm_i8_tc(
                                    ctx, M, N, K, A8, lda, B8, ldb, Ci, ldc,
                                    Di, ldd, ws, b_row, true, true, false);
                              });
      return launch_gemm_i8_imma(ctx, M, N, K, A8, lda, B8, ldb, Ci, ldc, Di,
                                 ldd);
    }
    case MMA_F64:
      return launch_gemm_f64(ctx, M, N, K, static_cast<const double*>(A), lda,
                             static_cast<const double*>(B), ldb, b_row,
                             static_cast<const double*>(C), ldc,
                             static_cast<double*>(D), ldd);
    default:
      return MMA_ERR_UNSUPPORTED;
  }
}

extern "C" mma_status_t mma_gemm_i8_ex(int64_t M, int64_t N, int64_t K,
                                       const void* A, int64_t lda, int a_neg,
                                       const void* B, int64_t ldb, int b_neg,
                                       int layout_b, const void* C,
                                       int64_t ldc, void* D, int64_t ldd,
                                       int clamp, void* stream) {
  const bool a_signed = a_neg != 0, b_signed = b_neg != 0;
  // signed x signed without saturation is the plain INT8 product
  if (a_signed && b_signed && clamp == 0)
    return mma_gemm_ex(MMA_I8, MMA_I32, M, N, K, A, lda, B, ldb, layout_b, C,
                       ldc, D, ldd, stream);
  const mma_status_t chk = check_dense_args(1, 4, layout_b, M, N, K, A, lda,
                                            B, ldb, C, ldc, D, ldd);
  if (chk != MMA_OK || M == 0 || N == 0) return chk;
  int dev = -1;
  const DeviceInfo* info = device_info(&dev);
  if (!info) return MMA_ERR_NO_DEVICE;
  Ctx ctx = make_ctx(stream, dev, info);
  attach_profile(ctx);
  if (K == 0) {
    // D = C: a 32-bit C is in range, so saturation changes nothing
    return launch_copy_c(ctx, M, N, 4, C, ldc, D, ldd);
  }
  const bool b_row = layout_b == MMA_ROW_MAJOR;
  return with_workspace(
      ctx, gemm_i8_tc_workspace_bytes(M, N, K), [&](void* ws) {
        return launch_gemm_i8_tc(ctx, M, N, K, static_cast<const int8_t*>(A),
                                 lda, static_cast<const int8_t*>(B), ldb,
                                 static_cast<const int32_t*>(C), ldc,
                                 static_cast<int32_t*>(D), ldd, ws, b_row,
                                 a_signed, b_signed, clamp != 0);
      });
}

extern "C" mma_status_t mma_gemm(int dtype_in, int dtype_acc, int64_t M,
                                 int64_t N, int64_t K, const void* A,
                                 int64_t lda, const void* B, int64_t ldb,
                                 const void* C, int64_t ldc, void* D,
                                 int64_t ldd, void* stream) {
  return mma_gemm_ex(dtype_in, dtype_acc, M, N, K, A, lda, B, ldb,
                     MMA_COL_MAJOR, C, ldc, D, ldd, stream);
}

extern "C" mma_status_t mma_gemm_batched_ex(
    int dtype_in, int dtype_acc, int64_t M, int64_t N, int64_t K,
    const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
    int64_t ldc, void* D, int64_t ldd, int64_t batch, int a_broadcast_group,
    int a_broadcast_id, int b_lane_group_pattern, void* stream) {
  int64_t eb = 0, ea = 0;
  if (!pair_sizes(dtype_in, dtype_acc, &eb, &ea)) return MMA_ERR_UNSUPPORTED;
  const int G = a_broadcast_group;
  const int blgp = b_lane_group_pattern;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return MMA_ERR_INVALID_ARG;
  if (a_broadcast_id < 0 || a_broadcast_id >= G) return MMA_ERR_INVALID_ARG;
  if (blgp < 0 || blgp > 7) return MMA_ERR_INVALID_ARG;
  if (batch < 0 || batch % G != 0) return MMA_ERR_INVALID_ARG;
  if (blgp != 0 && batch % 4 != 0) return MMA_ERR_INVALID_ARG;
  if (batch > int64_t(INT32_MAX)) return MMA_ERR_UNSUPPORTED;
  if (M < 0 || N < 0 || K < 0) return MMA_ERR_INVALID_ARG;
  if (batch == 0) return MMA_OK;
  // each tile is checked as a single column-major-B problem
  const mma_status_t chk = check_dense_args(eb, ea, MMA_COL_MAJOR, M, N, K, A,
                                            lda, B, ldb, C, ldc, D, ldd);
  if (chk != MMA_OK || batch == 0 || M == 0 || N == 0) return chk;
  int dev = -1;
  const DeviceInfo* info = device_info(&dev);
  if (!info) return MMA_ERR_NO_DEVICE;
  Ctx ctx = make_ctx(stream, dev, info);
  attach_profile(ctx);
  // K == 0: D = C tile by tile; the tiles are contiguous, so batch * M rows
  if (K == 0) return launch_copy_c(ctx, batch * M, N, int(ea), C, ldc, D, ldd);
  const int abid = a_broadcast_id;
  switch (dtype_in) {
    case MMA_F16:
    case MMA_BF16: {
      const bool bf16 = dtype_in == MMA_BF16;
      const bool out16 = dtype_acc != MMA_F32;
      // 16 x 16 x 16 FP32-accumulate tiles stored densely: the HBM-streaming
      // kernel; every other shape: the tcgen05 kernel over 3-D tensor maps
      if (!out16 && M == 16 && N == 16 && K == 16 && lda == 16 && ldb == 16 &&
          ldd == 16 && (C == nullptr || ldc == 16))
        return launch_batched16(ctx, bf16, batch, G, abid, blgp, A, B,
                                static_cast<const float*>(C),
                                static_cast<float*>(D));
      // mid-size dense blocks in multiples of 64: CTA-cooperative tiles
      if (batched_tile_fits(M, N, K, lda, ldb, ldc, ldd, C != nullptr))
        return launch_batched_tile(ctx, bf16, out16, M, N, K, A, B, C, D,
                                   batch, G, abid, blgp);
      // small and mid-size dense blocks: warp-level MMAs streaming from HBM
      if (batched_mma_fits(M, N, K, lda, ldb, ldc, ldd, C != nullptr, false))
        return launch_batched_mma(ctx, bf16, out16, M, N, K, A, B, C, D, batch,
                                  G, abid, blgp);
      return launch_gemm_tc_batched(ctx, bf16, out16, M, N, K, A, lda, B, ldb,
                                    C, ldc, D, ldd, batch, G, abid, blgp);
    }
    case MMA_I8:
      // small and mid-size dense blocks: integer warp-level MMAs, exact
      if (batched_mma_fits(M, N, K, lda, ldb, ldc, ldd, C != nullptr, true))
        return launch_batched_i8_mma(ctx, M, N, K, A, B, C, D, batch, G, abid,
                                     blgp);
      return with_workspace(
          ctx, gemm_i8_tc_batched_workspace_bytes(M, N, K, batch),
          [&](void* ws) {
            return launch_gemm_i8_tc_batched(
                ctx, M, N, K, static_cast<const int8_t*>(A), lda,
                static_cast<const int8_t*>(B), ldb,
                static_cast<const int32_t*>(C), ldc, static_cast<int32_t*>(D),
                ldd, batch, G, abid, blgp, ws);
          });
    case MMA_F64:
      return launch_gemm_f64_batched(ctx, M, N, K,
                                     static_cast<const double*>(A), lda,
                                     static_cast<const double*>(B), ldb,
                                     static_cast<const double*>(C), ldc,
                                     static_cast<double*>(D), ldd, batch, G,
                                     abid, blgp);
    default:
      return MMA_ERR_UNSUPPORTED;
  }
}

extern "C" mma_status_t mma_gemm_batched(int dtype_in, int dtype_acc,
                                         int64_t M, int64_t N, int64_t K,
                                         const void* A, int64_t lda,
                                         const void* B, int64_t ldb,
                                         const void* C, int64_t ldc, void* D,
                                         int64_t ldd, int64_t batch,
                                         int a_broadcast_group,
                                         int a_broadcast_id, void* stream) {
  return mma_gemm_batched_ex(dtype_in, dtype_acc, M, N, K, A, lda, B, ldb, C,
                             ldc, D, ldd, batch, a_broadcast_group,
                             a_broadcast_id, 0, stream);
}

extern "C" mma_status_t mma_device_status(void* stream) {
  int dev = -1;
  const DeviceInfo* info = device_info(&dev);
  if (!info) return MMA_ERR_NO_DEVICE;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MMA_ERR_LAUNCH;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_mma_status, sizeof(v)) != cudaSuccess)
    return MMA_ERR_LAUNCH;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_mma_status, &zero, sizeof(zero)) != cudaSuccess)
      return MMA_ERR_LAUNCH;
    return MMA_ERR_TIMEOUT;
  }
  return MMA_OK;
}

extern "C" mma_status_t mma_profile_begin(void) {
  int dev = -1;
  const DeviceInfo* info = device_info(&dev);
  if (!info) return MMA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof.created && g_prof.device != dev) return MMA_ERR_INVALID_ARG;
  if (g_prof.created && g_prof.gen != info->gen) {
    // the events belonged to a context that has since been replaced
    g_prof.created = false;
  }
  if (!g_prof.created) {
    for (int i = 0; i < 2 * kProfMax; ++i) {
      if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaEventDestroy(g_prof.ev[j]);
        cudaGetLastError();
        return MMA_ERR_LAUNCH;
      }
    }
    g_prof.created = true;
    g_prof.device = dev;
    g_prof.gen = info->gen;
  }
  g_prof.active = true;
  g_prof.count = 0;
  return MMA_OK;
}

extern "C" mma_status_t mma_profile_end(float* ms, int max_count,
                                        int* count) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof.active) return MMA_ERR_INVALID_ARG;
  g_prof.active = false;
  const int n = g_prof.count < max_count ? g_prof.count : max_count;
  if (count) *count = g_prof.count;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms[i], g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) !=
            cudaSuccess) {
      cudaGetLastError();
      return MMA_ERR_LAUNCH;
    }
  }
  return MMA_OK;
}

extern "C" const char* mma_status_string(int status) {
  switch (status) {
    case MMA_OK: return "MMA_OK";
    case MMA_ERR_INVALID_ARG: return "MMA_ERR_INVALID_ARG";
    case MMA_ERR_UNSUPPORTED: return "MMA_ERR_UNSUPPORTED";
    case MMA_ERR_MISALIGNED: return "MMA_ERR_MISALIGNED";
    case MMA_ERR_LAUNCH: return "MMA_ERR_LAUNCH";
    case MMA_ERR_TIMEOUT: return "MMA_ERR_TIMEOUT";
    case MMA_ERR_NO_DEVICE: return "MMA_ERR_NO_DEVICE";
    case MMA_ERR_NO_MEMORY: return "MMA_ERR_NO_MEMORY";
    default: return "MMA_ERR_UNKNOWN";
  }
}

extern "C" int mma_version(void) { return 200; }
