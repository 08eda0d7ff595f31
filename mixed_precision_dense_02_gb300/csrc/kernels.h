// Internal launcher interface between the C ABI (api.cu) and the kernels.
// Arguments arrive here already validated (sizes, pointers, alignment).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mma_gb300.h"

namespace mmagb {

constexpr int kMaxDevices = 64;

struct Ctx {
  cudaStream_t stream;
  int device;
  int num_sms;
  unsigned* status;  // device status word (bounded-wait timeouts)
  // Identifier of the device's current CUDA context (unique within the
  // process, never 0): state cached for one context (kernel attributes,
  // symbol addresses, buffers) is set up again when it changes, e.g. after
  // cudaDeviceReset.
  uint64_t gen = 0;
  // When profiling is active: events recorded on `stream` immediately
  // before and after the call's dominant (contraction) kernel; else null.
  cudaEvent_t prof_start = nullptr;
  cudaEvent_t prof_stop = nullptr;

  void mark_start() const {
    if (prof_start) cudaEventRecord(prof_start, stream);
  }
  void mark_stop() const {
    if (prof_stop) cudaEventRecord(prof_stop, stream);
  }
};

// TMA tensor maps (gemm_tc.cu).  K-major operand: `count` tiles of `rows`
// rows of K contiguous 16-bit elements (leading dimension ld_elems, tile t
// rows * ld_elems elements after tile t - 1), box 64 x box_rows x 1,
// 128-byte swizzle, zero fill out of bounds.  Row-major C/D: `count` M x N
// tiles, box 64 bytes x 32 rows x 1, 64-byte swizzle.
bool make_kmajor_map(CUtensorMap* map, const void* base, int64_t K,
                     int64_t rows, int64_t ld_elems, int box_rows, bool bf16,
                     int64_t count = 1);
bool make_cd_map(CUtensorMap* map, const void* base, int64_t N, int64_t M,
                 int64_t ld_elems, CUtensorMapDataType dt, int elem_bytes,
                 int64_t count = 1);

// tcgen05 GEMM, FP16/BF16 inputs, column-major B; C and D are FP32, or
// with out16 of the input's 16-bit type (FP32 accumulation, one rounding).
mma_status_t launch_gemm_tc_f16(const Ctx& ctx, bool bf16, bool out16,
                                int64_t M, int64_t N, int64_t K, const void* A,
                                int64_t lda, const void* B, int64_t ldb,
                                const void* C, int64_t ldc, void* D,
                                int64_t ldd);

// Stream-K tcgen05 GEMM (gemm_sk.cu) for FP16/BF16 -> FP32 products with
// fewer 128 x 128 output tiles than SMs: the tiles' K steps are split
// evenly over all SMs, partial tiles meet in `partials`
// (gemm_sk_workspace_bytes) behind per-warp release flags (`flags`,
// gemm_sk_flag_count entries, each last written with an earlier sequence
// number, 0 at allocation); `seq` is this call's nonzero sequence number.
bool gemm_sk_fits(int num_sms, int64_t M, int64_t N, int64_t K);
size_t gemm_sk_workspace_bytes(int num_sms);
size_t gemm_sk_flag_count(int num_sms);
mma_status_t launch_gemm_sk(const Ctx& ctx, bool bf16, int64_t M, int64_t N,
                            int64_t K, const void* A, int64_t lda,
                            const void* B, int64_t ldb, const float* C,
                            int64_t ldc, float* D, int64_t ldd,
                            float* partials, unsigned* flags, unsigned seq);

// Exact 8-bit integer GEMM on the tcgen05 BF16 pipe.  `workspace` holds
// gemm_i8_tc_workspace_bytes(M, N, K) bytes of device scratch for the BF16
// copies of A and B (B is transposed into it when b_row_major).  A and B
// hold int8 (a_signed / b_signed) or uint8 values; D wraps modulo 2^32, or
// with `clamp` is the exact result saturated to the INT32 range.
size_t gemm_i8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K);
mma_status_t launch_gemm_i8_tc(const Ctx& ctx, int64_t M, int64_t N,
                               int64_t K, const int8_t* A, int64_t lda,
                               const int8_t* B, int64_t ldb, const int32_t* C,
                               int64_t ldc, int32_t* D, int64_t ldd,
                               void* workspace, bool b_row_major,
                               bool a_signed, bool b_signed, bool clamp);

// Batched tcgen05 GEMMs: `batch` entries of contiguous M x N x K tiles
// (tile b of A at A + b*M*lda, of B at B + b*N*ldb, of C/D at b*M*ldc,
// b*M*ldd elements); entry b reads A tile (b/group)*group + abid and the B
// tile of lane-group pattern blgp (0..7; batch % 4 == 0 when nonzero).
mma_status_t launch_gemm_tc_batched(const Ctx& ctx, bool bf16, bool out16,
                                    int64_t M, int64_t N, int64_t K,
                                    const void* A, int64_t lda, const void* B,
                                    int64_t ldb, const void* C, int64_t ldc,
                                    void* D, int64_t ldd, int64_t batch,
                                    int group, int abid, int blgp);
// INT8 -> INT32 (exact), through BF16 copies of every tile in `workspace`.
size_t gemm_i8_tc_batched_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                          int64_t batch);
mma_status_t launch_gemm_i8_tc_batched(const Ctx& ctx, int64_t M, int64_t N,
                                       int64_t K, const int8_t* A, int64_t lda,
                                       const int8_t* B, int64_t ldb,
                                       const int32_t* C, int64_t ldc,
                                       int32_t* D, int64_t ldd, int64_t batch,
                                       int group, int abid, int blgp,
                                       void* workspace);

// Batched FP16/BF16 blocks streamed from HBM by warp-level MMAs (small and
// mid-size blocks; see batched_mma_fits), FP32 or 16-bit C and D.
bool batched_mma_fits(int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int64_t ldc, int64_t ldd, bool has_c,
                      bool i8);
mma_status_t launch_batched_mma(const Ctx& ctx, bool bf16, bool out16,
                                int64_t M, int64_t N, int64_t K, const void* A,
                                const void* B, const void* C, void* D,
                                int64_t batch, int group, int abid, int blgp);
// Batched FP16/BF16 blocks with M, N, K multiples of 64 (see
// batched_tile_fits): CTAs of four warps, operands staged once per CTA tile
// through a cp.async ring.
bool batched_tile_fits(int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldc, int64_t ldd, bool has_c);
mma_status_t launch_batched_tile(const Ctx& ctx, bool bf16, bool out16,
                                 int64_t M, int64_t N, int64_t K,
                                 const void* A, const void* B, const void* C,
                                 void* D, int64_t batch, int group, int abid,
                                 int blgp);
// The same for INT8 -> INT32 (exact), with integer warp-level MMAs.
mma_status_t launch_batched_i8_mma(const Ctx& ctx, int64_t M, int64_t N,
                                   int64_t K, const void* A, const void* B,
                                   const void* C, void* D, int64_t batch,
                                   int group, int abid, int blgp);

// Batched FP64 (DMMA), same tile conventions.
mma_status_t launch_gemm_f64_batched(const Ctx& ctx, int64_t M, int64_t N,
                                     int64_t K, const double* A, int64_t lda,
                                     const double* B, int64_t ldb,
                                     const double* C, int64_t ldc, double* D,
                                     int64_t ldd, int64_t batch, int group,
                                     int abid, int blgp);

// tcgen05 FP16/BF16 GEMM with row-major B: B is transposed into
// `workspace` (gemm_tc_rowb_workspace_bytes(N, K) bytes) first.
size_t gemm_tc_rowb_workspace_bytes(int64_t N, int64_t K);
mma_status_t launch_gemm_tc_f16_rowb(const Ctx& ctx, bool bf16, bool out16,
                                     int64_t M, int64_t N, int64_t K,
                                     const void* A, int64_t lda, const void* B,
                                     int64_t ldb, const void* C, int64_t ldc,
                                     void* D, int64_t ldd, void* workspace);

// INT8 GEMM on the warp-level IMMA pipe, column-major B.
mma_status_t launch_gemm_i8_imma(const Ctx& ctx, int64_t M, int64_t N,
                                 int64_t K, const int8_t* A, int64_t lda,
                                 const int8_t* B, int64_t ldb,
                                 const int32_t* C, int64_t ldc, int32_t* D,
                                 int64_t ldd);

// FP64 GEMM (DMMA), B column- or row-major.
mma_status_t launch_gemm_f64(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                             const double* A, int64_t lda, const double* B,
                             int64_t ldb, bool b_row_major, const double* C,
                             int64_t ldc, double* D, int64_t ldd);

// Batched 16x16x16 FP16/BF16 -> FP32 with A-block broadcast.
mma_status_t launch_batched16(const Ctx& ctx, bool bf16, int64_t batch,
                              int group, int abid, int blgp, const void* A,
                              const void* B, const float* C, float* D);

// Failure-detection self-test of the tcgen05 GEMM itself: a 256 x 256 x
// 256 BF16 product on single CTAs (cluster 1) or a CTA pair (cluster 2)
// whose producer issues no loads and whose bounded waits give up after
// limit_ns, so the real abort path runs (A, B, D: caller buffers of that
// size, never read or written).
mma_status_t launch_gemm_tc_abort_selftest(const Ctx& ctx, int cluster,
                                           int64_t limit_ns, const void* A,
                                           const void* B, void* D);

// Launch context for the current device (false if it is not a usable
// sm_103 device).
bool current_ctx(void* stream, Ctx* out);

// Attach the next profiling event pair (if profiling is active) to a launch
// context.
void attach_profile(Ctx& ctx);

// A value set up once per device context (a kernel attribute, an occupancy
// figure, a symbol address): `compute(&value)` runs on the first use in a
// context, under a lock, so concurrent first calls from several host
// threads neither race nor repeat it, and runs again when the device's
// context has been replaced.  Returns false, and caches nothing, when
// compute fails.
template <class T>
class PerContext {
 public:
  template <class F>
  bool get(const Ctx& ctx, T* out, F&& compute) {
    if (ctx.device < 0 || ctx.device >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(mu_);
    Slot& s = slot_[ctx.device];
    if (s.gen != ctx.gen) {
      T v{};
      if (!compute(&v)) return false;
      s.value = v;
      s.gen = ctx.gen;
    }
    *out = s.value;
    return true;
  }

 private:
  struct Slot {
    uint64_t gen = 0;
    T value{};
  };
  std::mutex mu_;
  Slot slot_[kMaxDevices];
};

// K == 0: D = C (or 0), elementwise, element size 2, 4 or 8 bytes.
mma_status_t launch_copy_c(const Ctx& ctx, int64_t M, int64_t N,
                           int elem_bytes, const void* C, int64_t ldc, void* D,
                           int64_t ldd);

}  // namespace mmagb
