/*
 * mma_gb300.h -- C ABI of the GB300 (sm_103a) dense multiply-accumulate
 * library  D = A * B + C.
 *
 * Operation (page "CDNA2 dense MFMA builtins", section "Naming convention"):
 * one matrix instruction adds the contribution of an M x K panel of A and a
 * K x N panel of B to an M x N output tile, and the caller loops over K to
 * accumulate the full product.  Each call here performs that whole K loop:
 *
 *     D[i][j] = C[i][j] + sum_{k < K} A[i][k] * B[k][j]
 *
 * with the input/accumulator pairs of the pages' builtin lists ("CDNA2 dense
 * MFMA builtins", section "Builtin reference"; "RDNA3 dense WMMA builtins",
 * section "Builtin reference", which defines every builtin's result as
 * srcA x srcB + srcC):
 *
 *     dtype_in  dtype_acc   A, B element     C, D element
 *     MMA_F16   MMA_F32     IEEE binary16    float
 *     MMA_BF16  MMA_F32     bfloat16 bits    float
 *     MMA_F16   MMA_F16     IEEE binary16    IEEE binary16  (16-bit accumulate)
 *     MMA_BF16  MMA_BF16    bfloat16 bits    bfloat16 bits  (16-bit accumulate)
 *     MMA_I8    MMA_I32     signed int8      int32_t  (exact; wraps mod 2^32)
 *     MMA_F64   MMA_F64     double           double
 *
 * The 16-bit-accumulate pairs ("RDNA3 dense WMMA builtins", section
 * "Builtin reference", FP16/BF16-accumulate builtins) accumulate in FP32
 * inside and round A*B + C once to the 16-bit format (nearest, ties to
 * even); the builtins round their 16-bit accumulator after every K step.
 *
 * Any other pair returns MMA_ERR_UNSUPPORTED.
 *
 * Layouts (elements, not bytes; "RDNA3 dense WMMA builtins", section
 * "Using WMMA builtins as a compute policy": A rows and B columns are read
 * K-contiguous, the output is written row-major):
 *   A  M x K row-major:     A[i][k] at A[i*lda + k],  lda >= K
 *   B  column-major:        B[k][j] at B[j*ldb + k],  ldb >= K   (mma_gemm)
 *      or row-major:        B[k][j] at B[k*ldb + j],  ldb >= N   (mma_gemm_ex)
 *   C, D  M x N row-major:  C[i][j] at C[i*ldc + j],  ldc, ldd >= N
 *
 * Pointers and ownership: A, B, C and D are device pointers owned by the
 * caller; the library keeps no reference to them after the call returns.
 * C may be NULL (read as zero).  C may equal D (in place) only when
 * ldc == ldd; any other overlap between D and an input is undefined.
 *
 * Device memory owned by the library: some paths first rewrite an operand
 * into a scratch buffer -- INT8 products with M*N*K >= 2^24 (and every INT8
 * product with row-major B, and every mma_gemm_i8_ex product other than
 * signed x signed without clamp) widen A and B to BF16 for the tensor pipe,
 * (M + N) * roundup(K, 8) * 2 bytes, plus (M + N) * 8 bytes of correction
 * terms; batched INT8 products widen every tile, batch * (M + N) *
 * roundup(K, 8) * 2 bytes; FP16/BF16 products with row-major B transpose
 * B, N * roundup(K, 8) * 2 bytes; FP16/BF16 -> FP32 products with
 * column-major B, fewer than half as many 128 x 128 output tiles as SMs
 * and deep enough K (at least eight 64-deep K steps per tile, and either at
 * most a quarter as many tiles as SMs or at least 128 steps) split K over
 * the SMs and meet in it, SMs * 128 KiB, plus a hand-off flag buffer of
 * SMs * 32 bytes allocated (and zeroed) once per device.  That buffer is allocated once
 * per device by the first such call, grown (cudaMalloc, after the previous
 * user finishes) only when a larger problem arrives, and kept until the
 * process exits; calls on different streams are ordered on it by an event.
 * Failure to grow it returns MMA_ERR_NO_MEMORY.  No other call allocates.
 *
 * Alignment: every non-NULL base pointer must be 16-byte aligned and every
 * leading dimension times the element size must be a multiple of 16 bytes
 * (the tensor-memory-access engine's rule); otherwise MMA_ERR_MISALIGNED.
 * M, N and K themselves are arbitrary (>= 0): ragged edges are handled
 * inside the kernels.  M == 0 or N == 0 is a no-op; K == 0 gives D = C.
 *
 * Streams and errors: `stream` is a cudaStream_t (NULL = the legacy default
 * stream).  Work is enqueued on it and the call returns without
 * synchronising.  Argument errors are detected before anything is launched
 * and reported by the return value; a failed launch returns MMA_ERR_LAUNCH.
 * No C++ exception crosses this interface.  Every pipeline wait inside the
 * kernels is bounded; a wait that runs out records MMA_ERR_TIMEOUT in a
 * device-side status word that mma_device_status() reads back.  Calls on
 * different streams may run concurrently; the library holds no per-call
 * state.
 */
#ifndef MMA_GB300_H
#define MMA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MMA_F16 = 1,
  MMA_BF16 = 2,
  MMA_I8 = 3,
  MMA_F64 = 4,
  MMA_F32 = 5,
  MMA_I32 = 6
} mma_dtype_t;

typedef enum { MMA_COL_MAJOR = 0, MMA_ROW_MAJOR = 1 } mma_layout_t;

typedef enum {
  MMA_OK = 0,
  MMA_ERR_INVALID_ARG = 1, /* negative size, short leading dimension, NULL
                              operand, bad broadcast group/id            */
  MMA_ERR_UNSUPPORTED = 2, /* dtype pair or batched shape not provided    */
  MMA_ERR_MISALIGNED = 3,  /* pointer or leading dimension not 16 B       */
  MMA_ERR_LAUNCH = 4,      /* CUDA reported an error at launch            */
  MMA_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait ran out            */
  MMA_ERR_NO_DEVICE = 6,   /* no usable sm_103 device is current          */
  MMA_ERR_NO_MEMORY = 7    /* the scratch buffer could not be grown       */
} mma_status_t;

/*
 * mma_gemm -- D = A * B + C with column-major B.
 *
 * Passage: "CDNA2 dense MFMA builtins", sections "Naming convention" (the
 * K-loop contract) and "Builtin reference" (FP16/BF16 -> FP32, INT8 ->
 * INT32, FP64 -> FP64 with round-to-nearest-even); "RDNA3 dense WMMA
 * builtins", section "Builtin reference" (srcA x srcB + srcC; signed int8).
 *
 * dtype_in, dtype_acc : one of the pairs in the table above.
 * M, N, K             : problem size, each >= 0.
 * A, lda              : M x K row-major input, lda >= K.
 * B, ldb              : K x N column-major input (stored as N rows of K
 *                       contiguous elements), ldb >= K.
 * C, ldc              : M x N row-major addend of type dtype_acc, or NULL.
 * D, ldd              : M x N row-major output of type dtype_acc.
 * stream              : cudaStream_t to enqueue on.
 * Returns MMA_OK or an error code; see the header comment for each case.
 */
mma_status_t mma_gemm(int dtype_in, int dtype_acc, int64_t M, int64_t N,
                      int64_t K, const void *A, int64_t lda, const void *B,
                      int64_t ldb, const void *C, int64_t ldc, void *D,
                      int64_t ldd, void *stream);

/*
 * mma_gemm_ex -- as mma_gemm, with the layout of B chosen by `layout_b`:
 * MMA_COL_MAJOR (same as mma_gemm) or MMA_ROW_MAJOR (B[k][j] at
 * B[k*ldb + j], ldb >= N).  Same passages as mma_gemm; the row-major form
 * is the plain storage of a K x N matrix.
 */
mma_status_t mma_gemm_ex(int dtype_in, int dtype_acc, int64_t M, int64_t N,
                         int64_t K, const void *A, int64_t lda, const void *B,
                         int64_t ldb, int layout_b, const void *C, int64_t ldc,
                         void *D, int64_t ldd, void *stream);

/*
 * mma_gemm_i8_ex -- 8-bit integer D = A * B + C with INT32 C and D, each of
 * A and B signed or unsigned, and optional saturation.
 *
 * Passage: "RDNA3 dense WMMA builtins", sections "INT32-accumulate
 * builtins" (integer inputs signed or unsigned, chosen per operand by
 * a_neg and b_neg) and "INT8 and UINT8 inputs" (the iu8 builtin:
 * srcA x srcB + srcC, and `clamp`: saturate the output on overflow).
 *
 * a_neg, b_neg : nonzero -- A (B) holds int8 values in [-128, 127];
 *                zero    -- uint8 values in [0, 255].
 * clamp        : zero    -- D is the exact value modulo 2^32 (wrapping, as
 *                           mma_gemm's INT8 product);
 *                nonzero -- D is the exact value of A*B + C, saturated once
 *                           to [INT32_MIN, INT32_MAX].
 * Other arguments, layouts, alignment rules and status codes are those of
 * mma_gemm_ex with dtype_in = MMA_I8, dtype_acc = MMA_I32 (A, B: 1-byte
 * elements; layout_b MMA_COL_MAJOR or MMA_ROW_MAJOR).  Signed x signed
 * without clamp is exactly mma_gemm_ex; every other combination runs on the
 * tensor pipe and grows the library's scratch buffer like it
 * ((M + N) * roundup(K, 8) * 2 bytes; MMA_ERR_NO_MEMORY if it cannot).
 */
mma_status_t mma_gemm_i8_ex(int64_t M, int64_t N, int64_t K, const void *A,
                            int64_t lda, int a_neg, const void *B, int64_t ldb,
                            int b_neg, int layout_b, const void *C,
                            int64_t ldc, void *D, int64_t ldd, int clamp,
                            void *stream);

/*
 * mma_gemm_batched -- `batch` independent M x N x K products with A-block
 * broadcast:
 *
 *     for b in [0, batch):  D_b = A_{src(b)} * B_b + C_b,
 *                           src(b) = (b / G) * G + a_broadcast_id
 *
 * Passage: "Common MFMA parameters", section "Shared parameters" (cbsz:
 * one chosen input block of A is broadcast to the 2^cbsz - 1 neighbouring
 * blocks of its group; abid: which block of each group is the source;
 * worked example cbsz = 2, abid = 1: block 1's A goes to blocks 0, 2, 3 and
 * block 5's to 4, 6, 7), and "CDNA2 dense MFMA builtins", section
 * "Accumulator layout" (one instruction computes several independent
 * blocks, each with its own A, B, C and D).  Here a batch entry plays the
 * role of a block and G = a_broadcast_group = 2^cbsz.
 *
 * Storage: tiles are contiguous, tile b of A at A + b*M*lda, of B at
 * B + b*N*ldb (column-major tiles), of C and D at b*M*ldc and b*M*ldd
 * (elements).  A holds `batch` tiles; only tile src(b) is read for entry b.
 * B, C and D are never broadcast here (see mma_gemm_batched_ex for B).
 * Pairs: the four of mma_gemm plus 16-bit accumulate; any M, N, K >= 0;
 * leading dimensions and alignment as for mma_gemm (each tile is one
 * mma_gemm problem).  The kernel follows the block shape (dense tiles,
 * leading dimensions equal to the tile's row length):
 *   - 16 x 16 x 16 FP16/BF16 -> FP32: an HBM-streaming kernel;
 *   - FP16/BF16 with M, N, K multiples of 64 and M*N*K <= 2^20: a
 *     CTA-cooperative kernel (64 x 64 tiles, operands staged once in shared
 *     memory);
 *   - FP16/BF16 with M, N, K multiples of 16 and M*N*K <= 96*96*64, and
 *     INT8 with M, N, K multiples of 16 and M*N*K <= 128^3: warp-level
 *     streaming kernels;
 *   - everything else: the tensor-memory GEMM over per-entry tensor maps
 *     (INT8: through BF16 copies of every tile in the library's scratch
 *     buffer, grown like mma_gemm's); FP64: DMMA tiles.
 * The choice changes speed only: FP16/BF16 results agree within the
 * accumulation tolerance (the routes sum in different orders), and INT8
 * results are bit-identical across routes.
 * Constraints: a_broadcast_group in {1, 2, 4, 8, 16}; 0 <= a_broadcast_id
 * < a_broadcast_group; batch % a_broadcast_group == 0 (else
 * MMA_ERR_INVALID_ARG); batch < 2^31 (else MMA_ERR_UNSUPPORTED).
 */
mma_status_t mma_gemm_batched(int dtype_in, int dtype_acc, int64_t M,
                              int64_t N, int64_t K, const void *A, int64_t lda,
                              const void *B, int64_t ldb, const void *C,
                              int64_t ldc, void *D, int64_t ldd, int64_t batch,
                              int a_broadcast_group, int a_broadcast_id,
                              void *stream);

/*
 * mma_gemm_batched_ex -- mma_gemm_batched with a B-group pattern as well:
 *
 *     D_b = A_{src(b)} * B_{bsrc(b)} + C_b,
 *     bsrc(b) = (b / 4) * 4 + P[b_lane_group_pattern][b % 4]
 *
 * Passage: "Common MFMA parameters", section "Dense MFMA parameters"
 * (blgp: a constrained swizzle of B between the lanes of the 64-lane
 * operand).  Read at matrix level: consecutive groups of four batch entries
 * play the four 16-lane quarters, and P[p][q] is the quarter whose B the
 * entry at quarter q reads:
 *   p = 0  q            (no swizzling)
 *   p = 1  q & 1        (lanes 0-31 broadcast into lanes 32-63)
 *   p = 2  2 + (q & 1)  (lanes 32-63 broadcast into lanes 0-31)
 *   p = 3  (q + 1) % 4  (all lanes rotated down by 16)
 *   p = 4..7  p - 4     (one quarter broadcast into the other three)
 * b_lane_group_pattern in 0..7, and batch % 4 == 0 when it is nonzero (else
 * MMA_ERR_INVALID_ARG).  Everything else is as for mma_gemm_batched, which
 * is this call with b_lane_group_pattern = 0.
 */
mma_status_t mma_gemm_batched_ex(int dtype_in, int dtype_acc, int64_t M,
                                 int64_t N, int64_t K, const void *A,
                                 int64_t lda, const void *B, int64_t ldb,
                                 const void *C, int64_t ldc, void *D,
                                 int64_t ldd, int64_t batch,
                                 int a_broadcast_group, int a_broadcast_id,
                                 int b_lane_group_pattern, void *stream);

/*
 * mma_device_status -- synchronise `stream`, then read and clear the
 * library's device-side status word on the current device.  Returns MMA_OK
 * when no in-kernel wait has run out since the last call, MMA_ERR_TIMEOUT
 * otherwise, or MMA_ERR_LAUNCH if the synchronisation itself failed.
 * (The pages check errors after every launch: "RDNA3 dense WMMA builtins",
 * section "Instantiating the kernel"; this is the matching device-side
 * check.)
 */
mma_status_t mma_device_status(void *stream);

/*
 * mma_selftest_wait_timeout -- exercise the failure-detection path of the
 * kernels without faulting or hanging the GPU.  The pages have no
 * counterpart; it backs mma_device_status's contract with a test.
 *
 * Every pipeline wait inside the kernels is bounded: when one runs out, the
 * kernel records MMA_ERR_TIMEOUT in the device status word, drains and
 * returns.  This call enqueues on `stream` one tiny kernel that performs
 * that same bounded wait on a barrier that nothing ever signals, with the
 * limit `limit_ns` (1000 .. 10^10 nanoseconds), so the wait runs out after
 * about limit_ns and the kernel returns.  A following mma_device_status
 * (stream) then returns MMA_ERR_TIMEOUT once and clears the word; the
 * context stays usable.  Returns MMA_ERR_INVALID_ARG for a limit out of
 * range, MMA_ERR_NO_DEVICE without a device, else MMA_OK.
 */
mma_status_t mma_selftest_wait_timeout(int64_t limit_ns, void *stream);

/*
 * mma_selftest_gemm_abort -- exercise the tcgen05 GEMM kernel's own abort
 * path without faulting or hanging the GPU.  The pages have no counterpart;
 * it backs the bounded-wait contract of the GEMM kernels with a test.
 *
 * Enqueues on `stream` the BF16 -> FP32 GEMM kernel for a 256 x 256 x 256
 * product on single CTAs (cluster = 1) or on a CTA pair sharing one MMA
 * (cluster = 2), with its operand producer told to issue no loads and every
 * pipeline wait limited to limit_ns (10^6 .. 10^10 ns).  The MMA issuer's
 * first stage wait therefore runs out with nothing in flight; the kernel
 * raises its abort flag, records MMA_ERR_TIMEOUT in the device status word,
 * drains, frees its tensor memory and exits, so the context stays usable.
 * A and B (256 x 256 BF16) and D (256 x 256 FP32) are caller device
 * buffers, 16-byte aligned; nothing reads or writes them.  Returns
 * MMA_ERR_INVALID_ARG (bad cluster, limit or NULL buffer),
 * MMA_ERR_MISALIGNED, MMA_ERR_NO_DEVICE or the launch status; a following
 * mma_device_status(stream) returns MMA_ERR_TIMEOUT once.
 */
mma_status_t mma_selftest_gemm_abort(int cluster, int64_t limit_ns,
                                     const void *A, const void *B, void *D,
                                     void *stream);

/*
 * mma_peak_probe -- enqueue one issue-rate probe of a compute pipe on every
 * SM of the current device and report the operations it performs.
 *
 * Passage: "CDNA2 dense MFMA builtins", section "Instruction throughput":
 * peak throughput = operations per instruction / cycles per instruction x
 * clock.  The probe measures that rate instead of deriving it: every SM
 * issues `iterations` rounds of independent back-to-back instructions of
 * one kind on register or shared-memory operands (no DRAM traffic), so
 * *ops_per_launch (written before the launch) divided by the launch's
 * duration (CUDA events around the call, on `stream`) is the pipe's rate
 * at the clock the launch ran at.  Kinds:
 *   MMA_PEAK_TC_F16  tcgen05.mma kind::f16, BF16 in, FP32 accumulate
 *                    (M = 128, N = 256, K = 16; the FP16/BF16 and exact
 *                    INT8 GEMMs' pipe); iterations <= 2^21
 *   MMA_PEAK_DMMA    mma.sync m8n8k4 FP64 (the FP64 GEMM's instruction)
 *   MMA_PEAK_IMMA    mma.sync m16n8k32 int8 -> int32 (small INT8 products)
 *   MMA_PEAK_DFMA    scalar FP64 fused multiply-add
 * One operation is one multiply or one add (a multiply-add counts 2).
 * Returns MMA_ERR_INVALID_ARG for an unknown kind, iterations < 1 or above
 * the kind's limit (2^40 for the warp-level kinds), or a NULL
 * ops_per_launch; MMA_ERR_NO_DEVICE without a device; else the launch
 * status.  Recorded by mma_profile_begin like the GEMM calls.
 */
typedef enum {
  MMA_PEAK_TC_F16 = 1,
  MMA_PEAK_DMMA = 2,
  MMA_PEAK_IMMA = 3,
  MMA_PEAK_DFMA = 4
} mma_peak_kind_t;
mma_status_t mma_peak_probe(int kind, int64_t iterations,
                            double *ops_per_launch, void *stream);

/*
 * mma_profile_begin / mma_profile_end -- per-launch timing of the dominant
 * kernel (the contraction kernel of each mma_gemm* call), for measuring it
 * against its roofline.  The pages time each kernel launch after warm-up
 * runs ("RDNA3 dense WMMA builtins", section "Instantiating the kernel");
 * this is the device-side counterpart.
 *
 * mma_profile_begin: start recording, on the current device, one CUDA event
 * pair on the caller's stream immediately around the dominant kernel of
 * each subsequent call (at most 4096 calls; later calls are not recorded).
 * The event pool is created on the first begin (never per call).  Returns
 * MMA_ERR_NO_DEVICE without a device, MMA_ERR_INVALID_ARG if the pool
 * belongs to another device.
 *
 * mma_profile_end: stop recording, wait for the recorded events, write the
 * durations in milliseconds of the first min(count, max_count) recorded
 * launches to ms[] (host array owned by the caller) and the number recorded
 * to *count.  Returns MMA_ERR_INVALID_ARG if profiling was not active.
 * Not thread-safe with concurrent calls on other threads.
 */
mma_status_t mma_profile_begin(void);
mma_status_t mma_profile_end(float *ms, int max_count, int *count);

/*
 * mma_gemm_i8_noalloc -- the exact INT8 -> INT32 product of mma_gemm
 * (column-major B, same layouts, alignment, C handling and status codes),
 * computed on the tensor pipe without allocating any device memory.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot let a library allocate device memory.  mma_gemm grows a scratch
 * buffer with cudaMalloc for large INT8 problems; a program whose pool
 * allocator has already reserved the memory it may use, or a service that
 * forbids allocation after start-up (cudaMalloc/cudaFree can block and
 * synchronise the device), calls this instead.  Its scratch is a fixed
 * array of MMA_NOALLOC_SCRATCH_BYTES in the library's device image, held by
 * every GPU that loads the library until the process exits.
 *
 * Limit: (M + N) * roundup(K, 8) * 2 bytes must fit in
 * MMA_NOALLOC_SCRATCH_BYTES (for example M = N = K = 4096); larger problems
 * return MMA_ERR_UNSUPPORTED and launch nothing.
 * Set-up: the first call on each device, made with that device current,
 * looks up the array's device address (cudaGetSymbolAddress) and caches it
 * for the device's current context (after cudaDeviceReset the next call
 * looks it up again); make that first call before any stream capture
 * begins.  Status codes and profiling (mma_profile_begin) as for mma_gemm.
 * Sharing: all calls on a device use the same array and leave their data in
 * it (nothing there needs to start at zero); calls whose work overlaps on
 * the GPU race on it, so order calls issued on different streams.
 */
#define MMA_NOALLOC_SCRATCH_BYTES (64u << 20)
mma_status_t mma_gemm_i8_noalloc(int64_t M, int64_t N, int64_t K,
                                 const void *A, int64_t lda, const void *B,
                                 int64_t ldb, const void *C, int64_t ldc,
                                 void *D, int64_t ldd, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *mma_status_string(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int mma_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MMA_GB300_H */
