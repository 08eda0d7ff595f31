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
//   * persistent CTAs (one per SM, or CTA pairs sharing one 256-row MMA
//     tile through cta_group::2), tiles visited in M-grouped order so the
//     A and B panels in flight stay resident in L2;
//   * warp 0 drives TMA: 128x64 A and BNx64 B boxes (a pair's CTAs each
//     load half of B), 128-byte swizzled, into a STAGES-deep shared-memory
//     ring guarded by mbarriers;
//   * warp 1 issues tcgen05.mma (M=128 or 256, N=BN, K=16) from one thread
//     into a double-buffered FP32 accumulator in tensor memory;
//   * warps 2..9 (two per tensor-memory lane quarter, one per column half)
//     drain the accumulator with tcgen05.ld and emit 32-row x 16-column
//     blocks through a small per-warp staging ring: C arrives by TMA load,
//     D leaves by TMA store, overlapping the next tile's MMAs.
// The same kernel carries the exact INT8 -> INT32 product on the BF16
// tensor pipe (sm_103a has no integer kind of tcgen05.mma): int8 operands
// are widened to BF16 (exact), K is split into chunks short enough that
// every FP32 partial sum is an exactly representable integer, and the
// epilogue sums the chunks in INT32 registers (see Epi::I32EXACT; C joins
// those sums while the chunks run).
// Ragged M/N/K edges: TMA zero-fills out-of-bounds load boxes (so they add
// nothing to the sum) and clips stores to the tensor's extent.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
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
//   H16      D = acc + C rounded once to the 16-bit input format (FP16 or
//            BF16 addend and result; FP32 accumulation inside)
//   I32SAT   as I32EXACT, but D is the exact value of A*B + C saturated to
//            the INT32 range: the chunk sums are gathered without wrapping
//            (INT32 registers for up to kSatFlush chunks, folded into 64-bit
//            sums held in spare tensor-memory columns every kSatFlush chunks
//            and after the last), and each 64-bit sum plus C is clamped
//            once.  BN = 128 only (the 64-bit sums take the other half of
//            TMEM).
//   I32SATW  as I32SAT, on any tile width, for problems whose correction
//            terms plus chunk sums stay inside the INT32 range (checked on
//            the host; K up to about 32000): the INT32 sums start from the
//            terms like I32EXACT's, never wrap, and each output is widened
//            to 64 bits only to add C and clamp; no TMEM folds.
//   I32SATE  as I32SATW, with C added to the INT32 sums while the chunks
//            run (I32EXACT's early C), for problems whose exact product S
//            lies in [-2^30, 2^30) (checked on the host from K and the
//            operands' signedness).  The register sum then holds S + C
//            modulo 2^32, and with the sign of C (one bit per output, kept
//            as C is added) it fixes the saturated value: for C >= 0,
//            S + C overflowed exactly when the wrapped sum is below -2^30;
//            for C < 0, exactly when it is at least 2^30.  Both ranges are
//            disjoint from the values the sum takes without overflow.
enum class Epi { F32, I32EXACT, H16, I32SAT, I32SATW, I32SATE };

constexpr bool int_mode(Epi e) {
  return e == Epi::I32EXACT || e == Epi::I32SAT || e == Epi::I32SATW ||
         e == Epi::I32SATE;
}

// Chunk depth of the exact 8-bit integer modes: every partial sum must stay
// within 2^24 in magnitude, the range where FP32 represents all integers.
// The stored values lie in [-128, 127] (unsigned inputs are shifted by -128,
// see widen_rows_kernel), so |a*b| <= 2^14 and 1024 products per chunk.
constexpr int kI8ChunkK = 1024;

// I32SAT: 127 chunk sums of magnitude <= 2^24 stay below 2^31, so the INT32
// registers hold them exactly; every kSatFlush chunks they are folded into
// the 64-bit partial sums.
constexpr int kSatFlush = 127;

// Epilogue staging: each epilogue warp owns NSTG 32-row x 16-column blocks
// of 4-byte elements (64-byte rows, 64-byte TMA swizzle), a ring through
// which C arrives and D leaves by TMA.
constexpr int kStgBytes = 32 * 16 * 4;

// CL = 2: each CTA of a pair stages its own half of the B box.
template <int BN, int STAGES, int CL, int NSTG>
struct Layout {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (BN / CL) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STG_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFFSET = STG_OFFSET + kEpiWarps * NSTG * kStgBytes;
  static constexpr int NUM_BARS = 2 * STAGES + 5 + NSTG * kEpiWarps;
  static constexpr int TOTAL = BAR_OFFSET + NUM_BARS * 8 + 16;
  static constexpr int ALLOC = TOTAL + 1024;  // room to align the base
  // two accumulators of BN columns, rounded up to a power of two
  static constexpr uint32_t TMEM_COLS =
      2 * BN <= 256 ? 256u : 512u;
};

// I32SATE: per epilogue warp, one 32-bit word per lane and 32 columns of
// its half tile holding the sign bits of the C elements it added (word w of
// lane l at index w * 32 + l), placed after the barriers.
template <int BN>
constexpr int sign_words() { return (BN / 2 + 31) / 32; }
template <int BN>
constexpr int sign_bytes() { return kEpiWarps * 32 * sign_words<BN>() * 4; }
template <int BN, int STAGES, int CL, int NSTG, Epi EPI>
constexpr int smem_alloc() {
  return Layout<BN, STAGES, CL, NSTG>::ALLOC +
         (EPI == Epi::I32SATE ? sign_bytes<BN>() : 0);
}

// Batched problems: `batch` entries of the same M x N x K shape, each tile
// of A, B, C and D contiguous (the batch entry is the third tensor-map
// coordinate).  Entry b reads the A tile (b / group) * group + abid (the
// cbsz/abid broadcast of "Common MFMA parameters", section "Shared
// parameters", group = 2^cbsz) and the B tile (b / 4) * 4 + blgp_source(q)
// for q = b % 4 (the blgp lane-group patterns of section "Dense MFMA
// parameters", read at matrix level: the four entries of a group play the
// four 16-lane quarters of a 64-lane B operand).  A single problem is
// batch = 1, group = 1, abid = 0, blgp = 0.
struct BatchArgs {
  int batch;
  int group;
  int abid;
  int blgp;
};

// The quarter whose B data quarter q receives under lane-group pattern p:
// 0 none moved; 1 lanes 0-31 copied to 32-63; 2 lanes 32-63 copied to 0-31;
// 3 all lanes rotated down by 16 (lane 16 -> lane 0, lane 0 -> lane 48);
// 4..7 the quarter p - 4 copied to the other three.
__device__ __forceinline__ int blgp_source(int p, int q) {
  if (p == 0) return q;
  if (p == 1) return q & 1;
  if (p == 2) return 2 | (q & 1);
  if (p == 3) return (q + 1) & 3;
  return p - 4;
}

// Failure-detection self-test hook, set only by the library's self-test
// entry point (every GEMM call passes {kWaitLimitNs, 0}): the limit of the
// kernel's bounded waits, and whether the producer issues no operand loads
// at all, so that the MMA issuer's first stage wait runs out with nothing
// in flight and the abort path (flag, drain, tensor-memory release, exit)
// runs for real.
struct TestHook {
  unsigned long long wait_limit_ns;
  int skip_loads;
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

// 16-bit float (bit pattern) <-> FP32, BF16 or FP16; rounding to nearest,
// ties to even.
template <bool BF16>
__device__ __forceinline__ float half_to_f32(uint32_t bits) {
  if constexpr (BF16)
    return __uint_as_float(bits << 16);
  else
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
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

// 320 threads (10 warps, so three share an SM sub-partition's 16K
// registers): at most 168 registers per thread.
//
// CL = 2 runs one MMA over a pair of CTAs (a cluster of two SMs): the
// pair computes a 256 x BN tile with tcgen05.mma.cta_group::2, each CTA
// holding 128 rows of A, half (BN/2 rows) of B and its 128 rows of the
// accumulator.  Per K step each SM stages 128 + BN/2 operand rows instead
// of 128 + BN, which cuts the shared-memory traffic (TMA writes plus MMA
// reads) that bounds the single-CTA kernel.  Both CTAs' loads complete on
// the leader CTA's (rank 0) full barrier; the leader's one MMA thread
// issues the pair's MMAs, whose commits release the stage in both CTAs and
// announce the accumulator to both CTAs' epilogues; every epilogue warp of
// the pair returns the accumulator on the leader's tempty barrier.
template <int BN, int STAGES, bool BF16, Epi EPI, int CL, int NSTG>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmD,
                   const void* __restrict__ Cv, int64_t ldc,
                   void* __restrict__ Dv, int64_t ldd, int M, int N, int K,
                   int kb_per_chunk, BatchArgs bat,
                   const int64_t* __restrict__ row_term,
                   const int64_t* __restrict__ col_term, unsigned* status,
                   int stream_operands, const TestHook hook) {
  using L = Layout<BN, STAGES, CL, NSTG>;
  constexpr int HALF = BN / 2;  // columns per epilogue warp
  static_assert(EPI != Epi::I32SAT || BN == 128, "I32SAT uses 128-wide tiles");
  // I32SAT: the two accumulators take columns [0, 256); the 64-bit partial
  // sums of column half h the 128 columns from 256 + 128 h.
  constexpr uint32_t TMEM_COLS = EPI == Epi::I32SAT ? 512u : L::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFFSET);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint64_t* cbar = done + 1;  // NSTG per epilogue warp: C block landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cbar + NSTG * kEpiWarps);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  // Work units: CL vertically adjacent tiles per cluster, of one batch entry
  // (entries in order, tiles M-grouped within an entry).  The CTA of rank r
  // in its cluster takes m-block (unit row) * CL + r.
  const int unit_m = (num_m + CL - 1) / CL;
  const int per_entry = unit_m * num_n;
  const int units = per_entry * bat.batch;
  // Tile coordinates of unit u and the tensor-map batch coordinates of its
  // A, B and C/D tiles.
  auto decode = [&](int u, int& mu, int& nb, int& za, int& zb, int& zc) {
    const int b = u / per_entry;
    tile_coords(u - b * per_entry, unit_m, num_n, mu, nb);
    za = (b / bat.group) * bat.group + bat.abid;
    zb = (b & ~3) + blgp_source(bat.blgp, b & 3);
    zc = b;
  };
  const int first_unit = blockIdx.x / CL;
  const int unit_step = gridDim.x / CL;
  const int rank = CL > 1 ? int(cluster_ctarank()) : 0;
  const int num_kb = (K + BK - 1) / BK;
  // only the exact integer modes cut K into chunks (one accumulator each)
  const int kpc = int_mode(EPI) ? kb_per_chunk : num_kb;
  const int chunks = (num_kb + kpc - 1) / kpc;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], CL * kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(done, 1);
    for (int i = 0; i < NSTG * kEpiWarps; ++i) mbar_init(&cbar[i], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
    if (Cv) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    if constexpr (CL == 1) {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    }
  }
  tc_fence_before();
  if constexpr (CL > 1)
    cluster_sync();  // the peer's barriers exist before anything targets them
  else
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
      // the leader CTA's full barriers, which count both CTAs' bytes
      const uint32_t full_lead =
          CL > 1 ? mapa_shared(smem_u32(&full[0]), 0) : 0u;
      // A and B may be produced by the kernel launched just before this one
      // (the INT8 widening pass, launched as a programmatic dependency):
      // only the operand loads wait for it; the rest of the prologue and
      // the epilogue's C prefetch overlap its tail.
      grid_dependency_wait();
      // operands read by a single tile each (one column or one row of
      // tiles): evict-first, so the streamed panels leave L2 to C and to
      // the other operand
      uint64_t pol_op = 0;
      if (stream_operands)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
                     : "=l"(pol_op));
      for (int u = first_unit; u < units && ok; u += unit_step) {
        int mu, nb, za, zb, zc;
        decode(u, mu, nb, za, zb, zc);
        const int mb = mu * CL + rank;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status, hook.wait_limit_ns)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * L::STAGE_BYTES;
          if (hook.skip_loads) {
            // self-test: no load, so the stage never fills
          } else if constexpr (CL == 1) {
            mbar_arrive_expect_tx(&full[stage], L::STAGE_BYTES);
            if (stream_operands) {
              tma_load_3d_hint(&tmA, &full[stage], sa, kb * BK, mb * BM, za,
                               pol_op);
              tma_load_3d_hint(&tmB, &full[stage], sa + L::A_BYTES, kb * BK,
                               nb * BN, zb, pol_op);
            } else {
              tma_load_3d(&tmA, &full[stage], sa, kb * BK, mb * BM, za);
              tma_load_3d(&tmB, &full[stage], sa + L::A_BYTES, kb * BK,
                          nb * BN, zb);
            }
          } else {
            // the leader expects the bytes of both CTAs' stage
            if (rank == 0)
              mbar_arrive_expect_tx(&full[stage], CL * L::STAGE_BYTES);
            const uint32_t fb = full_lead + uint32_t(stage) * 8u;
            if (stream_operands) {
              tma_load_3d_pair_hint(&tmA, fb, sa, kb * BK, mb * BM, za, pol_op);
              tma_load_3d_pair_hint(&tmB, fb, sa + L::A_BYTES, kb * BK,
                                    nb * BN + rank * (BN / CL), zb, pol_op);
            } else {
              tma_load_3d_pair(&tmA, fb, sa, kb * BK, mb * BM, za);
              tma_load_3d_pair(&tmB, fb, sa + L::A_BYTES, kb * BK,
                               nb * BN + rank * (BN / CL), zb);
            }
          }
          if (!hook.skip_loads) ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t fills = issued / STAGES + (uint32_t(s) < issued % STAGES);
        if (!fills) continue;
        // Let every load still in flight land before the CTA exits (the
        // leader's full barriers also count the peer's loads).
        if (!ok && rank == 0)
          mbar_wait_drain(&full[s], (fills - 1) & 1u, status);
        // With a pair, the last release of each stage is the leader's
        // commit; wait until it has arrived on this CTA.
        if (CL > 1) mbar_wait_drain(&empty[s], (fills - 1) & 1u, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // (with a pair, only the leader CTA issues)
    if (rank == 0 && elect_one()) {
      constexpr uint32_t idesc = idesc_f16_f32(BF16, BM * CL, BN);
      constexpr uint16_t kPairMask = 3u;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = first_unit; u < units && ok; u += unit_step) {
        for (int ch = 0; ch < chunks && ok; ++ch) {
          if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, status, hook.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
          const int kb0 = ch * kpc;
          const int kb1 = min(num_kb, kb0 + kpc);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, status, hook.wait_limit_ns)) {
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
              const uint32_t accum = (kb != kb0 || k != 0) ? 1u : 0u;
              if constexpr (CL == 1)
                umma_f16(d_tmem, da + uint64_t(2 * k), db + uint64_t(2 * k),
                         idesc, accum);
              else
                umma_f16_pair(d_tmem, da + uint64_t(2 * k),
                              db + uint64_t(2 * k), idesc, accum);
            }
            if constexpr (CL == 1)
              umma_commit(&empty[stage]);
            else
              umma_commit_pair(&empty[stage], kPairMask);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if constexpr (CL == 1)
            umma_commit(&tfull[acc]);
          else
            umma_commit_pair(&tfull[acc], kPairMask);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      // Every MMA issued above completes before tensor memory is released.
      if constexpr (CL == 1)
        umma_commit(done);
      else
        umma_commit_pair(done, 1u);
      mbar_wait_drain(done, 0, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue warps
    // Each warp owns a 32-row quarter of the tile (its TMEM lane quarter)
    // and one column half, emitted as 16-column blocks through a ring of
    // NSTG staging blocks: D leaves by TMA store, and C arrives by TMA PF
    // blocks ahead of its use -- across tile boundaries, so the next tile's
    // first C blocks are in flight while this tile finishes.  In the
    // integer modes the chunks' INT32 sums are kept in registers; C joins
    // them either as each block is emitted or, with two staging blocks per
    // warp, while the chunks run (early C, below).  (Accumulating the
    // chunks into D with TMA reduce-add instead was measured slower: the L2
    // atomics cost more than the registers.)
    // Integer modes: C is read once and D written once, while the widened
    // operands (64 MB at 4096^3) are re-read from L2 by every wave of
    // tiles; C and D take an evict-first L2 policy so they do not push
    // the operands out (INT8 4096^3: 102.9 -> 101.4 us per call; the
    // FP32 and 16-bit modes keep the default, BF16 8192^3 lost 1 % with it).
    [[maybe_unused]] uint64_t pol_cd = 0;
    if constexpr (int_mode(EPI))
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
                   : "=l"(pol_cd));
    const int ew = warp - 2;           // 0 .. 7
    const int q = warp & 3;            // tensor-memory lane quarter
    const int h = ew >> 2;             // column half of the tile
    const int lane = threadIdx.x & 31;
    uint8_t* stg = smem + L::STG_OFFSET + ew * NSTG * kStgBytes;
    uint64_t* wbar = &cbar[NSTG * ew];
    [[maybe_unused]] uint32_t* sgn =
        reinterpret_cast<uint32_t*>(smem + L::TOTAL) + ew * sign_words<BN>() * 32;
    const bool has_c = Cv != nullptr;
    // columns per 64-byte staging row: 16 of 4 bytes, or 32 of 2 bytes
    constexpr int COLS = EPI == Epi::H16 ? 32 : 16;
    constexpr int NBLK = HALF / COLS;
    // The C of block g + PF is requested while block g is processed; its
    // ring slot last held block g + PF - NSTG, whose store must have
    // finished reading it, which leaves at most WAITN later stores pending.
    constexpr int PF = NSTG > 2 ? NSTG - 2 : 1;
    constexpr int WAITN = NSTG - PF - 1;
    static_assert(PF <= NBLK, "C is prefetched at most one tile ahead");
    // Before the first unit every ring slot is free, so the C of its first
    // PF0 blocks is requested at once (a CTA with a single tile then has
    // all of its C in flight while its main loop runs).
    constexpr int PF0 = NSTG < NBLK ? NSTG : NBLK;
    // Exact INT8 (sums modulo 2^32, so C may join them in any order): the
    // C blocks are added to the INT32 register sums while the unit's
    // chunks run, two blocks per chunk through staging slots 0 and 1 (one
    // step: both requested, then both consumed after the next chunk's
    // drain), and the emission only stores D.  Its C latency hides behind
    // MMA work, and two staging blocks per warp suffice.
    // (Instances with two staging blocks per warp; with one or two chunks
    // per tile the host picks the four-block ring, whose C loads run ahead
    // in the emission instead.)
    // I32SATE takes the same early C and also keeps the sign bit of each
    // C element it adds.
    constexpr bool kEarlyC =
        (EPI == Epi::I32EXACT || EPI == Epi::I32SATE) && NSTG == 2;
    static_assert(!kEarlyC || NSTG >= 2, "early C uses staging slots 0 and 1");
    static_assert(EPI != Epi::I32SATE || kEarlyC,
                  "I32SATE adds C while the chunks run");
    constexpr int NMP = (NBLK + 1) / 2;  // early-C steps per unit
    uint32_t cpar = 0;                   // phase parity of slots 0 and 1
    uint32_t g = 0;  // blocks emitted so far by this warp
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    // Row `lane` of a staging block, 16-byte chunk c, 64-byte swizzle.
    auto chunk = [&](uint8_t* buf, int c) {
      return reinterpret_cast<uint4*>(buf + lane * 64 +
                                      ((c ^ ((lane >> 1) & 3)) << 4));
    };
    // Return accumulator buffer `a` to the MMA issuer once this warp's TMEM
    // reads of it are complete (to the leader CTA's barrier for a pair).
    auto release_acc = [&](int a) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CL == 1)
          mbar_arrive(&tempty[a]);
        else
          mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[a]), 0));
      }
    };
    // Integer modes with an unsigned operand: the correction terms are
    // written by the widening pass this kernel may overlap (programmatic
    // launch), so wait for it before reading them.
    const bool has_terms = int_mode(EPI) && (row_term || col_term);
    if (has_terms) grid_dependency_wait();
    // Correction terms of a unit: this lane's row term, and the column
    // terms of the warp's HALF columns, one per lane per group of 32 (each
    // lane loads one; shuffles hand them to the others).  Zero when absent
    // or outside the problem.
    constexpr int TG = (HALF + 31) / 32;
    [[maybe_unused]] auto load_terms = [&](int r0, int c0, int64_t& rt,
                                           int64_t (&ct)[TG]) {
      const int row = r0 + lane;
      rt = (row_term && row < M) ? __ldg(row_term + row) : 0;
#pragma unroll
      for (int g = 0; g < TG; ++g) {
        const int col = c0 + g * 32 + lane;
        ct[g] = (col_term && col < N) ? __ldg(col_term + col) : 0;
      }
    };
    // The term of column c0 + jj of the unit whose terms are in ct.
    [[maybe_unused]] auto col_term_of = [&](const int64_t (&ct)[TG], int jj) {
      return __shfl_sync(0xffffffffu, ct[jj / 32], jj % 32);
    };
    // I32SAT: this warp's 64-bit partial sums, 16 columns per 32-column
    // group (low words, then high words), in the TMEM columns beyond the
    // two accumulators.
    [[maybe_unused]] const uint32_t xaddr =
        tmem_base + uint32_t(2 * BN + h * 2 * HALF) + (uint32_t(q * 32) << 16);
    // Add the INT32 chunk sums to the 64-bit partial sums (or start them,
    // from the unit's correction terms rt, ct) and clear the INT32 sums.
    [[maybe_unused]] auto fold_partials =
        [&](bool started, uint32_t (&ia)[int_mode(EPI) ? HALF : 1], int64_t rt,
            const int64_t (&ct)[TG]) {
      if constexpr (EPI == Epi::I32SAT) {
#pragma unroll
        for (int c = 0; c < HALF / 16; ++c) {
          uint32_t x[32];
          if (started) {
            tmem_ld_32x32b_x32(xaddr + uint32_t(c * 32), x);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const uint64_t t0 =
                  has_terms ? uint64_t(rt + col_term_of(ct, c * 16 + e)) : 0u;
              x[e] = uint32_t(t0);
              x[16 + e] = uint32_t(t0 >> 32);
            }
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int64_t v = int64_t((uint64_t(x[16 + e]) << 32) | x[e]) +
                              int64_t(int32_t(ia[c * 16 + e]));
            x[e] = uint32_t(uint64_t(v));
            x[16 + e] = uint32_t(uint64_t(v) >> 32);
            ia[c * 16 + e] = 0u;
          }
          tmem_st_32x32b_x32(xaddr + uint32_t(c * 32), x);
        }
        tmem_st_wait();
      }
    };
    // Store staging block `buf` to D at (col, row0) of entry z, or close an
    // empty bulk group when the block lies wholly outside D.  A TMA store
    // clipped at a row end that is not 16-byte aligned still writes that
    // 16-byte chunk whole, which would overwrite the caller's columns past
    // N; so D's tensor map ends at N_TMA (N rounded down to 16 bytes) and
    // the columns [N_TMA, N) are stored by the lanes, one element each
    // (lane = row of the block).
    constexpr int EB = EPI == Epi::H16 ? 2 : 4;  // bytes per D element
    const int n_tma = N & ~(16 / EB - 1);
    auto emit_block = [&](uint8_t* buf, int col, int row0, int z) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (col < n_tma && row0 < M) {
          if constexpr (int_mode(EPI))
            tma_store_3d_hint(&tmD, buf, col, row0, z, pol_cd);
          else
            tma_store_3d(&tmD, buf, col, row0, z);
        }
        bulk_commit_group();
      }
      if (col + COLS > n_tma && col < N && row0 + lane < M) {
        const int c0 = col > n_tma ? col : n_tma;
        const int c1 = col + COLS < N ? col + COLS : N;
        uint8_t* drow = static_cast<uint8_t*>(Dv) +
                        (int64_t(z) * M + row0 + lane) * ldd * EB;
        for (int c = c0; c < c1; ++c) {
          const int byte = (c - col) * EB;  // within the 64-byte block row
          const uint8_t* src = buf + lane * 64 +
                               (((byte >> 4) ^ ((lane >> 1) & 3)) << 4) +
                               (byte & 15);
          if constexpr (EB == 4)
            *reinterpret_cast<uint32_t*>(drow + int64_t(c) * 4) =
                *reinterpret_cast<const uint32_t*>(src);
          else
            *reinterpret_cast<uint16_t*>(drow + int64_t(c) * 2) =
                *reinterpret_cast<const uint16_t*>(src);
        }
      }
      __syncwarp();
    };
    // This warp's first row and first column in work unit u, and the
    // unit's batch entry.
    auto unit_origin = [&](int u, int& row0, int& colh, int& z) {
      int mu, nb, za, zb;
      decode(u, mu, nb, za, zb, z);
      row0 = (mu * CL + rank) * BM + q * 32;
      colh = nb * BN + h * HALF;
    };
    // (lane 0) Request the C of block gg, which is block jj of unit u.
    auto request_c = [&](uint32_t gg, int u, int jj) {
      const uint32_t b = gg % NSTG;
      int row0, colh, z;
      unit_origin(u, row0, colh, z);
      bulk_wait_group_read<WAITN>();
      if (row0 < M && colh + jj * COLS < N) {
        mbar_arrive_expect_tx(&wbar[b], kStgBytes);
        if constexpr (int_mode(EPI))
          tma_load_3d_hint(&tmC, &wbar[b], stg + b * kStgBytes, colh + jj * COLS,
                           row0, z, pol_cd);
        else
          tma_load_3d(&tmC, &wbar[b], stg + b * kStgBytes, colh + jj * COLS,
                      row0, z);
      } else {
        mbar_arrive(&wbar[b]);  // wholly outside C and D: nothing to load
      }
    };
    if (!kEarlyC && has_c && lane == 0 && first_unit < units)
      for (int jj = 0; jj < PF0; ++jj) request_c(uint32_t(jj), first_unit, jj);
    __syncwarp();
    // Early C, step m of the unit at (row0, colh, z): (lane 0) request
    // blocks 2m and 2m + 1 into slots 0 and 1, once every store that read
    // them has finished; a block outside C (or beyond the unit) only
    // arrives, so both slots advance one phase per step.
    [[maybe_unused]] auto early_c_issue = [&](int m, int row0, int colh, int z) {
      if (lane == 0) {
        bulk_wait_group_read<0>();
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
          const int jj = 2 * m + sl;
          if (jj < NBLK && row0 < M && colh + jj * COLS < N) {
            mbar_arrive_expect_tx(&wbar[sl], kStgBytes);
            tma_load_3d_hint(&tmC, &wbar[sl], stg + sl * kStgBytes,
                             colh + jj * COLS, row0, z, pol_cd);
          } else {
            mbar_arrive(&wbar[sl]);
          }
        }
      }
      __syncwarp();
    };
    for (int u = first_unit; u < units && ok; u += unit_step) {
      int row0, colh, zc;
      unit_origin(u, row0, colh, zc);
      [[maybe_unused]] uint32_t iacc[int_mode(EPI) ? HALF : 1];
      // I32SAT: whether this unit's 64-bit sums in TMEM hold chunks yet
      [[maybe_unused]] bool folded = false;
      uint32_t taddr = 0;
      [[maybe_unused]] int64_t rt = 0;
      [[maybe_unused]] int64_t ct[TG];
      if constexpr (int_mode(EPI)) {
        // I32EXACT and I32SATE start from the correction terms modulo
        // 2^32 and I32SATW from their exact value (in range by the host's
        // check);
        // I32SAT adds them in 64 bits at its first fold.
        if (has_terms) load_terms(row0, colh, rt, ct);
        if (EPI != Epi::I32SAT && has_terms) {
#pragma unroll
          for (int j = 0; j < HALF; ++j)
            iacc[j] = uint32_t(uint64_t(rt + col_term_of(ct, j)));
        } else {
#pragma unroll
          for (int j = 0; j < HALF; ++j) iacc[j] = 0u;
        }
        // early C: steps issued and consumed in this unit
        [[maybe_unused]] int mp_issued = 0, mp_done = 0;
        // Wait for the oldest issued step's two blocks and add them to the
        // sums (the step number selects registers through an unrolled
        // match, so iacc stays in registers).
        [[maybe_unused]] auto early_c_finish = [&]() -> bool {
          bool okc = mbar_wait(&wbar[0], cpar, abort_flag, status, hook.wait_limit_ns) &&
                     mbar_wait(&wbar[1], cpar, abort_flag, status, hook.wait_limit_ns);
          if (!__all_sync(0xffffffffu, okc)) return false;
#pragma unroll
          for (int m = 0; m < NMP; ++m) {
            if (m != mp_done) continue;
            // I32SATE: step m's two blocks are columns [32 m, 32 m + 32)
            // of the warp's half, one sign word per lane
            [[maybe_unused]] uint32_t neg = 0u;
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
              const int jj = 2 * m + sl;
              if (jj >= NBLK) continue;
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint4 w = *chunk(stg + sl * kStgBytes, c);
                iacc[jj * 16 + 4 * c + 0] += w.x;
                iacc[jj * 16 + 4 * c + 1] += w.y;
                iacc[jj * 16 + 4 * c + 2] += w.z;
                iacc[jj * 16 + 4 * c + 3] += w.w;
                if constexpr (EPI == Epi::I32SATE) {
                  const int b0 = sl * 16 + 4 * c;
                  neg |= ((w.x >> 31) << b0) | ((w.y >> 31) << (b0 + 1)) |
                         ((w.z >> 31) << (b0 + 2)) | ((w.w >> 31) << (b0 + 3));
                }
              }
            }
            if constexpr (EPI == Epi::I32SATE) sgn[m * 32 + lane] = neg;
          }
          __syncwarp();  // every lane has read both slots
          cpar ^= 1u;
          ++mp_done;
          return true;
        };
        if constexpr (kEarlyC) {
          if (has_c) early_c_issue(mp_issued++, row0, colh, zc);
        }
        for (int ch = 0; ch < chunks; ++ch) {
          ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, status, hook.wait_limit_ns);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          taddr = tmem_base + uint32_t(acc * BN + h * HALF) +
                  (uint32_t(q * 32) << 16);
#pragma unroll
          for (int c = 0; c < HALF / 16; ++c) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(taddr + uint32_t(c * 16), r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              iacc[c * 16 + j] += uint32_t(__float2int_rn(__uint_as_float(r[j])));
          }
          release_acc(acc);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
          if constexpr (kEarlyC) {
            if (has_c && mp_done < mp_issued) {
              if (!early_c_finish()) {
                ok = false;
                break;
              }
              if (mp_issued < NMP) early_c_issue(mp_issued++, row0, colh, zc);
            }
          }
          if constexpr (EPI == Epi::I32SAT) {
            // every kSatFlush chunks, and after the last one
            if ((ch + 1) % kSatFlush == 0 || ch + 1 == chunks) {
              fold_partials(folded, iacc, rt, ct);
              folded = true;
            }
          }
        }
        if (!ok) break;
        if constexpr (kEarlyC) {
          // fewer chunks than steps: the remaining C blocks now
          while (has_c && ok && mp_done < NMP) {
            if (mp_done == mp_issued) early_c_issue(mp_issued++, row0, colh, zc);
            ok = early_c_finish();
          }
          if (!ok) break;
        }
      } else {
        ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, status, hook.wait_limit_ns);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        taddr = tmem_base + uint32_t(acc * BN + h * HALF) +
                (uint32_t(q * 32) << 16);
      }
#pragma unroll
      for (int j = 0; j < NBLK; ++j, ++g) {
        uint8_t* buf = stg + (g % NSTG) * kStgBytes;
        if (lane == 0) {
          if (has_c && !kEarlyC) {
            // the C of block g + PF, possibly in this warp's next unit
            int jj = j + PF, uu = u;
            if (jj >= NBLK) {
              jj -= NBLK;
              uu = u + unit_step;
            }
            if (uu < units && g + PF >= uint32_t(PF0))
              request_c(g + PF, uu, jj);
          } else {
            bulk_wait_group_read<NSTG - 1>();  // slot's last store has read it
          }
        }
        __syncwarp();
        [[maybe_unused]] uint32_t r[EPI == Epi::I32SAT ? 32 : COLS];
        if constexpr (EPI == Epi::F32) {
          tmem_ld_32x32b_x16(taddr + uint32_t(j * 16), r);
        } else if constexpr (EPI == Epi::H16) {
          tmem_ld_32x32b_x32(taddr + uint32_t(j * 32), r);
        } else if constexpr (EPI == Epi::I32SAT) {
          // the 64-bit sums of this block's 16 columns (every chunk folded
          // in): low words in r[0..15], high words in r[16..31]
          tmem_ld_32x32b_x32(xaddr + uint32_t(j * 32), r);
          tmem_ld_wait();
        }
        if constexpr (!int_mode(EPI)) {
          tmem_ld_wait();
          // every TMEM read of this accumulator is done: release it
          if (j == NBLK - 1) release_acc(acc);
        }
        if (has_c && !kEarlyC) {
          ok = mbar_wait(&wbar[g % NSTG], (g / NSTG) & 1u, abort_flag, status, hook.wait_limit_ns);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        // I32SATE: the sign bits of this block's C (none without C)
        [[maybe_unused]] uint32_t negw = 0u;
        if constexpr (EPI == Epi::I32SATE)
          negw = has_c ? sgn[(j / 2) * 32 + lane] : 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4* p = chunk(buf, c);
          const uint4 w =
              has_c && !kEarlyC ? *p : make_uint4(0u, 0u, 0u, 0u);
          uint4 o;
          if constexpr (EPI == Epi::H16) {
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
            uint32_t ov[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float f0 = half_to_f32<BF16>(wv[e] & 0xFFFFu) +
                               __uint_as_float(r[8 * c + 2 * e]);
              const float f1 = half_to_f32<BF16>(wv[e] >> 16) +
                               __uint_as_float(r[8 * c + 2 * e + 1]);
              ov[e] = f32x2_to_half2<BF16>(f0, f1);
            }
            o = make_uint4(ov[0], ov[1], ov[2], ov[3]);
          } else if constexpr (EPI == Epi::F32) {
            o.x = __float_as_uint(__uint_as_float(w.x) + __uint_as_float(r[4 * c + 0]));
            o.y = __float_as_uint(__uint_as_float(w.y) + __uint_as_float(r[4 * c + 1]));
            o.z = __float_as_uint(__uint_as_float(w.z) + __uint_as_float(r[4 * c + 2]));
            o.w = __float_as_uint(__uint_as_float(w.w) + __uint_as_float(r[4 * c + 3]));
          } else if constexpr (EPI == Epi::I32EXACT) {
            // INT32 adds wrap modulo 2^32
            o.x = w.x + iacc[j * 16 + 4 * c + 0];
            o.y = w.y + iacc[j * 16 + 4 * c + 1];
            o.z = w.z + iacc[j * 16 + 4 * c + 2];
            o.w = w.w + iacc[j * 16 + 4 * c + 3];
          } else if constexpr (EPI == Epi::I32SATE) {
            // iacc holds S + C modulo 2^32 with S in [-2^30, 2^30): the
            // sign of C tells an overflow from a wrapped value
            auto sat = [&](int e) {
              const int32_t v = int32_t(iacc[j * 16 + 4 * c + e]);
              const bool neg = (negw >> ((j & 1) * 16 + 4 * c + e)) & 1u;
              const int32_t out = !neg && v < -(1 << 30) ? INT32_MAX
                                  : neg && v >= (1 << 30) ? INT32_MIN
                                                          : v;
              return uint32_t(out);
            };
            o.x = sat(0);
            o.y = sat(1);
            o.z = sat(2);
            o.w = sat(3);
          } else {
            // exact 64-bit sum, saturated once to the INT32 range
            auto sat = [&](uint32_t cw, int e) {
              int64_t v;
              if constexpr (EPI == Epi::I32SAT)
                v = int64_t((uint64_t(r[16 + e]) << 32) | r[e]);
              else  // I32SATW: the exact sum (terms included) in INT32
                v = int64_t(int32_t(iacc[j * 16 + e]));
              v += int64_t(int32_t(cw));
              v = v < int64_t(INT32_MIN) ? int64_t(INT32_MIN) : v;
              v = v > int64_t(INT32_MAX) ? int64_t(INT32_MAX) : v;
              return uint32_t(int32_t(v));
            };
            o.x = sat(w.x, 4 * c + 0);
            o.y = sat(w.y, 4 * c + 1);
            o.z = sat(w.z, 4 * c + 2);
            o.w = sat(w.w, 4 * c + 3);
          }
          *p = o;
        }
        emit_block(buf, colh + j * COLS, row0, zc);
      }
      if constexpr (!int_mode(EPI)) {
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
    // every store of this warp has landed before the CTA finishes
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before();
  if constexpr (CL > 1)
    cluster_sync();  // neither CTA leaves while the other may still signal it
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CL == 1)
      tmem_dealloc(tmem_base, TMEM_COLS);
    else
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// 8-bit integer -> bfloat16, exactly.  Each input byte x is stored as the
// value (x ^ flip) - 128: for int8 (flip = 0x80) that is the value itself,
// for uint8 u (flip = 0) it is u - 128, shifted into the int8 range so that
// every product keeps the signed bound |a*b| <= 2^14 (the exact sum is
// restored by the correction terms of widen_rows_kernel).  Both lie in
// [-128, 127] and have at most 8 significant bits.  Full-rate integer/FP32
// ALU operations replace the slower int-to-float conversion unit: with
// u = x ^ flip, the float whose bits are 0x4B0000uu is 2^23 + u, so
// subtracting 2^23 + 128 leaves the stored value exactly, and its top 16
// bits are its bfloat16.
constexpr uint32_t kFlipSigned = 0x80808080u;

__device__ __forceinline__ uint32_t i8x2_to_bf16x2(uint32_t u, int lo_byte) {
  // byte_perm picks byte `lo_byte` of u (already flipped) into the low byte
  // of 0x4B000000
  const uint32_t f0 = __byte_perm(u, 0x4B000000u, 0x7540u + lo_byte);
  const uint32_t f1 = __byte_perm(u, 0x4B000000u, 0x7541u + lo_byte);
  const float v0 = __uint_as_float(f0) - 8388736.0f;  // 2^23 + 128
  const float v1 = __uint_as_float(f1) - 8388736.0f;
  // high halves of the two floats: (bf16(v1) << 16) | bf16(v0)
  return __byte_perm(__float_as_uint(v0), __float_as_uint(v1), 0x7632);
}

// The bfloat16 bit pattern of one stored value u - 128 (u = x ^ flip; plain
// conversion, for ragged row tails and the transposing pass).
__device__ __forceinline__ uint16_t flipped_byte_to_bf16(uint32_t u) {
  return uint16_t(__float_as_uint(float(int(u) - 128)) >> 16);
}

// 16 bytes (already flipped) -> 16 bfloat16 values.
__device__ __forceinline__ void u8x16_to_bf16(const uint32_t (&u)[4],
                                              uint4& o0, uint4& o1) {
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) o[j] = i8x2_to_bf16x2(u[j >> 1], 2 * (j & 1));
  o0 = make_uint4(o[0], o[1], o[2], o[3]);
  o1 = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void flip4(const int4 v, uint32_t flip,
                                      uint32_t (&u)[4]) {
  u[0] = uint32_t(v.x) ^ flip;
  u[1] = uint32_t(v.y) ^ flip;
  u[2] = uint32_t(v.z) ^ flip;
  u[3] = uint32_t(v.w) ^ flip;
}

// Signed x signed inputs (no correction terms): one flat index over the
// 16-byte chunks of the rows of A then of B.  Each block takes 2 x 512
// consecutive chunks, thread t the chunks t and t + 512 of them: both loads
// are in flight together and every warp-wide load and store covers one
// contiguous run of memory.  (Measured on the 4096^3 INT8 step against
// 256 threads x 4 chunks: 108.9 against 114.5 us per step; 1024 x 1 and
// 256 x 2 with a larger grid were within 0.5 us of it.)
constexpr int kConvThreads = 512;
constexpr int kConvUnroll = 2;

__global__ void __launch_bounds__(kConvThreads)
    i8_to_bf16_kernel(const int8_t* __restrict__ A, int64_t lda, int M,
                      const int8_t* __restrict__ B, int64_t ldb, int N, int K,
                      uint16_t* __restrict__ W, int64_t ldw) {
  const int64_t cpr = (K + 15) / 16;  // chunks per row
  const int64_t total = int64_t(M + N) * cpr;
  constexpr int64_t kSpan = int64_t(kConvThreads) * kConvUnroll;
  // the 8-bit inputs are read once (evict first); the widened operands
  // are read back by the GEMM right after this pass (evict last), which
  // then finds most of them in L2
  uint64_t pol_first, pol_last;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_first));
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_last));
  for (int64_t base = int64_t(blockIdx.x) * kSpan; base < total;
       base += int64_t(gridDim.x) * kSpan) {
    int4 v[kConvUnroll];
#pragma unroll
    for (int u = 0; u < kConvUnroll; ++u) {
      const int64_t i = base + threadIdx.x + int64_t(u) * kConvThreads;
      v[u] = make_int4(0, 0, 0, 0);
      if (i < total) {
        const int64_t r = i / cpr;
        const int c = int(i - r * cpr) * 16;
        if (c + 16 <= K) {
          const int8_t* src = r < M ? A + r * lda + c : B + (r - M) * ldb + c;
          asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.s32 {%0, %1, %2, %3}, [%4], %5;"
                       : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                       : "l"(src), "l"(pol_first));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kConvUnroll; ++u) {
      const int64_t i = base + threadIdx.x + int64_t(u) * kConvThreads;
      if (i >= total) continue;
      const int64_t r = i / cpr;
      const int c = int(i - r * cpr) * 16;
      uint16_t* dst = W + r * ldw + c;
      if (c + 16 <= K) {
        uint32_t w[4];
        flip4(v[u], kFlipSigned, w);
        uint4 o0, o1;
        u8x16_to_bf16(w, o0, o1);
        asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;"
                     :: "l"(dst), "r"(o0.x), "r"(o0.y), "r"(o0.z), "r"(o0.w), "l"(pol_last) : "memory");
        asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;"
                     :: "l"(dst + 8), "r"(o1.x), "r"(o1.y), "r"(o1.z), "r"(o1.w), "l"(pol_last) : "memory");
      } else {
        const int8_t* src = r < M ? A + r * lda + c : B + (r - M) * ldb + c;
        for (int j = 0; c + j < K; ++j)
          dst[j] = flipped_byte_to_bf16(uint32_t(uint8_t(src[j])) ^ 0x80u);
      }
    }
  }
}

// Inputs with an unsigned operand.  With oa, ob = 128 for an unsigned A, B
// (else 0) and A', B' the stored (shifted) values, A = A' + oa and
// B = B' + ob elementwise, so
//   (A B)_ij = (A' B')_ij + ob * r_i + oa * c_j + oa * ob * K,
//   r_i = sum_k A'_ik,  c_j = sum_k B'_kj,
// exactly; the GEMM computes A' B' with the signed chunk depth and its
// epilogue adds the per-row term row_term[i] = ob * r_i + oa * ob * K and the
// per-column term col_term[j] = oa * c_j (each array only when nonzero).
//
// This pass widens rows [0, M) of A and then rows [0, nb) of column-major B
// (nb = 0 when B is row-major and transposed separately) and writes those
// terms.  G lanes share a row (G a power of two <= 32): lane t of the group
// takes the row's 16-byte chunks t, t + G, ... (G * 16 contiguous bytes per
// warp access), four in flight, and the group adds its sums by shuffles.
constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads)
    widen_rows_kernel(const uint8_t* __restrict__ A, int64_t lda, int M,
                      const uint8_t* __restrict__ B, int64_t ldb, int nb,
                      int K, uint16_t* __restrict__ W, int64_t ldw,
                      uint32_t flip_a, uint32_t flip_b, int G,
                      int64_t* __restrict__ row_term, int64_t a_mul,
                      int64_t a_add, int64_t* __restrict__ col_term,
                      int64_t b_mul) {
  const int64_t rows = int64_t(M) + nb;
  const int64_t cpr = (K + 15) / 16;
  const int lane = threadIdx.x & 31;
  const int t = lane & (G - 1);
  const int64_t rows_per_warp = 32 / G;
  const int64_t warp0 =
      (int64_t(blockIdx.x) * kRowThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kRowThreads) >> 5;
  // as in i8_to_bf16_kernel: the 8-bit inputs are read once (evict first),
  // the widened operands are read back by the GEMM next (evict last)
  uint64_t pol_first, pol_last;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_first));
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_last));
  for (int64_t base = warp0 * rows_per_warp; base < rows;
       base += nwarps * rows_per_warp) {
    const int64_t r = base + lane / G;
    const bool live = r < rows;
    const bool is_a = r < M;
    uint64_t s = 0;  // sum over this lane's bytes of (x ^ flip)
    if (live) {
      const uint8_t* src = is_a ? A + r * lda : B + (r - M) * ldb;
      uint16_t* dst = W + r * ldw;
      const uint32_t flip = is_a ? flip_a : flip_b;
      for (int64_t c0 = t; c0 < cpr; c0 += 4 * G) {
        int4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t c = c0 + int64_t(u) * G;
          v[u] = make_int4(0, 0, 0, 0);
          if (c < cpr && c * 16 + 16 <= K)
            asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.s32 {%0, %1, %2, %3}, [%4], %5;"
                         : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                         : "l"(src + c * 16), "l"(pol_first));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t c = c0 + int64_t(u) * G;
          if (c >= cpr) continue;
          if (c * 16 + 16 <= K) {
            uint32_t w[4];
            flip4(v[u], flip, w);
            uint4 o0, o1;
            u8x16_to_bf16(w, o0, o1);
            asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;"
                         :: "l"(dst + c * 16), "r"(o0.x), "r"(o0.y), "r"(o0.z), "r"(o0.w), "l"(pol_last) : "memory");
            asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;"
                         :: "l"(dst + c * 16 + 8), "r"(o1.x), "r"(o1.y), "r"(o1.z), "r"(o1.w), "l"(pol_last) : "memory");
            // the 16 bytes' unsigned sum, four at a time
            const unsigned ones = 0x01010101u;
            s += __dp4a(w[0], ones, __dp4a(w[1], ones,
                        __dp4a(w[2], ones, __dp4a(w[3], ones, 0u))));
          } else {
            for (int64_t k = c * 16; k < K; ++k) {
              const uint32_t x = uint32_t(src[k]) ^ (flip & 0xFFu);
              dst[k] = flipped_byte_to_bf16(x);
              s += x;
            }
          }
        }
      }
    }
    for (int off = G >> 1; off > 0; off >>= 1)
      s += __shfl_xor_sync(0xffffffffu, s, off);
    if (live && t == 0) {
      // the sum of the row's stored values (x ^ flip) - 128
      const int64_t sum = int64_t(s) - 128 * int64_t(K);
      if (is_a) {
        if (row_term) row_term[r] = a_mul * sum + a_add;
      } else if (col_term) {
        col_term[r - M] = b_mul * sum;
      }
    }
  }
}

// ----------------------------------------------------------------- host

}  // namespace

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

// K-major operand: `count` tiles of `rows` rows of K contiguous 16-bit
// elements (leading dimension ld_elems; tile t starts rows * ld_elems
// elements after tile t - 1).  Inner dim K, then rows, then the tile; box
// 64 x box_rows x 1, 128-byte swizzle, zero fill out of bounds (so a box
// overhanging a tile's last row or K reads zeros, never the next tile).
bool make_kmajor_map(CUtensorMap* map, const void* base, int64_t K,
                     int64_t rows, int64_t ld_elems, int box_rows, bool bf16,
                     int64_t count) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cuuint64_t(K), cuuint64_t(rows), cuuint64_t(count)};
  cuuint64_t strides[2] = {cuuint64_t(ld_elems) * 2,
                           cuuint64_t(rows) * cuuint64_t(ld_elems) * 2};
  cuuint32_t box[3] = {cuuint32_t(BK), cuuint32_t(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map,
                   bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major C/D map over `count` M x N tiles (tile t starts M * ld_elems
// elements after tile t - 1): 64-byte (16 x 4-byte or 32 x 2-byte) x 32-row
// x 1 box, 64-byte swizzle, matching the epilogue's staging blocks.
bool make_cd_map(CUtensorMap* map, const void* base, int64_t N, int64_t M,
                 int64_t ld_elems, CUtensorMapDataType dt, int elem_bytes,
                 int64_t count) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cuuint64_t(N), cuuint64_t(M), cuuint64_t(count)};
  cuuint64_t strides[2] = {
      cuuint64_t(ld_elems) * cuuint64_t(elem_bytes),
      cuuint64_t(M) * cuuint64_t(ld_elems) * cuuint64_t(elem_bytes)};
  cuuint32_t box[3] = {cuuint32_t(64 / elem_bytes), 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt,
                   3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// pdl: launch as a programmatic dependent of the kernel just before it on
// the stream (a pass that produced A or B).
template <int BN, int STAGES, bool BF16, Epi EPI, int CL, int NSTG>
mma_status_t run(const Ctx& ctx, bool pdl, int64_t M, int64_t N, int64_t K,
                 const void* A, int64_t lda, const void* B, int64_t ldb,
                 const void* C, int64_t ldc, void* D, int64_t ldd,
                 int kb_per_chunk, BatchArgs bat, const int64_t* row_term,
                 const int64_t* col_term,
                 TestHook hook = TestHook{kWaitLimitNs, 0}) {
  constexpr int kSmem = smem_alloc<BN, STAGES, CL, NSTG, EPI>();
  static_assert(kSmem <= 232448, "shared memory per CTA");
  const CUtensorMapDataType cd_type =
      int_mode(EPI)        ? CU_TENSOR_MAP_DATA_TYPE_INT32
      : EPI == Epi::F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
      : BF16               ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int cd_bytes = EPI == Epi::H16 ? 2 : 4;
  CUtensorMap ta, tb, tc, td;
  const int64_t nt = bat.batch;  // tiles of each operand
  // D's map ends at the last 16-byte boundary of its rows (the kernel's
  // lanes store any columns beyond it); a map is still needed when that
  // leaves none, though the kernel then never stores through it.
  const int64_t n_tma = N & ~int64_t(16 / cd_bytes - 1);
  if (!make_kmajor_map(&ta, A, K, M, lda, BM, BF16, nt) ||
      !make_kmajor_map(&tb, B, K, N, ldb, BN / CL, BF16, nt) ||
      !make_cd_map(&td, D, n_tma > 0 ? n_tma : N, M, ldd, cd_type, cd_bytes, nt))
    return MMA_ERR_LAUNCH;
  if (C != nullptr) {
    if (!make_cd_map(&tc, C, N, M, ldc, cd_type, cd_bytes, nt))
      return MMA_ERR_LAUNCH;
  } else {
    tc = td;  // never read: the kernel loads C only when it is given
  }
  auto kern = gemm_tc_kernel<BN, STAGES, BF16, EPI, CL, NSTG>;
  // the dynamic shared-memory limit, once per context and instantiation
  static PerContext<bool> smem_attr;
  bool attr_ok = false;
  if (!smem_attr.get(ctx, &attr_ok, [&](bool* v) {
        *v = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSmem) == cudaSuccess;
        if (!*v) cudaGetLastError();
        return *v;
      }))
    return MMA_ERR_LAUNCH;
  const int64_t units =
      ((M + BM * CL - 1) / (BM * CL)) * ((N + BN - 1) / BN) * bat.batch;
  if (units > int64_t(INT32_MAX)) return MMA_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent: as many clusters as can be resident at once (at most one
  // per unit of work)
  int64_t clusters = ctx.num_sms / CL;
  if (CL > 1) {
    // clusters resident at once, once per context and instantiation
    static PerContext<int> resident;
    int r = 0;
    if (!resident.get(ctx, &r, [&](int* v) {
          cudaLaunchConfig_t probe = cfg;
          probe.gridDim = dim3(unsigned(CL * (ctx.num_sms / CL)), 1, 1);
          int n = 0;
          if (cudaOccupancyMaxActiveClusters(&n, kern, &probe) != cudaSuccess ||
              n < 1) {
            cudaGetLastError();
            return false;
          }
          *v = n;
          return true;
        }))
      return MMA_ERR_LAUNCH;
    clusters = r;
  }
  if (clusters > units) clusters = units;
  cfg.gridDim = dim3(unsigned(clusters * CL), 1, 1);
  if (pdl) cfg.numAttrs = 2;
  // Each A panel feeds one tile when there is one column of tiles, and each
  // B panel when there is one row: the operands then stream through L2
  // once (evict-first loads).  16384 x 128 x 4096 BF16: 32.9 -> 30.3 us;
  // the same hint on 4096^3 and 8192^3 products, whose panels are re-read
  // by later waves, was neutral or slower (BF16 8192^3 608 -> 670 us).
  const int stream_operands =
      ((N + BN - 1) / BN == 1 || (M + BM * CL - 1) / (BM * CL) == 1) ? 1 : 0;
  ctx.mark_start();
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, td, C, ldc, D, ldd, int(M), int(N),
                         int(K), kb_per_chunk, bat, row_term, col_term,
                         ctx.status, stream_operands, hook);
  ctx.mark_stop();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MMA_ERR_LAUNCH;
  }
  return MMA_OK;
}

// Cluster size: CTA pairs sharing one MMA (cta_group::2) for problems large
// enough to keep many pairs busy (at least two m-blocks, 2^30 multiply-adds
// and a full wave of 256 x 256 pair tiles); single CTAs otherwise.  With
// fewer pair tiles than pairs every SM would hold one tile and the pairs'
// synchronisation would buy nothing: the 16384 x 128 x 4096 BF16 product
// (64 pair tiles) ran in 34.6 us as pairs and 32.6 us as 128 single CTAs.
// MMA_GB300_CLUSTER (1 or 2) overrides the choice, for tuning.
int cluster_size(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                 int64_t batch = 1) {
  static const int forced = [] {
    const char* e = getenv("MMA_GB300_CLUSTER");
    const int v = e ? atoi(e) : 0;
    return (v == 1 || v == 2) ? v : 0;
  }();
  if (forced) return forced;
  const double work = double(M) * double(N) * double(K) * double(batch);
  const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256) * batch;
  return (M > BM && work >= 1073741824.0 && pair_tiles >= ctx.num_sms / 2)
             ? 2
             : 1;
}

// Tile width (columns of D per CTA or CTA pair): 256 when there are enough
// such tiles to occupy every SM, else 128 (more, smaller tiles).  CTA pairs
// with FP32 or exact-INT32 results may also take 224-wide tiles: the width
// with the smaller wave cost ceil(units / pairs) * width wins (ties go to
// 256).  Measured: at 4096^3 the 224-wide tiles fill exactly four waves of
// the 76 pairs (304 units) where 256-wide ones leave the fourth wave 37 %
// full, 6 % faster for INT8 and BF16; at 8192^3 both need the same waves
// and 256 is 6 % faster.  MMA_GB300_TILE_N (128, 224 or 256) overrides the
// choice, for tuning.
int tile_n(const Ctx& ctx, int64_t M, int64_t N, int64_t batch = 1,
           int cl = 1, bool allow224 = false) {
  static const int forced = [] {
    const char* e = getenv("MMA_GB300_TILE_N");
    const int v = e ? atoi(e) : 0;
    return (v == 128 || v == 224 || v == 256) ? v : 0;
  }();
  if (forced) return forced;
  const int64_t wide_tiles = ((M + BM - 1) / BM) * ((N + 255) / 256) * batch;
  if (!(N > 128 && wide_tiles >= ctx.num_sms)) return 128;
  if (cl == 2 && allow224) {
    const int64_t pairs = ctx.num_sms / 2;
    const int64_t m_units = (M + 2 * BM - 1) / (2 * BM) * batch;
    auto cost = [&](int64_t bn) {
      const int64_t units = m_units * ((N + bn - 1) / bn);
      return (units + pairs - 1) / pairs * bn;
    };
    if (cost(224) < cost(256)) return 224;
  }
  return 256;
}

template <bool BF16, Epi EPI>
mma_status_t dispatch(const Ctx& ctx, bool pdl, int bn, int cl, int64_t M,
                      int64_t N, int64_t K, const void* A, int64_t lda,
                      const void* B, int64_t ldb, const void* C, int64_t ldc,
                      void* D, int64_t ldd, const int64_t* row_term = nullptr,
                      const int64_t* col_term = nullptr,
                      BatchArgs bat = BatchArgs{1, 1, 0, 0}) {
  constexpr int kpc = kI8ChunkK / BK;
  // Shared memory: operand ring (a pair stages half of B per CTA) plus the
  // epilogue's staging ring.  Wide pair tiles: the MMA issuer spends most
  // of its time waiting for operand stages to land, so FP32, 16-bit and
  // exact-INT32 results take six stages and 2 staging blocks per warp
  // (FP32 and 16-bit drain one accumulator per tile, with a whole tile of
  // MMA work to hide it; exact INT32 adds C to its register sums while the
  // chunks run, from three 1024-deep chunks per tile up; so do saturated
  // INT32 results whose products stay below 2^30, I32SATE).  The other
  // saturating modes, and exact INT32 with one or two chunks, add C as
  // each block is emitted, within one chunk's MMA time, which needs 4
  // staging blocks per warp (2 C loads ahead), so they keep five stages.  Single-CTA wide
  // tiles (48 KB stages) take four stages and 2 staging blocks.
  if constexpr (EPI == Epi::I32SATE) {
    // early C only: 224-wide pair tiles with two staging blocks per warp
    // (256-wide ones leave no room for the sign words); the host picks
    // this mode for those tiles and three or more chunks
    if (cl == 2 && bn == 224)
      return run<224, 6, BF16, EPI, 2, 2>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
  } else if constexpr (EPI != Epi::I32SAT) {
    // 224-wide pair tiles (FP32 and exact-INT32 results: 112 columns per
    // epilogue warp, seven 16-column blocks)
    if constexpr (EPI == Epi::F32 || EPI == Epi::I32EXACT ||
                  EPI == Epi::I32SATW) {
      if (bn == 224 && cl == 2) {
        if constexpr (EPI == Epi::F32) {
          return run<224, 6, BF16, EPI, 2, 2>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
        } else if constexpr (EPI == Epi::I32EXACT) {
          if (K > 2 * kI8ChunkK)
            return run<224, 6, BF16, EPI, 2, 2>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
          return run<224, 5, BF16, EPI, 2, 4>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
        } else {
          return run<224, 5, BF16, EPI, 2, 4>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
        }
      }
    }
    if (bn >= 224) {
      if (cl == 2) {
        if constexpr (EPI == Epi::F32 || EPI == Epi::H16) {
          return run<256, 6, BF16, EPI, 2, 2>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
        } else if constexpr (EPI == Epi::I32EXACT) {
          if (K > 2 * kI8ChunkK)
            return run<256, 6, BF16, EPI, 2, 2>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
          return run<256, 5, BF16, EPI, 2, 4>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
        } else {
          return run<256, 5, BF16, EPI, 2, 4>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
        }
      }
      return run<256, 4, BF16, EPI, 1, 2>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
    }
  }
  // Single CTAs on 128-wide tiles with at most four K steps per tile (small
  // or batched small-block problems): the C stream is as large as the
  // operand stream, so trade a ring stage for two more C staging slots
  // (a whole tile of C in flight per warp).
  if constexpr (EPI == Epi::F32) {
    if (cl == 1 && (K + BK - 1) / BK <= 4)
      return run<128, 4, BF16, EPI, 1, 6>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
  }
  if constexpr (EPI == Epi::I32SATE) {
    return MMA_ERR_UNSUPPORTED;
  } else {
    return cl == 2 ? run<128, 6, BF16, EPI, 2, 4>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term)
                   : run<128, 5, BF16, EPI, 1, 4>(ctx, pdl, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, kpc, bat, row_term, col_term);
  }
}

// Row-major B (K x N, N contiguous) -> K-major copy W (N rows of K, leading
// dimension ldw) of 16-bit elements, through 64 x 64 shared-memory tiles
// with 16-byte global accesses on both sides:
//   * load: each thread reads 16 contiguous bytes of one row k of B (16
//     int8 or 8 16-bit values) into the tile [k][n];
//   * store: warp w writes the 8-deep K run w of the tile's 64 columns, 32
//     columns per pass: each thread gathers tile[8w .. 8w+7][n] (a warp
//     reads 32 consecutive columns of one tile row, conflict-free) and
//     writes them as one 16-byte run of row n of W.
// With I8 the 8-bit inputs are widened to their stored bfloat16 values on
// the way (exactly; x -> (x ^ flip) - 128, as in i8x2_to_bf16x2), and with
// col_term each column's sum of stored values times b_mul is added to
// col_term[n] (64-bit atomics, one per column per tile; col_term starts at
// zero).  Ragged edges fall back to element accesses.
constexpr int kTrTile = 64;
constexpr int kTrPad = 8;  // uint16 padding per tile row (16 bytes)

template <bool I8>
__global__ void __launch_bounds__(256)
    transpose_b_kernel(const void* __restrict__ Bv, int64_t ldb, int K, int N,
                       uint16_t* __restrict__ W, int64_t ldw, uint32_t flip,
                       int64_t* __restrict__ col_term, int64_t b_mul) {
  __shared__ __align__(16) uint16_t tile[kTrTile][kTrTile + kTrPad];  // [k][n]
  __shared__ int psum[8][kTrTile];
  const int n0 = blockIdx.x * kTrTile, k0 = blockIdx.y * kTrTile;
  const int tid = threadIdx.x;
  // ---- load: rows of B into the tile
  if constexpr (I8) {
    const uint8_t* B8 = static_cast<const uint8_t*>(Bv);
    const int kk = tid >> 2, c = (tid & 3) * 16;  // 64 rows x 4 chunks
    const int k = k0 + kk, n = n0 + c;
    uint32_t u[16];
    if (k < K && n + 16 <= N &&
        (reinterpret_cast<uintptr_t>(B8 + int64_t(k) * ldb + n) & 15) == 0) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(B8 + int64_t(k) * ldb + n));
      const uint32_t w[4] = {v.x ^ flip, v.y ^ flip, v.z ^ flip, v.w ^ flip};
#pragma unroll
      for (int e = 0; e < 16; ++e) u[e] = (w[e >> 2] >> (8 * (e & 3))) & 0xFFu;
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e)
        u[e] = (k < K && n + e < N)
                   ? (uint32_t(B8[int64_t(k) * ldb + n + e]) ^ (flip & 0xFFu))
                   : 128u;  // stored value 0
    }
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      o[e] = uint32_t(flipped_byte_to_bf16(u[2 * e])) |
             (uint32_t(flipped_byte_to_bf16(u[2 * e + 1])) << 16);
    uint4* dst = reinterpret_cast<uint4*>(&tile[kk][c]);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  } else {
    const uint16_t* B16 = static_cast<const uint16_t*>(Bv);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int kk = (tid >> 3) + 32 * r, c = (tid & 7) * 8;  // 32 rows x 8
      const int k = k0 + kk, n = n0 + c;
      uint4 v;
      if (k < K && n + 8 <= N &&
          (reinterpret_cast<uintptr_t>(B16 + int64_t(k) * ldb + n) & 15) == 0) {
        v = __ldcs(reinterpret_cast<const uint4*>(B16 + int64_t(k) * ldb + n));
      } else {
        uint16_t e16[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          e16[e] = (k < K && n + e < N) ? B16[int64_t(k) * ldb + n + e] : 0;
        v = make_uint4(e16[0] | (uint32_t(e16[1]) << 16),
                       e16[2] | (uint32_t(e16[3]) << 16),
                       e16[4] | (uint32_t(e16[5]) << 16),
                       e16[6] | (uint32_t(e16[7]) << 16));
      }
      *reinterpret_cast<uint4*>(&tile[kk][c]) = v;
    }
  }
  __syncthreads();
  // ---- store: 16-byte K runs of the rows of W
  const int warp = tid >> 5, lane = tid & 31;
  const int kr = warp * 8;  // this warp's K run within the tile
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int nn = lane + 32 * r;
    uint16_t e16[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e16[i] = tile[kr + i][nn];
    const int n = n0 + nn, k = k0 + kr;
    if (n < N) {
      uint16_t* dst = W + int64_t(n) * ldw + k;
      if (k + 8 <= K) {
        *reinterpret_cast<uint4*>(dst) =
            make_uint4(e16[0] | (uint32_t(e16[1]) << 16),
                       e16[2] | (uint32_t(e16[3]) << 16),
                       e16[4] | (uint32_t(e16[5]) << 16),
                       e16[6] | (uint32_t(e16[7]) << 16));
      } else {
        for (int i = 0; k + i < K; ++i) dst[i] = e16[i];
      }
    }
    if constexpr (I8) {
      // the run's stored values (exact small integers in bfloat16)
      int part = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (k + i < K) part += int(__uint_as_float(uint32_t(e16[i]) << 16));
      psum[warp][nn] = part;
    }
  }
  if constexpr (I8) {
    if (col_term != nullptr) {
      __syncthreads();
      if (tid < kTrTile && n0 + tid < N) {
        int64_t c = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) c += psum[w][tid];
        atomicAdd(reinterpret_cast<unsigned long long*>(col_term + n0 + tid),
                  static_cast<unsigned long long>(b_mul * c));
      }
    }
  }
}

template <bool I8>
mma_status_t launch_transpose_b(const Ctx& ctx, const void* B, int64_t ldb,
                                int64_t K, int64_t N, uint16_t* W,
                                int64_t ldw, uint32_t flip = kFlipSigned,
                                int64_t* col_term = nullptr,
                                int64_t b_mul = 0) {
  const int64_t gy = (K + 63) / 64;
  if (gy > 65535) return MMA_ERR_UNSUPPORTED;
  const dim3 grid{unsigned((N + 63) / 64), unsigned(gy), 1u};
  transpose_b_kernel<I8><<<grid, 256, 0, ctx.stream>>>(
      B, ldb, int(K), int(N), W, ldw, flip, col_term, b_mul);
  return cudaGetLastError() == cudaSuccess ? MMA_OK : MMA_ERR_LAUNCH;
}

}  // namespace

template <Epi EPI>
mma_status_t dispatch_f16(const Ctx& ctx, bool pdl, bool bf16, int64_t M,
                          int64_t N, int64_t K, const void* A, int64_t lda,
                          const void* B, int64_t ldb, const void* C,
                          int64_t ldc, void* D, int64_t ldd) {
  const int cl = cluster_size(ctx, M, N, K);
  const int bn = tile_n(ctx, M, N, 1, cl, EPI == Epi::F32);
  return bf16 ? dispatch<true, EPI>(ctx, pdl, bn, cl, M, N, K, A, lda, B, ldb,
                                    C, ldc, D, ldd)
              : dispatch<false, EPI>(ctx, pdl, bn, cl, M, N, K, A, lda, B,
                                     ldb, C, ldc, D, ldd);
}

mma_status_t launch_gemm_tc_f16(const Ctx& ctx, bool bf16, bool out16,
                                int64_t M, int64_t N, int64_t K, const void* A,
                                int64_t lda, const void* B, int64_t ldb,
                                const void* C, int64_t ldc, void* D,
                                int64_t ldd) {
  return out16 ? dispatch_f16<Epi::H16>(ctx, false, bf16, M, N, K, A, lda, B,
                                        ldb, C, ldc, D, ldd)
               : dispatch_f16<Epi::F32>(ctx, false, bf16, M, N, K, A, lda, B,
                                        ldb, C, ldc, D, ldd);
}

size_t gemm_tc_rowb_workspace_bytes(int64_t N, int64_t K) {
  const int64_t ldw = (K + 7) / 8 * 8;
  return size_t(N) * size_t(ldw) * 2;
}

mma_status_t launch_gemm_tc_f16_rowb(const Ctx& ctx, bool bf16, bool out16,
                                     int64_t M, int64_t N, int64_t K,
                                     const void* A, int64_t lda, const void* B,
                                     int64_t ldb, const void* C, int64_t ldc,
                                     void* D, int64_t ldd, void* workspace) {
  const int64_t ldw = (K + 7) / 8 * 8;
  uint16_t* W = static_cast<uint16_t*>(workspace);
  const mma_status_t st = launch_transpose_b<false>(ctx, B, ldb, K, N, W, ldw);
  if (st != MMA_OK) return st;
  return out16 ? dispatch_f16<Epi::H16>(ctx, true, bf16, M, N, K, A, lda, W,
                                        ldw, C, ldc, D, ldd)
               : dispatch_f16<Epi::F32>(ctx, true, bf16, M, N, K, A, lda, W,
                                        ldw, C, ldc, D, ldd);
}

size_t gemm_i8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int64_t ldw = (K + 7) / 8 * 8;
  // BF16 copies of A and B, then the 64-bit correction terms
  return size_t(M + N) * size_t(ldw) * 2 + size_t(M + N) * 8;
}

mma_status_t launch_gemm_i8_tc(const Ctx& ctx, int64_t M, int64_t N,
                               int64_t K, const int8_t* A, int64_t lda,
                               const int8_t* B, int64_t ldb, const int32_t* C,
                               int64_t ldc, int32_t* D, int64_t ldd,
                               void* workspace, bool b_row_major,
                               bool a_signed, bool b_signed, bool clamp) {
  const int64_t ldw = (K + 7) / 8 * 8;
  uint16_t* W = static_cast<uint16_t*>(workspace);
  uint16_t* Bw = W + M * ldw;
  // Offsets of the stored values (128 for an unsigned operand) and the
  // correction terms they need (see widen_rows_kernel).
  const int64_t oa = a_signed ? 0 : 128, ob = b_signed ? 0 : 128;
  int64_t* terms = reinterpret_cast<int64_t*>(W + (M + N) * ldw);
  int64_t* row_term = ob ? terms : nullptr;
  int64_t* col_term = oa ? terms + M : nullptr;
  const uint32_t flip_a = a_signed ? kFlipSigned : 0u;
  const uint32_t flip_b = b_signed ? kFlipSigned : 0u;
  if (b_row_major) {
    // B widened while transposed (its column sums gathered by atomics into
    // a zeroed col_term); the A pass below then runs last, so the GEMM's
    // programmatic dependency is on it (and on B by stream order).
    if (col_term &&
        cudaMemsetAsync(col_term, 0, size_t(N) * 8, ctx.stream) != cudaSuccess)
      return MMA_ERR_LAUNCH;
    const mma_status_t st = launch_transpose_b<true>(ctx, B, ldb, K, N, Bw,
                                                     ldw, flip_b, col_term, oa);
    if (st != MMA_OK) return st;
  }
  const int64_t nb = b_row_major ? 0 : N;
  if (oa == 0 && ob == 0) {
    const int64_t chunks = (M + nb) * ((K + 15) / 16);
    const int64_t span = int64_t(kConvThreads) * kConvUnroll;
    int64_t blocks = (chunks + span - 1) / span;
    if (blocks > int64_t(ctx.num_sms) * 8) blocks = int64_t(ctx.num_sms) * 8;
    i8_to_bf16_kernel<<<int(blocks), kConvThreads, 0, ctx.stream>>>(
        A, lda, int(M), B, ldb, int(nb), int(K), W, ldw);
  } else {
    // lanes per row: enough that each lane has about four 16-byte chunks
    const int64_t cpr = (K + 15) / 16;
    int G = 1;
    while (G < 32 && int64_t(G) * 4 < cpr) G *= 2;
    const int64_t warps = ((M + nb) * G + 31) / 32;
    int64_t blocks = (warps + kRowThreads / 32 - 1) / (kRowThreads / 32);
    if (blocks > int64_t(ctx.num_sms) * 8) blocks = int64_t(ctx.num_sms) * 8;
    widen_rows_kernel<<<int(blocks), kRowThreads, 0, ctx.stream>>>(
        reinterpret_cast<const uint8_t*>(A), lda, int(M),
        reinterpret_cast<const uint8_t*>(B), ldb, int(nb), int(K), W, ldw,
        flip_a, flip_b, G, row_term, ob, oa * ob * K,
        b_row_major ? nullptr : col_term, oa);
  }
  if (cudaGetLastError() != cudaSuccess) return MMA_ERR_LAUNCH;
  const int cl = cluster_size(ctx, M, N, K);
  if (clamp) {
    // C joins the INT32 sums while the chunks run (as in the exact mode)
    // when the exact product's magnitude stays below 2^30, on 224-wide
    // pair tiles, from three chunks per tile up.
    const int bn = tile_n(ctx, M, N, 1, cl, true);
    const double amax = a_signed ? 128.0 : 255.0;
    const double bmax = b_signed ? 128.0 : 255.0;
    if (cl == 2 && bn == 224 && K > 2 * kI8ChunkK &&
        double(K) * amax * bmax < 1073741824.0)
      return dispatch<true, Epi::I32SATE>(ctx, true, bn, cl, M, N, K, W, ldw,
                                          Bw, ldw, C, ldc, D, ldd, row_term,
                                          col_term);
    // Largest magnitude of any partial INT32 sum when the sums start from
    // the correction terms: each chunk adds at most 2^24, and
    // |row term| + |column term| <= K * (128 ob + 128 oa + oa ob).
    const double reach = double((K + kI8ChunkK - 1) / kI8ChunkK) * 16777216.0 +
                         double(K) * double(128 * ob + 128 * oa + oa * ob);
    if (reach < 2147483647.0)
      return dispatch<true, Epi::I32SATW>(ctx, true,
                                          tile_n(ctx, M, N, 1, cl, true), cl,
                                          M, N, K, W, ldw, Bw, ldw, C, ldc, D,
                                          ldd, row_term, col_term);
    return dispatch<true, Epi::I32SAT>(ctx, true, 128, cl, M, N, K, W, ldw,
                                       Bw, ldw, C, ldc, D, ldd, row_term,
                                       col_term);
  }
  return dispatch<true, Epi::I32EXACT>(ctx, true, tile_n(ctx, M, N, 1, cl, true),
                                       cl, M, N, K, W, ldw, Bw, ldw, C, ldc, D,
                                       ldd, row_term, col_term);
}

mma_status_t launch_gemm_tc_batched(const Ctx& ctx, bool bf16, bool out16,
                                    int64_t M, int64_t N, int64_t K,
                                    const void* A, int64_t lda, const void* B,
                                    int64_t ldb, const void* C, int64_t ldc,
                                    void* D, int64_t ldd, int64_t batch,
                                    int group, int abid, int blgp) {
  if (batch > int64_t(INT32_MAX)) return MMA_ERR_UNSUPPORTED;
  const BatchArgs bat{int(batch), group, abid, blgp};
  const int cl = cluster_size(ctx, M, N, K, batch);
  const int bn = tile_n(ctx, M, N, batch, cl, !out16);
  if (out16)
    return bf16 ? dispatch<true, Epi::H16>(ctx, false, bn, cl, M, N, K, A, lda,
                                           B, ldb, C, ldc, D, ldd, nullptr,
                                           nullptr, bat)
                : dispatch<false, Epi::H16>(ctx, false, bn, cl, M, N, K, A,
                                            lda, B, ldb, C, ldc, D, ldd,
                                            nullptr, nullptr, bat);
  return bf16 ? dispatch<true, Epi::F32>(ctx, false, bn, cl, M, N, K, A, lda, B,
                                         ldb, C, ldc, D, ldd, nullptr, nullptr,
                                         bat)
              : dispatch<false, Epi::F32>(ctx, false, bn, cl, M, N, K, A, lda,
                                          B, ldb, C, ldc, D, ldd, nullptr,
                                          nullptr, bat);
}

size_t gemm_i8_tc_batched_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                          int64_t batch) {
  const int64_t ldw = (K + 7) / 8 * 8;
  return size_t(batch) * size_t(M + N) * size_t(ldw) * 2;
}

mma_status_t launch_gemm_i8_tc_batched(const Ctx& ctx, int64_t M, int64_t N,
                                       int64_t K, const int8_t* A, int64_t lda,
                                       const int8_t* B, int64_t ldb,
                                       const int32_t* C, int64_t ldc,
                                       int32_t* D, int64_t ldd, int64_t batch,
                                       int group, int abid, int blgp,
                                       void* workspace) {
  // The tiles of A (and of B) are contiguous, so `batch` tiles of M rows
  // are one matrix of batch * M rows with leading dimension lda; every tile
  // is widened (the kernel then reads the broadcast sources among them).
  if (batch * (M + N) > int64_t(INT32_MAX) || batch > int64_t(INT32_MAX))
    return MMA_ERR_UNSUPPORTED;
  const int64_t ldw = (K + 7) / 8 * 8;
  uint16_t* W = static_cast<uint16_t*>(workspace);
  uint16_t* Bw = W + batch * M * ldw;
  const int64_t rows_a = batch * M, rows_b = batch * N;
  const int64_t chunks = (rows_a + rows_b) * ((K + 15) / 16);
  const int64_t span = int64_t(kConvThreads) * kConvUnroll;
  int64_t blocks = (chunks + span - 1) / span;
  if (blocks > int64_t(ctx.num_sms) * 8) blocks = int64_t(ctx.num_sms) * 8;
  i8_to_bf16_kernel<<<int(blocks), kConvThreads, 0, ctx.stream>>>(
      A, lda, int(rows_a), B, ldb, int(rows_b), int(K), W, ldw);
  if (cudaGetLastError() != cudaSuccess) return MMA_ERR_LAUNCH;
  const BatchArgs bat{int(batch), group, abid, blgp};
  const int cl = cluster_size(ctx, M, N, K, batch);
  return dispatch<true, Epi::I32EXACT>(ctx, true,
                                       tile_n(ctx, M, N, batch, cl, true), cl,
                                       M, N, K, W, ldw, Bw, ldw, C, ldc, D, ldd,
                                       nullptr, nullptr, bat);
}

mma_status_t launch_gemm_tc_abort_selftest(const Ctx& ctx, int cluster,
                                           int64_t limit_ns, const void* A,
                                           const void* B, void* D) {
  constexpr int64_t n = 256;
  const TestHook hook{static_cast<unsigned long long>(limit_ns), 1};
  const BatchArgs one{1, 1, 0, 0};
  if (cluster == 2)
    return run<128, 6, true, Epi::F32, 2, 4>(ctx, false, n, n, n, A, n, B, n,
                                             nullptr, 0, D, n, kI8ChunkK / BK,
                                             one, nullptr, nullptr, hook);
  return run<128, 5, true, Epi::F32, 1, 4>(ctx, false, n, n, n, A, n, B, n,
                                           nullptr, 0, D, n, kI8ChunkK / BK,
                                           one, nullptr, nullptr, hook);
}

}  // namespace mmagb
