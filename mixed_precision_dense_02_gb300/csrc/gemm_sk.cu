// tcgen05 GEMM for problems with fewer output tiles than SMs (a tall,
// narrow D such as 16384 x 128 with deep K): D = A * B + C, FP16/BF16
// inputs, FP32 accumulation, A row-major, B column-major, C/D FP32
// row-major.
//
// The K loop of each tile is the caller loop of "CDNA2 dense MFMA
// builtins", section "Naming convention" (each step adds one K panel's
// contribution to the M x N tile).  Here that loop is cut across CTAs so
// that every SM streams operands: the tiles' K steps form one sequence of
// tiles * ceil(K / 64) steps, and CTA c of G takes the contiguous range
// [c * total / G, (c + 1) * total / G) of it ("stream-K").  A range is cut
// at tile boundaries into pieces; a tile is finished by the CTA holding its
// first piece (the one that starts at K step 0):
//   * a piece that does not start at step 0 is always the first piece of
//     its CTA; its FP32 partial sums go to a scratch slot of that CTA,
//     followed by a release flag (the call's sequence number), and the CTA
//     never waits before writing it;
//   * the tile's first piece is its CTA's last piece; that CTA holds its C
//     in registers (requested while the piece's MMAs run), waits for the
//     other pieces' flags (acquire), adds ((acc_first + C) + partial_2) +
//     partial_3 ..., in that fixed order, one FP32 rounding per addition,
//     and stores D.
// The waits only point from a CTA to higher-numbered CTAs, which write
// their partials before waiting on anything, so no cycle of waits exists;
// the sum order depends only on M, N, K and G, so results are identical
// from run to run.  Every wait is bounded (MMA_ERR_TIMEOUT on expiry).
// When G is a whole number of ranges per tile (the host picks such a G
// when it idles at most a quarter of the units), every range lies in one
// tile and all tiles' ranges start at the same K offsets; on pairs every
// unit then stores its partial sums and the tile's units share the final
// additions (same order, same bits), each waiting only for flags that are
// written before any wait.
//
// Roles (320 threads): warp 0 TMA producer (128 x 64 A and B boxes,
// 128-byte swizzle, STAGES-deep ring), warp 1 tcgen05.mma issuer into a
// double-buffered FP32 accumulator in tensor memory, warps 2..9 epilogue
// (two per tensor-memory lane quarter, one per column half): each thread
// owns one row of its warp's columns, handled 64 at a time.
//
// CL = 1: 128 x 128 tiles, one per CTA (M = 128, N = 128 MMAs).
// CL = 2: 256 x 256 tiles on CTA pairs (clusters of two SMs): the pair is
// the unit of the stream-K ranges, each CTA stages 128 rows of A and 128
// of B per K step, the leader's one thread issues cta_group::2 MMAs
// (M = 256, N = 256) whose commits release both CTAs, and each CTA's
// epilogue holds its 128 rows of the tile.  Per SM and K step this moves
// the same 32 KB of operands as CL = 1 for twice the multiply-adds.  A
// tile's partial sums travel between the CTAs of the same rank.
#include <cudaTypedefs.h>

#include <cstdlib>

#include "kernels.h"
#include "ptx.cuh"

namespace mmagb {
namespace {

constexpr int kBM = 128;  // rows per CTA
constexpr int kBK = 64;
constexpr int kUK = 16;
constexpr int kEpi = 8;                     // epilogue warps
constexpr int kThreadsSK = 64 + 32 * kEpi;  // 320
constexpr int kPart = 64;                   // columns per epilogue pass
constexpr int kBlk = kPart / 16;            // 16-column blocks per pass
constexpr int kStages = 6;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kStageBytes = kABytes + 128 * kBK * 2;  // 128 rows of B
constexpr int kBarOffset = kStages * kStageBytes;
constexpr int kSmemBytes = kBarOffset + (2 * kStages + 5) * 8 + 16 + 1024;
// Tile of CL CTAs: (128 CL) x (128 CL); per CTA 128 x 128 CL accumulators.
template <int CL>
constexpr int kTileN = 128 * CL;
// FP32 partial sums of one CTA's piece: its 128 rows of the tile
template <int CL>
constexpr int kSlotFloats = kBM * kTileN<CL>;

// First K step (of the whole sequence) of CTA c's range.
__host__ __device__ __forceinline__ int64_t range_begin(int64_t c,
                                                        int64_t total,
                                                        int64_t grid) {
  return c * total / grid;
}

// The CTA whose range holds step x.
__device__ __forceinline__ int64_t owner_of(int64_t x, int64_t total,
                                            int64_t grid) {
  int64_t c = x * grid / total;
  while (c + 1 < grid && range_begin(c + 1, total, grid) <= x) ++c;
  while (c > 0 && range_begin(c, total, grid) > x) --c;
  return c;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until *flag == seq (bounded like mbar_wait: on expiry raise the
// CTA's abort flag and record MMA_ERR_TIMEOUT).
__device__ __forceinline__ bool wait_flag(const unsigned* flag, unsigned seq,
                                          volatile int* abort_flag,
                                          unsigned* status) {
  if (ld_acquire_u32(flag) == seq) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_u32(flag) == seq) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Piece of CTA c's range starting at step s: tile t, K steps [k0, k1).
struct Piece {
  int t, k0, k1;
};

__device__ __forceinline__ Piece piece_at(int64_t s, int64_t end, int nk) {
  Piece p;
  p.t = int(s / nk);
  p.k0 = int(s - int64_t(p.t) * nk);
  const int64_t room = end - s;
  p.k1 = room < int64_t(nk - p.k0) ? p.k0 + int(room) : nk;
  return p;
}

template <bool BF16, int CL>
__global__ void __launch_bounds__(kThreadsSK, 1)
    gemm_sk_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const float* C, int64_t ldc, float* D, int64_t ldd, int M,
                   int N, int K, float* __restrict__ partials,
                   unsigned* __restrict__ flags, unsigned seq,
                   int shared_ranges, unsigned* status) {
  constexpr int TN = kTileN<CL>;    // tile columns
  constexpr int TM = kBM * CL;      // tile rows
  constexpr int HALF = TN / 2;      // columns per epilogue warp
  constexpr int NP = HALF / kPart;  // 64-column passes per warp
  constexpr uint32_t kTmemCols = 2 * TN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int num_m = (M + TM - 1) / TM;
  const int nk = (K + kBK - 1) / kBK;
  const int64_t tiles = int64_t(num_m) * ((N + TN - 1) / TN);
  const int64_t total = tiles * nk;
  // the unit of the ranges: one CTA, or one pair
  const int64_t grid = gridDim.x / CL;
  const int64_t unit = blockIdx.x / CL;
  const int rank = CL > 1 ? int(cluster_ctarank()) : 0;
  const int64_t beg = range_begin(unit, total, grid);
  const int64_t end = range_begin(unit + 1, total, grid);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], CL * kEpi);  // every epilogue warp of the tile
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
    if constexpr (CL == 1) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(tmem_slot, kTmemCols);
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
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      // the leader CTA's full barriers, which count both CTAs' bytes
      const uint32_t full_lead =
          CL > 1 ? mapa_shared(smem_u32(&full[0]), 0) : 0u;
      for (int64_t s = beg; s < end && ok;) {
        const Piece p = piece_at(s, end, nk);
        const int mb = p.t % num_m, nb = p.t / num_m;
        for (int kb = p.k0; kb < p.k1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * kStageBytes;
          if constexpr (CL == 1) {
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            tma_load_3d(&tmA, &full[stage], sa, kb * kBK, mb * kBM, 0);
            tma_load_3d(&tmB, &full[stage], sa + kABytes, kb * kBK, nb * TN, 0);
          } else {
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], CL * kStageBytes);
            const uint32_t fb = full_lead + uint32_t(stage) * 8u;
            tma_load_3d_pair(&tmA, fb, sa, kb * kBK, mb * TM + rank * kBM, 0);
            tma_load_3d_pair(&tmB, fb, sa + kABytes, kb * kBK,
                             nb * TN + rank * 128, 0);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        s += p.k1 - p.k0;
      }
      for (int st = 0; st < kStages; ++st) {
        const uint32_t fills =
            issued / kStages + (uint32_t(st) < issued % kStages);
        if (!fills) continue;
        // on abort, let every load still in flight land before exiting (the
        // leader's full barriers also count the peer's loads)
        if (!ok && rank == 0) {
          const uint32_t a = smem_u32(&full[st]);
          const unsigned long long t0 = global_timer_ns();
          while (!mbar_try_wait(a, (fills - 1) & 1u))
            if (global_timer_ns() - t0 > kWaitLimitNs) break;
        }
        // with a pair, the last release of each stage is the leader's
        // commit: wait until it has arrived on this CTA
        if (CL > 1) {
          const uint32_t a = smem_u32(&empty[st]);
          const unsigned long long t0 = global_timer_ns();
          while (!mbar_try_wait(a, (fills - 1) & 1u))
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              atomicOr(status, kStatusTimeout);
              break;
            }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // (with a pair, only the leader CTA issues)
    if (rank == 0 && elect_one()) {
      constexpr uint32_t idesc = idesc_f16_f32(BF16, TM, TN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int64_t s = beg; s < end && ok;) {
        const Piece p = piece_at(s, end, nk);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * TN);
        for (int kb = p.k0; kb < p.k1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint64_t da = sw128_kmajor_desc(sa);
          const uint64_t db = sw128_kmajor_desc(sa + kABytes);
#pragma unroll
          for (int k = 0; k < kBK / kUK; ++k) {
            const uint32_t accum = (kb != p.k0 || k != 0) ? 1u : 0u;
            if constexpr (CL == 1)
              umma_f16(d_tmem, da + uint64_t(2 * k), db + uint64_t(2 * k),
                       idesc, accum);
            else
              umma_f16_pair(d_tmem, da + uint64_t(2 * k), db + uint64_t(2 * k),
                            idesc, accum);
          }
          if constexpr (CL == 1)
            umma_commit(&empty[stage]);
          else
            umma_commit_pair(&empty[stage], 3u);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (CL == 1)
          umma_commit(&tfull[acc]);
        else
          umma_commit_pair(&tfull[acc], 3u);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        s += p.k1 - p.k0;
      }
      // every MMA issued above completes before tensor memory is released
      if constexpr (CL == 1)
        umma_commit(done);
      else
        umma_commit_pair(done, 1u);
      const uint32_t a = smem_u32(done);
      const unsigned long long t0 = global_timer_ns();
      while (!mbar_try_wait(a, 0))
        if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue warps
    const int ew = warp - 2;   // 0 .. 7
    const int q = warp & 3;    // tensor-memory lane quarter
    const int h = ew >> 2;     // column half
    const int lane = threadIdx.x & 31;
    // this CTA's partial-sum slot and flags, and those of the CTAs of the
    // same rank in later units
    const int64_t me = unit * CL + rank;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    // (lane) 64 values of C's row `row` from column cc0 into v
    auto load_c = [&](int row, int cc0, float (&v)[kPart]) {
      const bool live = C != nullptr && row < M;
      const float* crow = live ? C + int64_t(row) * ldc : nullptr;
#pragma unroll
      for (int c = 0; c < kPart / 4; ++c) {
        const int cc = cc0 + 4 * c;
        float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && cc + 4 <= N) {
          w = *reinterpret_cast<const float4*>(crow + cc);
        } else if (live) {
          if (cc < N) w.x = crow[cc];
          if (cc + 1 < N) w.y = crow[cc + 1];
          if (cc + 2 < N) w.z = crow[cc + 2];
        }
        v[4 * c] = w.x;
        v[4 * c + 1] = w.y;
        v[4 * c + 2] = w.z;
        v[4 * c + 3] = w.w;
      }
    };
    // this warp's partial sums (its rows and HALF columns) to this CTA's
    // slot, laid out so that each warp-wide 16-byte store covers 512
    // contiguous bytes; then its release flag
    auto write_partial = [&](uint32_t taddr) {
      float4* slot = reinterpret_cast<float4*>(partials) +
                     (me * kEpi + ew) * (NP * kBlk * 4 * 32);
#pragma unroll
      for (int j = 0; j < NP * kBlk; ++j) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr + uint32_t(j * 16), r);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          slot[(j * 4 + c) * 32 + lane] =
              make_float4(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1]),
                          __uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3]));
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release_u32(&flags[me * kEpi + ew], seq);
    };
    // v += the pass `part` of unit o's partial sums in this warp's region
    // (after its flag), all of its 16-byte pieces in flight at once
    auto add_partial = [&](int64_t o, int part, float (&v)[kPart]) -> bool {
      const int64_t other = o * CL + rank;
      const bool okf = wait_flag(&flags[other * kEpi + ew], seq, abort_flag, status);
      if (!__all_sync(0xffffffffu, okf)) return false;
      const float4* slot = reinterpret_cast<const float4*>(partials) +
                           (other * kEpi + ew) * (NP * kBlk * 4 * 32) +
                           part * (kBlk * 4 * 32);
      float4 w[kPart / 4];
#pragma unroll
      for (int c = 0; c < kPart / 4; ++c) w[c] = __ldcg(&slot[c * 32 + lane]);
#pragma unroll
      for (int c = 0; c < kPart / 4; ++c) {
        v[4 * c] += w[c].x;
        v[4 * c + 1] += w[c].y;
        v[4 * c + 2] += w[c].z;
        v[4 * c + 3] += w[c].w;
      }
      return true;
    };
    // (lane) this row's 64 values from column cc0 to D
    auto store_d = [&](int row, int cc0, const float (&v)[kPart]) {
      if (row >= M) return;
      float* drow = D + int64_t(row) * ldd;
#pragma unroll
      for (int c = 0; c < kPart / 4; ++c) {
        const int cc = cc0 + 4 * c;
        if (cc + 4 <= N) {
          *reinterpret_cast<float4*>(drow + cc) =
              make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        } else {
          for (int e = 0; e < 4 && cc + e < N; ++e) drow[cc + e] = v[4 * c + e];
        }
      }
    };
    // This warp's accumulator reads are done (to the leader CTA's barrier
    // for a pair).
    auto release_acc = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CL == 1)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    };
    for (int64_t s = beg; s < end && ok;) {
      const Piece p = piece_at(s, end, nk);
      const int mb = p.t % num_m, nb = p.t / num_m;
      const int row = mb * TM + rank * kBM + q * 32 + lane;
      const int colh = nb * TN + h * HALF;
      if (shared_ranges > 1) {
        // Every tile is cut into shared_ranges whole ranges, one piece
        // each: every unit stores its partial sums, then finishes a share
        // of its tile -- the (warp region, 64-column pass) items whose
        // index modulo shared_ranges is its position in the tile -- as
        // (((C + partial_0) + partial_1) + ...) in unit order, the same
        // order (and bits) as a single finishing unit would add them in.
        const int P = shared_ranges;
        ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        write_partial(tmem_base + uint32_t(acc * TN + h * HALF) +
                      (uint32_t(q * 32) << 16));
        release_acc();
        const int64_t first = int64_t(p.t) * P;  // the tile's first unit
        const int pos = int(unit - first);
        for (int part = 0; part < NP && ok; ++part) {
          if ((ew * NP + part) % P != pos) continue;
          float v[kPart];
          load_c(row, colh + part * kPart, v);
          for (int k = 0; k < P && ok; ++k) ok = add_partial(first + k, part, v);
          if (ok) store_d(row, colh + part * kPart, v);
        }
        s += p.k1 - p.k0;
        continue;
      }
      const bool head = p.k0 == 0;
      const bool whole = head && p.k1 == nk;
      // The tile's other pieces (only for a first piece that is not the
      // whole tile): units unit + 1 .. last, each holding it as its first.
      int64_t last = unit;
      if (head && !whole) last = owner_of(int64_t(p.t) * nk + nk - 1, total, grid);
      // A first piece adds C: the first pass's 64 values of it are
      // requested now, while the piece's MMAs run, and held in registers.
      float v[kPart];
      if (head) load_c(row, colh, v);
      ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + uint32_t(acc * TN + h * HALF) + (uint32_t(q * 32) << 16);
      if (!head) {
        write_partial(taddr);
      } else {
        // D = ((acc + C) + partial of unit + 1) + partial of unit + 2 ...:
        // a fixed order, one FP32 rounding per addition; 64 columns a pass
        for (int part = 0; part < NP && ok; ++part) {
          if (part > 0) load_c(row, colh + part * kPart, v);
#pragma unroll
          for (int j = 0; j < kBlk; ++j) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(taddr + uint32_t((part * kBlk + j) * 16), r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[16 * j + e] += __uint_as_float(r[e]);
          }
          for (int64_t o = unit + 1; o <= last && ok; ++o)
            ok = add_partial(o, part, v);
          if (!ok) break;
          store_d(row, colh + part * kPart, v);
        }
        if (!ok) break;
      }
      release_acc();
      s += p.k1 - p.k0;
    }
  }

  tc_fence_before();
  if constexpr (CL > 1)
    cluster_sync();  // neither CTA leaves while the other may still signal it
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CL == 1)
      tmem_dealloc(tmem_base, kTmemCols);
    else
      tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

// Stream-K applies to FP32-result products whose 128 x 128 tiles are fewer
// than half the SMs, with at least two K steps per CTA on average and at
// least eight per tile, and either at most a quarter of the SMs busy on the
// regular kernel or at least 128 K steps per tile: the split only pays when
// the MMAs outweigh the fixed cost of a call and the partial-sum hand-off
// (3000 x 256 x 2048: 23.2 us split, 13.5 us regular; 1024 x 1024 x 4096:
// 25.1 against 21.5 us; 4096 x 128 x 4096: 19.0 against 22.9 us).
// MMA_GB300_STREAMK=0 turns it off, =1 on wherever the sizes allow it, for
// tuning.
bool gemm_sk_fits(int num_sms, int64_t M, int64_t N, int64_t K) {
  static const int forced = [] {
    const char* e = getenv("MMA_GB300_STREAMK");
    if (!e) return -1;
    return e[0] == '0' ? 0 : 1;
  }();
  if (forced == 0 || M <= 0 || N <= 0 || K <= 0) return false;
  const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + 127) / 128);
  const int64_t nk = (K + kBK - 1) / kBK;
  if (tiles * nk >= (int64_t(1) << 31)) return false;
  if (forced == 1) return tiles * nk >= 2 && tiles < (int64_t(1) << 31);
  return 2 * tiles < num_sms && nk >= 8 && tiles * nk >= 2 * int64_t(num_sms) &&
         (4 * tiles <= num_sms || nk >= 128);
}

size_t gemm_sk_workspace_bytes(int num_sms) {
  // slots for either tile shape
  return size_t(num_sms) * kSlotFloats<2> * sizeof(float);
}

size_t gemm_sk_flag_count(int num_sms) { return size_t(num_sms) * kEpi; }

namespace {

template <bool BF16, int CL>
mma_status_t launch_sk(const Ctx& ctx, int64_t M, int64_t N, int64_t K,
                       const void* A, int64_t lda, const void* B, int64_t ldb,
                       const float* C, int64_t ldc, float* D, int64_t ldd,
                       float* partials, unsigned* flags, unsigned seq) {
  CUtensorMap ta, tb;
  if (!make_kmajor_map(&ta, A, K, M, lda, kBM, BF16) ||
      !make_kmajor_map(&tb, B, K, N, ldb, 128, BF16))
    return MMA_ERR_LAUNCH;
  auto kern = gemm_sk_kernel<BF16, CL>;
  static PerContext<bool> smem_attr;
  bool attr_ok = false;
  if (!smem_attr.get(ctx, &attr_ok, [&](bool* v) {
        *v = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSmemBytes) == cudaSuccess;
        if (!*v) cudaGetLastError();
        return *v;
      }))
    return MMA_ERR_LAUNCH;
  constexpr int TN = kTileN<CL>;
  const int64_t tiles = ((M + kBM * CL - 1) / (kBM * CL)) * ((N + TN - 1) / TN);
  const int64_t total = tiles * ((K + kBK - 1) / kBK);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreadsSK, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // units (CTAs or pairs) resident at once: every unit may wait on a later
  // one, so the grid never exceeds them
  int64_t units = ctx.num_sms / CL;
  if (CL > 1) {
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
    units = r;
  }
  if (units > total) units = total;
  // With a whole number of ranges per tile, every tile's ranges start at
  // the same K offsets, so the tiles that share an A or B panel read each
  // K chunk of it at about the same time: one DRAM fetch, the other reads
  // L2 hits.  Whole ranges are used when they leave at most a quarter of
  // the units idle (1024 x 1024 x 32768: 64 of 76 pairs, 66.1 -> 59.2 us;
  // single CTAs 128 of 152, 68.6 -> 62.0 us).
  const int64_t per_tile = units / tiles;
  if (per_tile >= 1 && 4 * per_tile * tiles >= 3 * units) units = per_tile * tiles;
  // With whole ranges every unit holds one piece of one tile.  On pairs
  // the tile's units then finish it together (each adds the partial sums
  // of a share of the tile) instead of its first unit alone, whose warps
  // would each add (ranges - 1) partial blocks twice (two 64-column
  // passes) one after another: 1024 x 768 x 8192 35.7 -> 30.9 us, deep-K
  // 59.1 -> 57.9 us.  On single CTAs (one pass) sharing only lengthens
  // each warp's chain of dependent loads (4096 x 128 x 4096 18.1 -> 21.0
  // us), so their first unit finishes alone.
  const int shared_ranges =
      (CL == 2 && units == per_tile * tiles && per_tile > 1) ? int(per_tile) : 0;
  cfg.gridDim = dim3(unsigned(units * CL), 1, 1);
  ctx.mark_start();
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, ta, tb, C, ldc, D, ldd, int(M), int(N),
                         int(K), partials, flags, seq, shared_ranges,
                         ctx.status);
  ctx.mark_stop();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MMA_ERR_LAUNCH;
  }
  return MMA_OK;
}

}  // namespace

// CTA pairs on 256 x 256 tiles when the product is at least one such tile
// in each direction (half-empty pair tiles would waste the pair's operand
// saving) and has enough of them that a tile is cut into at most about 8
// ranges: the CTA finishing a tile adds the other ranges' partial tiles one
// after another (512 x 512 x 65536 on 4 pair tiles, 19 ranges each: 62 us;
// on 16 single-CTA tiles, 9 ranges each: 51 us).  MMA_GB300_STREAMK_CL (1
// or 2) overrides, for tuning.
mma_status_t launch_gemm_sk(const Ctx& ctx, bool bf16, int64_t M, int64_t N,
                            int64_t K, const void* A, int64_t lda,
                            const void* B, int64_t ldb, const float* C,
                            int64_t ldc, float* D, int64_t ldd,
                            float* partials, unsigned* flags, unsigned seq) {
  static const int forced = [] {
    const char* e = getenv("MMA_GB300_STREAMK_CL");
    const int v = e ? atoi(e) : 0;
    return (v == 1 || v == 2) ? v : 0;
  }();
  const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
  const bool pair = forced ? forced == 2
                           : (M >= 256 && N >= 256 &&
                              8 * pair_tiles >= int64_t(ctx.num_sms / 2));
  if (pair)
    return bf16 ? launch_sk<true, 2>(ctx, M, N, K, A, lda, B, ldb, C, ldc, D,
                                     ldd, partials, flags, seq)
                : launch_sk<false, 2>(ctx, M, N, K, A, lda, B, ldb, C, ldc, D,
                                      ldd, partials, flags, seq);
  return bf16 ? launch_sk<true, 1>(ctx, M, N, K, A, lda, B, ldb, C, ldc, D,
                                   ldd, partials, flags, seq)
              : launch_sk<false, 1>(ctx, M, N, K, A, lda, B, ldb, C, ldc, D,
                                    ldd, partials, flags, seq);
}

}  // namespace mmagb
