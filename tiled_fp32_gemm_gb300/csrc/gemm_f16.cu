// fp32-accumulating GEMM on 16-bit inputs (fp16 or bf16) on the 5th-generation
// tensor cores: tcgen05.mma kind::f16, accumulator in tensor memory (TMEM),
// operands moved by the Tensor Memory Accelerator (TMA) straight from the
// caller's matrices.
//
// The product is the general form of every other variant,
//     C = alpha * op(A) * op(B) + beta * C      (C fp32, masked to M x N),
// with A and B stored in 16 bits.  The pages announce mixed-precision types
// as their next part ("My Triton From Scratch, Part 18: Shared Memory
// Optimization", section "Next": Part 19, Mixed-Precision Types); the reading
// taken here is 16-bit storage with products and sums in fp32.  A product of
// two 16-bit values is exact in fp32, so only the fp32 accumulation rounds.
//
// Tiles are 128 x BN (BN = 256 or 128) with 64 values of K per stage: one
// 128-byte swizzle row of 16-bit values, so every operand tile sits in
// shared memory in the tensor core's 128-byte-swizzled layout and TMA writes
// it there directly (no packing pass):
//   K-major operand (A as stored, B stored transposed): one box of 64 k x
//     128 (or BN) rows; row r at r * 128 bytes, 8-row atoms 1024 bytes apart.
//   MN-major operand (B as stored, A stored transposed): boxes of 64 m/n x
//     64 k, one per 64 columns of the tile, 8192 bytes apart; k-row r of a
//     box at r * 128 bytes.  The MMA reads it MN-major (instruction
//     descriptor bit), so neither layout is transposed on the way.
// Zero fill: TMA returns 0 for every element outside the matrix, the masked
// load of the pages ("Part 14: Shared Memory Tiles", section "Zero-filled
// boundary tiles"), so ragged M, N and K need no special path.  A caller
// stride TMA cannot take (row pitch not a multiple of 16 bytes, or a base
// not 16-byte aligned) is first copied into a padded scratch matrix.
//
// The persistent kernel: one CTA per SM (192 threads) over units of a
// grouped raster of tiles, with the last partial round split along K:
//   warp 0, one thread: TMA loads of every K tile into a ring of STAGES
//     stages (full[s], expect_tx of the stage's bytes);
//   warp 1, one thread: per K tile 4 tcgen05.mma 128 x BN x 16 into one of
//     two TMEM accumulators, tcgen05.commit -> empty[s]; after the unit's
//     last K tile -> acc_full[b];
//   warps 2-5: drain the other accumulator to C (alpha, beta, mask) while
//     the next unit's MMAs run.
// Every wait is bounded (%globaltimer); on expiry the CTA records
// MT_ERR_TIMEOUT in this kernel's device status word, stops issuing, drains
// what it issued, frees TMEM and returns.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace mt {
namespace f16tc {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;            // 16-bit values of K per stage: one 128-byte row
constexpr int ROW_BYTES = BK * 2;
constexpr int ATOM_BYTES = 8 * ROW_BYTES;
constexpr int MN_BOX = 64;        // M/N values per box of an MN-major operand
constexpr int MN_BOX_BYTES = BK * MN_BOX * 2;
constexpr uint64_t SWIZZLE_128B = 2;  // descriptor layout code
constexpr int THREADS = 192;
constexpr int EPILOGUE_THREADS = 128;
constexpr int SMEM_STAGE_BUDGET = 200 * 1024;

__device__ unsigned int g_status;  // bit 0: a bounded wait expired

template <int BN_>
struct Geometry {
  static_assert(BN_ == 256 || BN_ == 128, "BN is 256 or 128");
  static constexpr int BN = BN_;
  static constexpr int A_BYTES = BM * ROW_BYTES;
  static constexpr int B_BYTES = BN * ROW_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_FIT = SMEM_STAGE_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static_assert(STAGES >= 2, "at least two stages");
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two fp32 accumulators
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*alignment*/ + 256 +
                                   EPI_STAGE_BYTES;
};

// Loads the `rows`-row tile of one operand for K tile k0 into `dst`.
template <int ROWS, bool MN>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, int r0,
                                             int k0, uint32_t bar) {
  if constexpr (!MN) {
    tma_load_2d(dst, map, k0, r0, bar);  // box: 64 k x ROWS rows
  } else {
#pragma unroll
    for (int c = 0; c < ROWS / MN_BOX; ++c)  // boxes: 64 m/n x 64 k
      tma_load_2d(dst + c * MN_BOX_BYTES, map, r0 + c * MN_BOX, k0, bar);
  }
}

// Descriptor of k-step j (16 values of K) of an operand tile at `base`.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int j) {
  if constexpr (!MN)
    return smem_desc(base + j * 32, 16, ATOM_BYTES, SWIZZLE_128B);  // 16 values = 32 bytes
  else
    return smem_desc(base + j * 16 * ROW_BYTES, MN_BOX_BYTES, ATOM_BYTES, SWIZZLE_128B);
}

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(THREADS, 1)
    f16tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_b, uint32_t idesc, Epilogue ep,
                      int Kt, int tiles_m, int tiles_n, int group_m, Sched sched,
                      int fault_inject) {
  using G = Geometry<BN>;
  constexpr int STAGES = G::STAGES;
  constexpr int STAGE_BYTES = G::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars: [0, S) full, [S, 2S) empty, 2S + b acc_full[b], 2S + 2 + b
  // acc_empty[b], 2S + 4 drain.
  constexpr int FULL = 0, EMPTY = STAGES, ACC_FULL = 2 * STAGES, ACC_EMPTY = 2 * STAGES + 2,
                DRAIN = 2 * STAGES + 4, NBARS = 2 * STAGES + 5;
  static_assert(NBARS * 8 + 8 <= 256, "barriers, TMEM slot and abort flag fit 256 bytes");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const WaitCtx wc{abort_flag, &g_status};
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int num_tiles = tiles_m * tiles_n;
  const int cta = static_cast<int>(blockIdx.x), ctas = static_cast<int>(gridDim.x);
  const int num_units = units_of(cta, ctas, sched, num_tiles, Kt);  // this CTA's units

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(FULL + s), 1);   // producer arrival + tx bytes
      mbar_init(bar(EMPTY + s), 1);  // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(ACC_FULL + b), 1);                  // MMA commit
      mbar_init(bar(ACC_EMPTY + b), EPILOGUE_THREADS);  // every epilogue thread
    }
    mbar_init(bar(DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), G::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint32_t issued = 0;  // producer: K tiles issued by this CTA, across its units
  if (warp == 0) {
    if (lane == 0) {
      // Producer.  With fault_inject set it issues nothing, so every wait
      // on its data runs out (the test of the timeout path).
      uint32_t& g = issued;
      bool stop = fault_inject != 0;
      for (int u = 0; u < num_units && !stop; ++u) {
        const Unit w = unit_at(u, cta, ctas, sched, tiles_m, tiles_n, group_m, Kt);
        for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
          const uint32_t s = g % STAGES, round = g / STAGES;
          if (g >= STAGES && !wait_phase(bar(EMPTY + s), (round + 1) & 1u, wc)) {
            stop = true;
            break;
          }
          const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
          mbar_arrive_expect_tx(bar(FULL + s), STAGE_BYTES);
          load_operand<BM, A_MN>(st, &tmap_a, w.tm * BM, kt * BK, bar(FULL + s));
          load_operand<BN, B_MN>(st + G::A_BYTES, &tmap_b, w.tn * BN, kt * BK, bar(FULL + s));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer.
      uint32_t g = 0;
      bool stop = false;
      int it = 0;
      for (int u = 0; u < num_units && !stop; ++u, ++it) {
        const Unit w = unit_at(u, cta, ctas, sched, tiles_m, tiles_n, group_m, Kt);
        const int b = it & 1;
        // The epilogue must have drained this accumulator (used by unit it-2).
        if (it >= 2 && !wait_phase(bar(ACC_EMPTY + b), ((it >> 1) + 1) & 1u, wc)) break;
        tc_fence_after();
        const uint32_t acc_tmem = tmem + static_cast<uint32_t>(b * BN);
        uint32_t acc = 0;
        for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
          const uint32_t s = g % STAGES, round = g / STAGES;
          if (!wait_phase(bar(FULL + s), round & 1u, wc)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t b_base = a_base + G::A_BYTES;
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            mma_f16(acc_tmem, operand_desc<A_MN>(a_base, j), operand_desc<B_MN>(b_base, j),
                    idesc, acc);
            acc = 1;
          }
          mma_commit(bar(EMPTY + s));
        }
        if (!stop) mma_commit(bar(ACC_FULL + b));
      }
      // Every MMA this thread issued has retired once DRAIN completes.
      mma_commit(bar(DRAIN));
      wait_phase(bar(DRAIN), 0, wc, false);
    }
  } else {
    // Epilogue warps: warp w may access TMEM lanes 32*(w%4) .. +31.
    const int q = warp & 3;
    // This warp's staging square, past the barriers.
    float* const epi_square =
        reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256) + q * EPI_WARP_FLOATS;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int it = 0;
    for (int u = 0; u < num_units; ++u, ++it) {
      const int b = it & 1;
      // A unit's accumulator is ready after its whole K loop.  The warp
      // goes on only if every lane saw it (tcgen05.ld needs the whole warp).
      const bool ready = wait_phase(bar(ACC_FULL + b), (it >> 1) & 1u, wc, true,
                                    TIMEOUT_NS + 20000ull * static_cast<uint64_t>(Kt));
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after();
      __syncwarp();
      const Unit w = unit_at(u, cta, ctas, sched, tiles_m, tiles_n, group_m, Kt);
      store_accumulator<BM, BN>(tmem + lane_base + static_cast<uint32_t>(b * BN), w, q, lane,
                                ep, sched.partial, epi_square);
      tc_fence_before();
      mbar_arrive(bar(ACC_EMPTY + b));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // Let the copies the producer issued land before the CTA exits.
    for (uint32_t q = issued > STAGES ? issued - STAGES : 0; q < issued; ++q)
      wait_phase(bar(FULL + q % STAGES), (q / STAGES) & 1u, wc, false);
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair kernel: a cluster of two CTAs on two SMs computes 256 x 256 tiles
// with tcgen05.mma.cta_group::2.  CTA r (0 or 1) of the pair holds rows
// m0 + 128 r .. +127 of A's tile and columns n0 + 128 r .. +127 of B's, so
// each SM stages 32 KB per 64-deep K tile for a 128 x 256 share of the
// product (a single-CTA 128 x 256 tile stages 48 KB for the same share).
//   both CTAs, warp 0: TMA loads of the CTA's halves into its own ring; the
//     bytes of both complete on the even CTA's full[s] (cta_group::2 copies),
//     and only the even CTA arms it (expect_tx of both halves);
//   even CTA, warp 1: per K tile 4 pair MMAs 256 x 256 x 16, then a commit
//     multicast to empty[s] of both CTAs, and after a unit's last K tile to
//     acc_full[b] of both;
//   both CTAs, warps 2-5: drain their own TMEM half (128 rows x 256) to C,
//     then one arrival per warp on the even CTA's acc_empty[b].
// ACC_BUFS accumulators of 256 columns each (1 or 2) sit in TMEM.
constexpr int PAIR_TILE = 256;
constexpr int PAIR_HALF = 128;

template <int ACC_BUFS_>
struct PairGeometry {
  static constexpr int ACC_BUFS = ACC_BUFS_;
  static constexpr int A_BYTES = PAIR_HALF * ROW_BYTES;  // this CTA's half of A
  static constexpr int B_BYTES = PAIR_HALF * ROW_BYTES;  // this CTA's half of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_FIT = SMEM_STAGE_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr uint32_t TMEM_COLS = ACC_BUFS * PAIR_TILE;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*alignment*/ + 256 +
                                   EPI_STAGE_BYTES;
};

template <bool A_MN, bool B_MN, int ACC_BUFS>
__global__ void __launch_bounds__(THREADS, 1)
    f16tc_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_b, uint32_t idesc, Epilogue ep,
                      int Kt, int tiles_m, int tiles_n, int group_m, Sched sched,
                      int fault_inject) {
  using G = PairGeometry<ACC_BUFS>;
  constexpr int STAGES = G::STAGES;
  constexpr int STAGE_BYTES = G::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars: [0, S) full (used on the even CTA), [S, 2S) empty, then
  // acc_full[ACC_BUFS], acc_empty[ACC_BUFS] (used on the even CTA), drain.
  constexpr int FULL = 0, EMPTY = STAGES, ACC_FULL = 2 * STAGES,
                ACC_EMPTY = 2 * STAGES + ACC_BUFS, DRAIN = 2 * STAGES + 2 * ACC_BUFS,
                NBARS = DRAIN + 1;
  static_assert(NBARS * 8 + 8 <= 256, "barriers, TMEM slot and abort flag fit 256 bytes");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const WaitCtx wc{abort_flag, &g_status};
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0: even (MMA issuer), 1: odd
  const bool leader = rank == 0;
  const int cluster = static_cast<int>(cluster_id_x());
  const int clusters = static_cast<int>(cluster_count_x());
  const int num_tiles = tiles_m * tiles_n;
  const int num_units = units_of(cluster, clusters, sched, num_tiles, Kt);  // this cluster's units

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(FULL + s), 1);   // the even CTA's arrival + both CTAs' bytes
      mbar_init(bar(EMPTY + s), 1);  // pair MMA commit
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      mbar_init(bar(ACC_FULL + b), 1);   // pair MMA commit
      mbar_init(bar(ACC_EMPTY + b), 8);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(bar(DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), G::TMEM_COLS);
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // Producer (both CTAs): this CTA's halves into its own stages.
      bool stop = fault_inject != 0;
      uint32_t g = 0;
      for (int u = 0; u < num_units && !stop; ++u) {
        const Unit w = unit_at(u, cluster, clusters, sched, tiles_m, tiles_n, group_m, Kt);
        const int r0a = w.tm * PAIR_TILE + static_cast<int>(rank) * PAIR_HALF;
        const int r0b = w.tn * PAIR_TILE + static_cast<int>(rank) * PAIR_HALF;
        for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
          const uint32_t s = g % STAGES, round = g / STAGES;
          if (g >= STAGES && !wait_phase(bar(EMPTY + s), (round + 1) & 1u, wc)) {
            stop = true;
            break;
          }
          const uint32_t full_even = map_to_cta(bar(FULL + s), 0);
          if (leader) mbar_arrive_expect_tx(bar(FULL + s), 2 * STAGE_BYTES);
          const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
          const int k0 = kt * BK;
          if constexpr (!A_MN) {
            tma_load_2d_pair(st, &tmap_a, k0, r0a, full_even);
          } else {
            tma_load_2d_pair(st, &tmap_a, r0a, k0, full_even);
            tma_load_2d_pair(st + MN_BOX_BYTES, &tmap_a, r0a + MN_BOX, k0, full_even);
          }
          const uint32_t sb = st + G::A_BYTES;
          if constexpr (!B_MN) {
            tma_load_2d_pair(sb, &tmap_b, k0, r0b, full_even);
          } else {
            tma_load_2d_pair(sb, &tmap_b, r0b, k0, full_even);
            tma_load_2d_pair(sb + MN_BOX_BYTES, &tmap_b, r0b + MN_BOX, k0, full_even);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // Pair MMA issuer (even CTA).
      uint32_t g = 0;
      bool stop = false;
      int it = 0;
      for (int u = 0; u < num_units && !stop; ++u, ++it) {
        const Unit w = unit_at(u, cluster, clusters, sched, tiles_m, tiles_n, group_m, Kt);
        const int b = it % ACC_BUFS, use = it / ACC_BUFS;
        // Both CTAs' epilogues must have drained this accumulator.
        if (use >= 1 && !wait_phase(bar(ACC_EMPTY + b), (use + 1) & 1u, wc)) break;
        tc_fence_after();
        const uint32_t acc_tmem = tmem + static_cast<uint32_t>(b * PAIR_TILE);
        uint32_t acc = 0;
        for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
          const uint32_t s = g % STAGES, round = g / STAGES;
          if (!wait_phase(bar(FULL + s), round & 1u, wc)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t b_base = a_base + G::A_BYTES;
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            mma_f16_pair(acc_tmem, operand_desc<A_MN>(a_base, j), operand_desc<B_MN>(b_base, j),
                         idesc, acc);
            acc = 1;
          }
          mma_commit_pair(bar(EMPTY + s), 0x3);
        }
        if (!stop) mma_commit_pair(bar(ACC_FULL + b), 0x3);
      }
      // Every pair MMA issued has retired once DRAIN completes.
      mma_commit_pair(bar(DRAIN), 0x1);
      wait_phase(bar(DRAIN), 0, wc, false);
    }
  } else {
    // Epilogue warps of both CTAs: warp w may access TMEM lanes 32*(w%4)..+31.
    const int q = warp & 3;
    // This warp's staging square, past the barriers.
    float* const epi_square =
        reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256) + q * EPI_WARP_FLOATS;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acc_empty_even = map_to_cta(bar(ACC_EMPTY), 0);
    int it = 0;
    for (int u = 0; u < num_units; ++u, ++it) {
      const int b = it % ACC_BUFS, use = it / ACC_BUFS;
      const bool ready = wait_phase(bar(ACC_FULL + b), use & 1u, wc, true,
                                    TIMEOUT_NS + 20000ull * static_cast<uint64_t>(Kt));
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after();
      __syncwarp();
      const Unit w = unit_at(u, cluster, clusters, sched, tiles_m, tiles_n, group_m, Kt);
      store_accumulator<PAIR_HALF, PAIR_TILE, PAIR_TILE>(
          tmem + lane_base + static_cast<uint32_t>(b * PAIR_TILE), w, q, lane, ep,
          sched.partial, epi_square, static_cast<int>(rank) * PAIR_HALF);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_even + 8u * static_cast<uint32_t>(b));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Copies this CTA issued complete on the even CTA's barriers, which it
    // cannot wait on: give any still in flight time to land (bounded).
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 200000ull) {
    }
  }
  // The even CTA's MMAs (which read the odd CTA's shared memory) have
  // retired and every cross-CTA arrival is done before either CTA leaves.
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, G::TMEM_COLS);
  }
}

// dst[r * ldd + c] = src[r * lds + c] for c < cols, 0 for cols <= c < ldd
// (16-bit values; ldd % 8 == 0 and dst 16-byte aligned, one 16-byte store
// per thread and step).
__global__ void __launch_bounds__(256) repack16_kernel(const uint16_t* __restrict__ src,
                                                       int64_t lds, uint16_t* __restrict__ dst,
                                                       int64_t ldd, int64_t rows, int64_t cols,
                                                       BoundsRecord* rec) {
  const int64_t per_row = ldd / 8;
  const int64_t total = rows * per_row;
  const int64_t src_extent = view_extent(rows, cols, lds), dst_extent = rows * ldd;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = e / per_row, c0 = (e % per_row) * 8;
    const uint16_t* s = src + r * lds;
    uint16_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      v[i] = c0 + i < cols && bounds_ok(rec, SITE_PREP_SRC, r * lds + c0 + i, 1, src_extent)
                 ? s[c0 + i]
                 : static_cast<uint16_t>(0);
    uint4 o;
    o.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
    o.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
    o.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
    o.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
    if (bounds_ok(rec, SITE_PREP_DST, r * ldd + c0, 8, dst_extent))
      *reinterpret_cast<uint4*>(dst + r * ldd + c0) = o;
  }
}

}  // namespace f16tc

// ---------------------------------------------------------------------------
// Host side.

namespace {

using f16tc::BK;
using f16tc::BM;

// 2-D map of a stored rows x cols matrix of 16-bit values (row pitch ld
// values), box of box_cols x box_rows, 128-byte swizzle, zero fill.
bool encode_map(CUtensorMap* map, int dtype, const void* base, int64_t rows, int64_t cols,
                int64_t ld, int box_cols, int box_rows) {
  return encode_tensor_map_2d(
      map, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
      base, rows, cols, ld, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Row pitch (elements) of a repacked 16-bit operand: whole 128-byte lines,
// so every row TMA reads starts on a line.
int64_t repack_pitch(int64_t cols) { return (cols + 63) / 64 * 64; }

// Operands TMA cannot read in place go through padded copies in the
// workspace; returns the matrices and leading dimensions to read.
// The staged epilogue (tc::store_accumulator) where it pays: rows of C that
// are not float4-aligned, or C of 2^20 elements or more.  Measured on GB300
// (single calls, L2 flushed), staged against not: 4097 x 3001 x 2053 67.2
// against 123.6 us, 4096^3 91.3 against 97.4 us, 1024^3 15.0 against 15.0
// us, but 100 x 72 x 80 (one tile) 10.9 against 8.8 us.
bool staged_epilogue(const GemmArgs& a, bool vec_c) {
  return !vec_c || static_cast<int64_t>(a.M) * a.N >= (int64_t(1) << 20);
}

cudaError_t repack_operands(const GemmArgs& a, const F16Operands& f, const F16Layout& L,
                            char* ws, const void** A, int64_t* lda, const void** B,
                            int64_t* ldb, cudaStream_t stream) {
  *A = f.A;
  *lda = a.lda;
  *B = f.B;
  *ldb = a.ldb;
  if (L.repack_a_bytes) {
    const int64_t rows = a.trans_a ? a.K : a.M, cols = a.trans_a ? a.M : a.K;
    const int64_t ldd = repack_pitch(cols);
    f16tc::repack16_kernel<<<1216, 256, 0, stream>>>(static_cast<const uint16_t*>(f.A), a.lda,
                                                     reinterpret_cast<uint16_t*>(ws), ldd, rows,
                                                     cols, a.bounds);
    *A = ws;
    *lda = ldd;
  }
  if (L.repack_b_bytes) {
    const int64_t rows = a.trans_b ? a.N : a.K, cols = a.trans_b ? a.K : a.N;
    const int64_t ldd = repack_pitch(cols);
    uint16_t* dst = reinterpret_cast<uint16_t*>(ws + L.repack_a_bytes);
    f16tc::repack16_kernel<<<1216, 256, 0, stream>>>(static_cast<const uint16_t*>(f.B), a.ldb,
                                                     dst, ldd, rows, cols, a.bounds);
    *B = dst;
    *ldb = ldd;
  }
  return cudaGetLastError();
}

template <int BN>
struct Cfg16 {
  using G = f16tc::Geometry<BN>;

  template <bool A_MN, bool B_MN>
  static constexpr auto kernel() {
    return f16tc::f16tc_gemm_kernel<BN, A_MN, B_MN>;
  }

  static cudaError_t prepare() {
    cudaError_t e = cudaSuccess;
    const void* ks[4] = {reinterpret_cast<const void*>(kernel<false, false>()),
                         reinterpret_cast<const void*>(kernel<false, true>()),
                         reinterpret_cast<const void*>(kernel<true, false>()),
                         reinterpret_cast<const void*>(kernel<true, true>())};
    for (const void* k : ks) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
      if (e != cudaSuccess) return e;
    }
    return e;
  }

  static cudaError_t launch(const GemmArgs& a, const F16Operands& f, void* workspace,
                            bool vec_c, int max_ctas, int fault_inject, cudaStream_t stream) {
    const int mt = (a.M + BM - 1) / BM, nt = (a.N + BN - 1) / BN, kt = (a.K + BK - 1) / BK;
    const F16Layout L = f16tc_layout(a, f, BM, BN);
    char* ws = static_cast<char*>(workspace);
    const void* A;
    const void* B;
    int64_t lda, ldb;
    cudaError_t e = repack_operands(a, f, L, ws, &A, &lda, &B, &ldb, stream);
    if (e != cudaSuccess) return e;
    // A: K-major as stored (M x K), MN-major when stored transposed (K x M).
    // B: MN-major as stored (K x N), K-major when stored transposed (N x K).
    CUtensorMap map_a, map_b;
    const bool a_mn = a.trans_a != 0, b_mn = a.trans_b == 0;
    const bool ok_a = a_mn ? encode_map(&map_a, f.dtype, A, a.K, a.M, lda, f16tc::MN_BOX, BK)
                           : encode_map(&map_a, f.dtype, A, a.M, a.K, lda, BK, BM);
    const bool ok_b = b_mn ? encode_map(&map_b, f.dtype, B, a.K, a.N, ldb, f16tc::MN_BOX, BK)
                           : encode_map(&map_b, f.dtype, B, a.N, a.K, ldb, BK, BN);
    if (!ok_a || !ok_b) return cudaErrorInvalidValue;
    const uint32_t fmt = f.dtype == 1 ? 0u : 1u;  // kind::f16 operand format: f16 0, bf16 1
    const uint32_t idesc = tc::instr_desc(BM, BN, fmt, fmt, a_mn ? 1u : 0u, b_mn ? 1u : 0u);
    const int tiles = mt * nt;
    tc::Sched sched{a.full_tiles, a.split, a.kt_per_slice, nullptr, a.sk_ctas, a.sk_iters};
    if (a.split > 1 || a.sk_ctas > 0)
      sched.partial = reinterpret_cast<float*>(ws + L.partial_offset);
    const int units = a.full_tiles + (tiles - a.full_tiles) * a.split;
    const int grid = persistent_grid(a, units, max_ctas);
    const tc::Epilogue ep =
        tc::make_epilogue(a, vec_c, tiles, BM, BN, staged_epilogue(a, vec_c));
    const int smem = tc::epilogue_smem(G::SMEM_BYTES, ep);
    auto go = [&](auto kern) {
      kern<<<grid, f16tc::THREADS, smem, stream>>>(map_a, map_b, idesc, ep, kt, mt, nt,
                                                   a.group_m, sched, fault_inject);
    };
    if (!a_mn && !b_mn) go(kernel<false, false>());
    else if (!a_mn && b_mn) go(kernel<false, true>());
    else if (a_mn && !b_mn) go(kernel<true, false>());
    else go(kernel<true, true>());
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_second_pass(a, sched.partial, BM, BN, kt, vec_c, stream);
  }
};

// Accumulators of the pair kernel in TMEM (256 columns each).
constexpr int kPairAccBufs = 2;

struct CfgPair {
  using G = f16tc::PairGeometry<kPairAccBufs>;

  template <bool A_MN, bool B_MN>
  static constexpr auto kernel() {
    return f16tc::f16tc_pair_kernel<A_MN, B_MN, kPairAccBufs>;
  }

  static const void* kernel_ptr(bool a_mn, bool b_mn) {
    if (!a_mn && !b_mn) return reinterpret_cast<const void*>(kernel<false, false>());
    if (!a_mn && b_mn) return reinterpret_cast<const void*>(kernel<false, true>());
    if (a_mn && !b_mn) return reinterpret_cast<const void*>(kernel<true, false>());
    return reinterpret_cast<const void*>(kernel<true, true>());
  }

  static cudaError_t prepare() {
    for (int i = 0; i < 4; ++i) {
      const cudaError_t e =
          cudaFuncSetAttribute(kernel_ptr(i & 1, i >> 1),
                               cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }

  // Clusters of two that can be resident at once (the persistent grid).
  static int max_clusters() {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(f16tc::THREADS, 1, 1);
    cfg.dynamicSmemBytes = G::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel_ptr(false, true), &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  }

  static cudaError_t launch(const GemmArgs& a, const F16Operands& f, void* workspace,
                            bool vec_c, int max_clusters, int fault_inject, cudaStream_t stream) {
    using f16tc::PAIR_HALF;
    using f16tc::PAIR_TILE;
    const int mt = (a.M + PAIR_TILE - 1) / PAIR_TILE, nt = (a.N + PAIR_TILE - 1) / PAIR_TILE;
    const int kt = (a.K + BK - 1) / BK;
    const void* A;
    const void* B;
    int64_t lda, ldb;
    char* ws = static_cast<char*>(workspace);
    const F16Layout L = f16tc_layout(a, f, PAIR_TILE, PAIR_TILE);
    cudaError_t e = repack_operands(a, f, L, ws, &A, &lda, &B, &ldb, stream);
    if (e != cudaSuccess) return e;
    CUtensorMap map_a, map_b;
    const bool a_mn = a.trans_a != 0, b_mn = a.trans_b == 0;
    // Each CTA loads 128 rows of A's tile and 128 columns of B's.
    const bool ok_a = a_mn ? encode_map(&map_a, f.dtype, A, a.K, a.M, lda, f16tc::MN_BOX, BK)
                           : encode_map(&map_a, f.dtype, A, a.M, a.K, lda, BK, PAIR_HALF);
    const bool ok_b = b_mn ? encode_map(&map_b, f.dtype, B, a.K, a.N, ldb, f16tc::MN_BOX, BK)
                           : encode_map(&map_b, f.dtype, B, a.N, a.K, ldb, BK, PAIR_HALF);
    if (!ok_a || !ok_b) return cudaErrorInvalidValue;
    const uint32_t fmt = f.dtype == 1 ? 0u : 1u;
    const uint32_t idesc =
        tc::instr_desc(PAIR_TILE, PAIR_TILE, fmt, fmt, a_mn ? 1u : 0u, b_mn ? 1u : 0u);
    const int tiles = mt * nt;
    tc::Sched sched{a.full_tiles, a.split, a.kt_per_slice, nullptr, a.sk_ctas, a.sk_iters};
    if (a.split > 1 || a.sk_ctas > 0)
      sched.partial = reinterpret_cast<float*>(ws + L.partial_offset);
    const int units = a.full_tiles + (tiles - a.full_tiles) * a.split;
    const int clusters = persistent_grid(a, units, max_clusters);
    const tc::Epilogue ep =
        tc::make_epilogue(a, vec_c, tiles, PAIR_TILE, PAIR_TILE, staged_epilogue(a, vec_c));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(f16tc::THREADS, 1, 1);
    cfg.dynamicSmemBytes = tc::epilogue_smem(G::SMEM_BYTES, ep);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int group_m = a.group_m;
    void* args[] = {&map_a, &map_b, const_cast<uint32_t*>(&idesc), const_cast<tc::Epilogue*>(&ep),
                    const_cast<int*>(&kt), const_cast<int*>(&mt), const_cast<int*>(&nt),
                    &group_m, &sched, const_cast<int*>(&fault_inject)};
    e = cudaLaunchKernelExC(&cfg, kernel_ptr(a_mn, b_mn), args);
    if (e != cudaSuccess) return e;
    return launch_second_pass(a, sched.partial, PAIR_TILE, PAIR_TILE, kt, vec_c, stream);
  }
};

template <class F>
bool dispatch16(int bn, F&& f) {
  if (bn == 256) { f(Cfg16<256>{}); return true; }
  if (bn == 128) { f(Cfg16<128>{}); return true; }
  return false;
}

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

// Rows x cols of 16-bit values TMA can read in place: 16-byte aligned base,
// row pitch a multiple of 16 bytes.
bool tma_readable(const void* p, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ld % 8 == 0 && ld < (int64_t(1) << 38);
}

}  // namespace

F16Layout f16tc_layout(const GemmArgs& a, const F16Operands& f, int tile_m, int bn) {
  F16Layout L{};
  if (!tma_readable(f.A, a.lda)) {
    const int64_t rows = a.trans_a ? a.K : a.M, cols = a.trans_a ? a.M : a.K;
    L.repack_a_bytes = round256(rows * repack_pitch(cols) * 2);
  }
  if (!tma_readable(f.B, a.ldb)) {
    const int64_t rows = a.trans_b ? a.N : a.K, cols = a.trans_b ? a.K : a.N;
    L.repack_b_bytes = round256(rows * repack_pitch(cols) * 2);
  }
  L.partial_offset = L.repack_a_bytes + L.repack_b_bytes;
  const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  // Partial tiles: two slots per stream-K CTA, or one per slice of a split tile.
  const int64_t partial_tiles =
      a.sk_ctas > 0 ? 2 * static_cast<int64_t>(a.sk_ctas)
                    : (tiles - a.full_tiles) * (a.split > 1 ? a.split : 0);
  L.workspace_bytes = L.partial_offset + partial_tiles * tile_m * bn * 4;
  return L;
}

bool f16tc_valid(int bm, int bn) {
  if (bm == f16tc::PAIR_TILE) return bn == f16tc::PAIR_TILE;
  return bm == BM && dispatch16(bn, [](auto) {});
}

int f16tc_smem_bytes(int bm, int bn) {
  if (bm == f16tc::PAIR_TILE) return CfgPair::G::SMEM_BYTES;
  int r = -1;
  dispatch16(bn, [&](auto c) { r = decltype(c)::G::SMEM_BYTES; });
  return r;
}

int f16tc_stages(int bm, int bn) {
  if (bm == f16tc::PAIR_TILE) return CfgPair::G::STAGES;
  int r = -1;
  dispatch16(bn, [&](auto c) { r = decltype(c)::G::STAGES; });
  return r;
}

namespace {
std::mutex g_pair_mutex;
int g_pair_clusters[64];
}  // namespace

int f16tc_pair_max_clusters(int device) {
  if (device < 0 || device >= 64) return 0;
  std::lock_guard<std::mutex> lock(g_pair_mutex);
  if (g_pair_clusters[device] == 0) {
    if (CfgPair::prepare() != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    g_pair_clusters[device] = CfgPair::max_clusters();
  }
  return g_pair_clusters[device];
}

int f16tc_threads() { return f16tc::THREADS; }
int f16tc_bm() { return f16tc::BM; }
int f16tc_bk() { return f16tc::BK; }

cudaError_t f16tc_prepare(int bm, int bn) {
  if (bm == f16tc::PAIR_TILE) return CfgPair::prepare();
  cudaError_t e = cudaErrorInvalidValue;
  dispatch16(bn, [&](auto c) { e = decltype(c)::prepare(); });
  return e;
}

bool f16tc_encoder_available() { return tensor_map_encoder_available(); }

cudaError_t launch_f16tc(const GemmArgs& a, const F16Operands& f, void* workspace, bool vec_c,
                         int bm, int bn, int max_ctas, int fault_inject, cudaStream_t stream) {
  if (bm == f16tc::PAIR_TILE)
    return CfgPair::launch(a, f, workspace, vec_c, max_ctas, fault_inject, stream);
  cudaError_t e = cudaErrorInvalidValue;
  dispatch16(bn, [&](auto c) {
    e = decltype(c)::launch(a, f, workspace, vec_c, max_ctas, fault_inject, stream);
  });
  return e;
}

cudaError_t f16tc_read_and_clear_status(unsigned int* status) {
  cudaError_t e = cudaMemcpyFromSymbol(status, f16tc::g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(f16tc::g_status, &zero, sizeof(unsigned int));
}

}  // namespace mt
