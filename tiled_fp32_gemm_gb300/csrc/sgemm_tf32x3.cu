// fp32 GEMM on the 5th-generation tensor cores: tcgen05.mma kind::tf32 with
// the 3xTF32 split, accumulator in tensor memory (TMEM).
//
// The product is the same C = A*B as every other variant (row-major, masked
// edges reading 0.0, "My Triton From Scratch, Part 14: Shared Memory Tiles",
// sections "The canonical source pattern" and "Zero-filled boundary tiles").
// The pages stop at CUDA cores ("Part 18", section "What Version 18 does not
// do": no tensor-core instructions); this variant keeps their structure —
// staged, zero-filled shared tiles and a multi-stage K pipeline — and moves
// the dot onto tcgen05.
//
// 3xTF32: a tf32 operand keeps 10 of fp32's 23 mantissa bits.  Each input x
// is split into big = x with the low 13 mantissa bits cleared (exactly
// representable in tf32) and small = x - big (exact in fp32, and its own
// top 11 bits survive the tensor core's tf32 conversion).  Then
//     A*B ~= A_big*B_small + A_small*B_big + A_big*B_big
// (A_small*B_small, about 2^-22 relative, is dropped), accumulated in fp32.
//
// Tiles are 128 x BN (BN = 256, 128 or 64) with a K depth BK of 16 (64-byte
// swizzle) or 32 (128-byte swizzle) per pipeline stage.
//   pack kernels (before): A and B are read once, every value is split into
//     big and small, and both halves are written as zero-padded, K-major
//     blocks of 128 (A) or BN (B) rows x BK k, already in the tensor core's
//     swizzled shared-memory order; so the main loop moves each operand
//     pair with one cp.async.bulk, does no arithmetic on the operands and
//     needs no alignment of the caller's leading dimensions.
//   GEMM kernel: persistent, one CTA per SM (192 threads) walking tiles
//     blockIdx.x, blockIdx.x + gridDim.x, ... of a grouped raster;
//     warp 0, one thread: bulk copies of the A and B block pairs of every
//       K tile of every tile into a ring of STAGES stages (full[s]);
//     warp 1, one thread: per K tile, BK/8 k-steps x 3 tcgen05.mma
//       (128 x BN x 8) into one of two TMEM accumulators, tcgen05.commit ->
//       empty[s] (frees the stage), and after a tile's last K tile ->
//       acc_full[b];
//     warps 2-5 (128 threads, TMEM lane quarters 2, 3, 0, 1): wait
//       acc_full[b], tcgen05.ld their 32 lanes (rows), masked stores to C,
//       arrive acc_empty[b] — while the MMAs of the next tile already run
//       into the other accumulator.
// Every wait is bounded (%globaltimer); on expiry the CTA records
// MT_ERR_TIMEOUT in a device status word, stops issuing, drains what it
// issued (again bounded), frees TMEM and returns.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace mt {
namespace tf32x3 {

constexpr int BM = 128;
constexpr int THREADS = 192;
constexpr int EPILOGUE_THREADS = 128;
using namespace tc;
constexpr int SMEM_STAGE_BUDGET = 200 * 1024;   // shared memory for the operand ring

__device__ unsigned int g_status;  // bit 0: a bounded wait expired

// Shared-memory geometry for tiles of 128 x BN with a K depth of BK fp32
// per stage.  Blocks are K-major: each of the 128 (A) or BN (B) rows holds
// BK consecutive k (ROW_BYTES), rows are grouped by 8 into swizzle atoms,
// and inside an atom the 16-byte chunk index of a row is XOR-ed with the
// row's position — all of it (BK = 32, 128-byte swizzle) or its upper two
// bits (BK = 16, 64-byte swizzle) — the pattern the tensor core applies to
// the address bits when it reads the operand.
template <int BK_, int BN_>
struct Geometry {
  static_assert(BK_ == 32 || BK_ == 16, "BK is 32 or 16");
  static_assert(BN_ == 256 || BN_ == 128 || BN_ == 64, "BN is 256, 128 or 64");
  static constexpr int BK = BK_;
  static constexpr int BN = BN_;
  static constexpr int ROW_BYTES = BK * 4;
  static constexpr int ATOM_BYTES = 8 * ROW_BYTES;
  static constexpr uint32_t CHUNK_MASK = ROW_BYTES / 16 - 1;
  static constexpr uint64_t LAYOUT = BK == 32 ? 2 : 4;  // descriptor: 128-B / 64-B swizzle
  static constexpr int A_BLOCK_BYTES = BM * ROW_BYTES;
  static constexpr int B_BLOCK_BYTES = BN * ROW_BYTES;
  // Packed pairs in global memory and stages in shared memory alike:
  // A big | A small and B big | B small.  Stage: A pair | B pair.
  static constexpr int A_PAIR_BYTES = 2 * A_BLOCK_BYTES;
  static constexpr int B_PAIR_BYTES = 2 * B_BLOCK_BYTES;
  static constexpr int STAGE_BYTES = A_PAIR_BYTES + B_PAIR_BYTES;
  static constexpr int STAGES_FIT = SMEM_STAGE_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static_assert(STAGES >= 2, "at least two stages");
  // Two fp32 accumulators of 128 lanes x BN columns.
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*alignment*/ + 256 /*barriers*/ +
                                   EPI_STAGE_BYTES /*epilogue squares*/;

  // Byte offset of element (r, k), k < BK, inside a block.
  __host__ __device__ static __forceinline__ uint32_t offset(uint32_t r, uint32_t k) {
    const uint32_t r8 = r & 7u;
    const uint32_t x = BK == 32 ? r8 : (r8 >> 1);
    return (r >> 3) * ATOM_BYTES + r8 * ROW_BYTES + ((((k >> 2) ^ x) & CHUNK_MASK) << 4) +
           (k & 3u) * 4u;
  }
};

// ---------------------------------------------------------------------------
// Pack kernels: caller's row-major A, B -> split, swizzled K-major block
// pairs (zero fill).

// big = x with the low 13 mantissa bits cleared; small = x - big (exact).
// Infinities and NaNs keep their bits in big and contribute 0 through small.
__device__ __forceinline__ void split_tf32(float x, float& big, float& small) {
  const uint32_t u = __float_as_uint(x);
  const bool special = (u & 0x7F800000u) == 0x7F800000u;
  big = special ? x : __uint_as_float(u & 0xFFFFE000u);
  small = special ? 0.0f : x - big;
}

__device__ __forceinline__ void split4(float4 x, float4& big, float4& small) {
  split_tf32(x.x, big.x, small.x);
  split_tf32(x.y, big.y, small.y);
  split_tf32(x.z, big.z, small.z);
  split_tf32(x.w, big.w, small.w);
}


// Both operands are packed as blocks of ROWS rows (128 for A, BN for B) x BK
// k, one block pair (big, small) per (row tile, K tile), block pairs of a
// row tile consecutive in K.  Two readers cover the four ways an operand
// can be stored:
//   pack_kc: element (r, k) at src[r*ld + k] (k contiguous): A as stored
//            row-major, or B stored transposed (N x K);
//   pack_rc: element (r, k) at src[k*ld + r] (rows contiguous): B as stored
//            row-major, or A stored transposed (K x M).

// grid (Kt, Rt), 256 threads: each thread moves 16-byte chunks (4 k of a row).
template <class G, int ROWS>
__global__ void __launch_bounds__(256) pack_kc_kernel(const float* __restrict__ src, int64_t ld,
                                                      float* __restrict__ dst_base, int R, int K,
                                                      int Kt, int vec, BoundsRecord* rec) {
  constexpr int BK = G::BK;
  constexpr int BLOCK = ROWS * G::ROW_BYTES;
  const int kt = blockIdx.x, rt = blockIdx.y;
  // The GEMM kernel launched after the packers as their programmatic
  // dependent may be scheduled from now on; it waits inside
  // (griddepcontrol.wait) until this grid has completed.
  asm volatile("griddepcontrol.launch_dependents;");
  // Checked builds: the source view and the gridDim.y x Kt packed blocks.
  const int64_t src_extent = view_extent(R, K, ld);
  const int64_t dst_words = static_cast<int64_t>(gridDim.y) * Kt * (2 * BLOCK / 4);
  char* dst = reinterpret_cast<char*>(dst_base) +
              (static_cast<int64_t>(rt) * Kt + kt) * static_cast<int64_t>(2 * BLOCK);
  for (int c = threadIdx.x; c < ROWS * (BK / 4); c += 256) {
    const int r = c / (BK / 4), ch = c % (BK / 4);
    const int row = rt * ROWS + r, k = kt * BK + ch * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row < R) {
      const int64_t o = static_cast<int64_t>(row) * ld + k;
      const float* p = src + o;
      if (vec) {
        if (k < K && bounds_ok(rec, SITE_PREP_SRC, o, 4, src_extent))
          v = *reinterpret_cast<const float4*>(p);
      } else {
        if (k + 0 < K && bounds_ok(rec, SITE_PREP_SRC, o + 0, 1, src_extent)) v.x = p[0];
        if (k + 1 < K && bounds_ok(rec, SITE_PREP_SRC, o + 1, 1, src_extent)) v.y = p[1];
        if (k + 2 < K && bounds_ok(rec, SITE_PREP_SRC, o + 2, 1, src_extent)) v.z = p[2];
        if (k + 3 < K && bounds_ok(rec, SITE_PREP_SRC, o + 3, 1, src_extent)) v.w = p[3];
      }
    }
    float4 big, small;
    split4(v, big, small);
    const uint32_t off = G::offset(r, ch * 4);
    const int64_t w = (dst - reinterpret_cast<char*>(dst_base) + off) / 4;
    if (bounds_ok(rec, SITE_PREP_DST, w, 4, dst_words) &&
        bounds_ok(rec, SITE_PREP_DST, w + BLOCK / 4, 4, dst_words)) {
      *reinterpret_cast<float4*>(dst + off) = big;
      *reinterpret_cast<float4*>(dst + BLOCK + off) = small;
    }
  }
}

// grid (Kt, ceil(Rt*ROWS/256)), 256 threads: the CTA packs rows
// n0 = blockIdx.y*256 .. n0+255 (ROWS divides 256, so they cover whole
// blocks).  It reads the 256 x BK tile with coalesced row-of-k loads into
// shared memory, then writes the blocks' 16-byte chunks in address order,
// so a warp stores 512 contiguous bytes.
template <class G, int ROWS>
__global__ void __launch_bounds__(256) pack_rc_kernel(const float* __restrict__ src, int64_t ld,
                                                      float* __restrict__ dst_base, int R, int K,
                                                      int Kt, int Rt, BoundsRecord* rec) {
  static_assert(256 % ROWS == 0, "a CTA covers whole blocks");
  constexpr int BK = G::BK;
  constexpr int BLOCK = ROWS * G::ROW_BYTES;
  constexpr int CPR = G::ROW_BYTES / 16;  // 16-byte chunks per packed row
  constexpr int TS = 256 + 1;             // tile row stride (words): k rows, banks spread
  __shared__ float tile[BK * TS];
  asm volatile("griddepcontrol.launch_dependents;");  // as in pack_kc_kernel
  const int kt = blockIdx.x;
  const int n0 = blockIdx.y * 256;
  // Checked builds: the source view (K rows of R) and the Rt x Kt blocks.
  const int64_t src_extent = view_extent(K, R, ld);
  const int64_t dst_words = static_cast<int64_t>(Rt) * Kt * (2 * BLOCK / 4);
#pragma unroll 4
  for (int j = 0; j < BK; ++j) {
    const int k = kt * BK + j, n = n0 + threadIdx.x;
    const int64_t o = static_cast<int64_t>(k) * ld + n;
    tile[j * TS + threadIdx.x] =
        (n < R && k < K && bounds_ok(rec, SITE_PREP_SRC, o, 1, src_extent)) ? src[o] : 0.f;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < 256 * CPR; p += 256) {
    const int rr = p / CPR, pc = p % CPR;  // row within the CTA, physical chunk
    const int rt = (n0 + rr) / ROWS, r = (n0 + rr) % ROWS;
    if (rt >= Rt) break;
    const int r8 = r & 7;
    const int lc = (pc ^ (BK == 32 ? r8 : (r8 >> 1))) & (CPR - 1);  // logical chunk
    float4 v = make_float4(tile[(lc * 4 + 0) * TS + rr], tile[(lc * 4 + 1) * TS + rr],
                           tile[(lc * 4 + 2) * TS + rr], tile[(lc * 4 + 3) * TS + rr]);
    float4 big, small;
    split4(v, big, small);
    char* dst = reinterpret_cast<char*>(dst_base) +
                (static_cast<int64_t>(rt) * Kt + kt) * static_cast<int64_t>(2 * BLOCK);
    const uint32_t off = (r >> 3) * G::ATOM_BYTES + r8 * G::ROW_BYTES + pc * 16;
    const int64_t w = (dst - reinterpret_cast<char*>(dst_base) + off) / 4;
    if (bounds_ok(rec, SITE_PREP_DST, w, 4, dst_words) &&
        bounds_ok(rec, SITE_PREP_DST, w + BLOCK / 4, 4, dst_words)) {
      *reinterpret_cast<float4*>(dst + off) = big;
      *reinterpret_cast<float4*>(dst + BLOCK + off) = small;
    }
  }
}

template <class G>
__global__ void __launch_bounds__(THREADS, 1)
    tf32x3_gemm_kernel(const float* __restrict__ Ap, const float* __restrict__ Bp,
                       Epilogue ep, int Kt, int tiles_m, int tiles_n, int group_m,
                       Sched sched, int fault_inject) {
  constexpr int BK = G::BK, BN = G::BN;
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
  // Launched as a programmatic dependent of the pack kernel before it on the
  // stream: the set-up above overlaps that kernel's end; nothing below reads
  // or writes global memory before it has completed and its stores are
  // visible (a no-op when launched without the attribute).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint32_t issued = 0;  // producer: K tiles issued by this CTA, across its tiles
  if (warp == 0) {
    if (lane == 0) {
      // Producer.  With fault_inject set it issues nothing, so every wait
      // on its data runs out (the test of the timeout path).
      uint32_t& g = issued;
      bool stop = fault_inject != 0;
      for (int u = 0; u < num_units && !stop; ++u) {
        const Unit w = unit_at(u, cta, ctas, sched, tiles_m, tiles_n, group_m, Kt);
        const char* a_src = reinterpret_cast<const char*>(Ap) +
                            static_cast<int64_t>(w.tm) * Kt * G::A_PAIR_BYTES;
        const char* b_src = reinterpret_cast<const char*>(Bp) +
                            static_cast<int64_t>(w.tn) * Kt * G::B_PAIR_BYTES;
        for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
          const uint32_t s = g % STAGES, round = g / STAGES;
          if (g >= STAGES && !wait_phase(bar(EMPTY + s), (round + 1) & 1u, wc)) {
            stop = true;
            break;
          }
          uint8_t* st = smem + s * STAGE_BYTES;
          mbar_arrive_expect_tx(bar(FULL + s), STAGE_BYTES);
          bulk_copy_g2s(smem_u32(st), a_src + static_cast<int64_t>(kt) * G::A_PAIR_BYTES,
                        G::A_PAIR_BYTES, bar(FULL + s));
          bulk_copy_g2s(smem_u32(st + G::A_PAIR_BYTES),
                        b_src + static_cast<int64_t>(kt) * G::B_PAIR_BYTES, G::B_PAIR_BYTES,
                        bar(FULL + s));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer.
      constexpr uint32_t idesc = instr_desc(BM, BN, 2, 2);  // tf32 x tf32
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
          const uint32_t a_big = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t a_small = a_big + G::A_BLOCK_BYTES;
          const uint32_t b_big = a_big + G::A_PAIR_BYTES;
          const uint32_t b_small = b_big + G::B_BLOCK_BYTES;
#pragma unroll
          for (int j = 0; j < BK / 8; ++j) {
            const uint32_t koff = j * 32;  // 8 tf32 = 32 bytes along K
            const uint64_t ab = smem_desc(a_big + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t as = smem_desc(a_small + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t bb = smem_desc(b_big + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t bs = smem_desc(b_small + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            mma_tf32(acc_tmem, ab, bs, idesc, acc);
            acc = 1;
            mma_tf32(acc_tmem, as, bb, idesc, 1);
            mma_tf32(acc_tmem, ab, bb, idesc, 1);
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
      // A tile's accumulator is ready after its whole K loop.  The warp
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
// Split-A kernel: A is not packed.  TMA copies each 128 x BK fp32 tile of A
// (row-major, k contiguous) into shared memory with the 128-byte (BK 32) or
// 64-byte (BK 16) swizzle, which is byte for byte the K-major layout the MMA
// reads; four converter
// warps then split it there — big in place, small into a second buffer —
// and publish it to the tensor core (fence.proxy.async, then conv[s]).  B
// is packed as in the other kernels.  For problems with few columns, where
// packing A (reading 4 and writing 8 bytes per element, then reading the 8
// again) costs more than the product; the tensor pipe has time to spare
// there, so the extra shared-memory traffic of the split is hidden.
//   warp 0: TMA of A, bulk copy of the B pair -> full[s];
//   warps 6-9: wait full[s], split, fence, arrive conv[s];
//   warp 1: wait conv[s], 3 MMAs per k8 step, commit -> empty[s];
//   warps 2-5: epilogue, as in the packed kernel.
constexpr int ASPLIT_THREADS = 320;
constexpr int CONVERT_THREADS = 128;

template <int BK_, int BN_>
struct ASplitGeometry {
  using G = Geometry<BK_, BN_>;
  static constexpr int BK = BK_;
  static constexpr int BN = BN_;
  // TMA swizzle of the fp32 A box: 128-byte rows (BK 32) or 64-byte rows
  // (BK 16), matching the layout codes of G.
  static constexpr CUtensorMapSwizzle TMA_SWIZZLE =
      BK_ == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static constexpr int A_BYTES = G::A_BLOCK_BYTES;  // fp32 tile, then its big part
  static constexpr int STAGE_BYTES = 2 * A_BYTES + G::B_PAIR_BYTES;  // A | A small | B pair
  static constexpr int STAGES_FIT = SMEM_STAGE_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static_assert(STAGES >= 2, "at least two stages");
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256 + EPI_STAGE_BYTES;
};

template <int BK, int BN>
__global__ void __launch_bounds__(ASPLIT_THREADS, 1)
    tf32x3_asplit_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const float* __restrict__ Bp, Epilogue ep, int Kt, int tiles_m,
                         int tiles_n, int group_m, Sched sched, int fault_inject) {
  using AG = ASplitGeometry<BK, BN>;
  using G = typename AG::G;
  constexpr int STAGES = AG::STAGES;
  constexpr int STAGE_BYTES = AG::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars: [0, S) full, [S, 2S) conv, [2S, 3S) empty, then acc_full[2],
  // acc_empty[2], drain.
  constexpr int FULL = 0, CONV = STAGES, EMPTY = 2 * STAGES, ACC_FULL = 3 * STAGES,
                ACC_EMPTY = 3 * STAGES + 2, DRAIN = 3 * STAGES + 4, NBARS = 3 * STAGES + 5;
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
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(FULL + s), 1);                // producer arrival + tx bytes
      mbar_init(bar(CONV + s), CONVERT_THREADS);  // every converter thread
      mbar_init(bar(EMPTY + s), 1);               // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(ACC_FULL + b), 1);
      mbar_init(bar(ACC_EMPTY + b), EPILOGUE_THREADS);
    }
    mbar_init(bar(DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), AG::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the pack kernel before it on the
  // stream: the set-up above overlaps that kernel's end; nothing below reads
  // or writes global memory before it has completed and its stores are
  // visible (a no-op when launched without the attribute).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint32_t issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      uint32_t& g = issued;
      bool stop = fault_inject != 0;
      for (int u = 0; u < num_units && !stop; ++u) {
        const Unit w = unit_at(u, cta, ctas, sched, tiles_m, tiles_n, group_m, Kt);
        const char* b_src = reinterpret_cast<const char*>(Bp) +
                            static_cast<int64_t>(w.tn) * Kt * G::B_PAIR_BYTES;
        for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
          const uint32_t s = g % STAGES, round = g / STAGES;
          if (g >= STAGES && !wait_phase(bar(EMPTY + s), (round + 1) & 1u, wc)) {
            stop = true;
            break;
          }
          const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
          mbar_arrive_expect_tx(bar(FULL + s), AG::A_BYTES + G::B_PAIR_BYTES);
          tma_load_2d(st, &tmap_a, kt * BK, w.tm * BM, bar(FULL + s));
          bulk_copy_g2s(st + 2 * AG::A_BYTES, b_src + static_cast<int64_t>(kt) * G::B_PAIR_BYTES,
                        G::B_PAIR_BYTES, bar(FULL + s));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(BM, BN, 2, 2);
      uint32_t g = 0;
      bool stop = false;
      int it = 0;
      for (int u = 0; u < num_units && !stop; ++u, ++it) {
        const Unit w = unit_at(u, cta, ctas, sched, tiles_m, tiles_n, group_m, Kt);
        const int b = it & 1;
        if (it >= 2 && !wait_phase(bar(ACC_EMPTY + b), ((it >> 1) + 1) & 1u, wc)) break;
        tc_fence_after();
        const uint32_t acc_tmem = tmem + static_cast<uint32_t>(b * BN);
        uint32_t acc = 0;
        for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
          const uint32_t s = g % STAGES, round = g / STAGES;
          if (!wait_phase(bar(CONV + s), round & 1u, wc)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_big = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t a_small = a_big + AG::A_BYTES;
          const uint32_t b_big = a_big + 2 * AG::A_BYTES;
          const uint32_t b_small = b_big + G::B_BLOCK_BYTES;
#pragma unroll
          for (int j = 0; j < BK / 8; ++j) {
            const uint32_t koff = j * 32;
            const uint64_t ab = smem_desc(a_big + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t as = smem_desc(a_small + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t bb = smem_desc(b_big + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t bs = smem_desc(b_small + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            mma_tf32(acc_tmem, ab, bs, idesc, acc);
            acc = 1;
            mma_tf32(acc_tmem, as, bb, idesc, 1);
            mma_tf32(acc_tmem, ab, bb, idesc, 1);
          }
          mma_commit(bar(EMPTY + s));
        }
        if (!stop) mma_commit(bar(ACC_FULL + b));
      }
      mma_commit(bar(DRAIN));
      wait_phase(bar(DRAIN), 0, wc, false);
    }
  } else if (warp < 6) {
    const int q = warp & 3;
    // This warp's staging square, past the barriers.
    float* const epi_square =
        reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256) + q * EPI_WARP_FLOATS;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int it = 0;
    for (int u = 0; u < num_units; ++u, ++it) {
      const int b = it & 1;
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
  } else {
    // Converters: thread t splits the 16-byte chunks t, t + 128, ... of the
    // stage's A tile (consecutive threads, consecutive chunks).
    const int t = threadIdx.x - (ASPLIT_THREADS - CONVERT_THREADS);
    uint32_t g = 0;
    bool stop = fault_inject != 0;
    for (int u = 0; u < num_units && !stop; ++u) {
      const Unit w = unit_at(u, cta, ctas, sched, tiles_m, tiles_n, group_m, Kt);
      for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
        const uint32_t s = g % STAGES, round = g / STAGES;
        if (!wait_phase(bar(FULL + s), round & 1u, wc)) {
          stop = true;
          break;
        }
        float4* a = reinterpret_cast<float4*>(smem + s * STAGE_BYTES);
        float4* a_small = reinterpret_cast<float4*>(smem + s * STAGE_BYTES + AG::A_BYTES);
#pragma unroll
        for (int i = 0; i < AG::A_BYTES / 16 / CONVERT_THREADS; ++i) {
          const int c = i * CONVERT_THREADS + t;
          float4 big, small;
          split4(a[c], big, small);
          a[c] = big;
          a_small[c] = small;
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(CONV + s));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    for (uint32_t q = issued > STAGES ? issued - STAGES : 0; q < issued; ++q)
      wait_phase(bar(FULL + q % STAGES), (q / STAGES) & 1u, wc, false);
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, AG::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair kernel: a cluster of two CTAs on two SMs computes 256 x 256 tiles
// with tcgen05.mma.cta_group::2 kind::tf32.  Both operands are packed in
// 128-row blocks; CTA r of the pair stages block 2*t + r of A's tile row t
// and of B's tile column, each K tile's (big, small) pair arriving by one
// TMA copy that completes on the even CTA's full barrier.  The even CTA issues
// 3 pair MMAs (256 x 256 x 8) per k8 step and commits to both CTAs' barriers;
// each CTA's epilogue drains its 128 rows x 256 columns of TMEM.  Roles,
// bounded waits and the exit protocol as the 16-bit pair kernel.
constexpr int PAIR_TILE = 256;
constexpr int PAIR_HALF = 128;

template <int BK_>
struct PairGeometry {
  static constexpr int BK = BK_;
  static constexpr int ROW_BYTES = BK * 4;
  static constexpr int ATOM_BYTES = 8 * ROW_BYTES;
  static constexpr uint64_t LAYOUT = BK == 32 ? 2 : 4;  // 128-B / 64-B swizzle
  static constexpr int BLOCK_BYTES = PAIR_HALF * ROW_BYTES;
  static constexpr int PAIR_BYTES = 2 * BLOCK_BYTES;  // big | small of one 128-row block
  static constexpr int STAGE_BYTES = 2 * PAIR_BYTES;  // A pair | B pair
  static constexpr int STAGES_FIT = SMEM_STAGE_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static_assert(STAGES >= 2, "at least two stages");
  static constexpr uint32_t TMEM_COLS = 2 * PAIR_TILE;  // two accumulators
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256 + EPI_STAGE_BYTES;
  // The packed buffers seen as 2-D tensors of 1 KB rows: one TMA box of
  // PAIR_ROWS rows is one block pair.
  static constexpr int PAIR_ROWS = PAIR_BYTES / 1024;
};

template <int BK>
__global__ void __launch_bounds__(THREADS, 1)
    tf32x3_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_b, Epilogue ep, int Kt,
                       int tiles_m, int tiles_n, int group_m, Sched sched, int fault_inject) {
  using G = PairGeometry<BK>;
  constexpr int STAGES = G::STAGES;
  constexpr int STAGE_BYTES = G::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  constexpr int FULL = 0, EMPTY = STAGES, ACC_FULL = 2 * STAGES, ACC_EMPTY = 2 * STAGES + 2,
                DRAIN = 2 * STAGES + 4, NBARS = 2 * STAGES + 5;
  static_assert(NBARS * 8 + 8 <= 256, "barriers, TMEM slot and abort flag fit 256 bytes");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const WaitCtx wc{abort_flag, &g_status};
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = static_cast<int>(cluster_id_x());
  const int clusters = static_cast<int>(cluster_count_x());
  const int num_tiles = tiles_m * tiles_n;
  const int num_units = units_of(cluster, clusters, sched, num_tiles, Kt);  // this cluster's units

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(FULL + s), 1);
      mbar_init(bar(EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(ACC_FULL + b), 1);
      mbar_init(bar(ACC_EMPTY + b), 8);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(bar(DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), G::TMEM_COLS);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the pack kernel before it on the
  // stream: the set-up above overlaps that kernel's end; nothing below reads
  // or writes global memory before it has completed and its stores are
  // visible (a no-op when launched without the attribute).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    if (lane == 0) {
      bool stop = fault_inject != 0;
      uint32_t g = 0;
      const uint32_t full_even0 = map_to_cta(bar(FULL), 0);
      for (int u = 0; u < num_units && !stop; ++u) {
        const Unit w = unit_at(u, cluster, clusters, sched, tiles_m, tiles_n, group_m, Kt);
        const int blk_a = 2 * w.tm + static_cast<int>(rank);
        const int blk_b = 2 * w.tn + static_cast<int>(rank);
        for (int kt = w.kt0; kt < w.kt1; ++kt, ++g) {
          const uint32_t s = g % STAGES, round = g / STAGES;
          if (g >= STAGES && !wait_phase(bar(EMPTY + s), (round + 1) & 1u, wc)) {
            stop = true;
            break;
          }
          const uint32_t full_even = full_even0 + 8u * s;
          if (leader) mbar_arrive_expect_tx(bar(FULL + s), 2 * STAGE_BYTES);
          const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
          tma_load_2d_pair(st, &tmap_a, 0, (blk_a * Kt + kt) * G::PAIR_ROWS, full_even);
          tma_load_2d_pair(st + G::PAIR_BYTES, &tmap_b, 0, (blk_b * Kt + kt) * G::PAIR_ROWS,
                           full_even);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = instr_desc(PAIR_TILE, PAIR_TILE, 2, 2);  // tf32 x tf32
      uint32_t g = 0;
      bool stop = false;
      int it = 0;
      for (int u = 0; u < num_units && !stop; ++u, ++it) {
        const Unit w = unit_at(u, cluster, clusters, sched, tiles_m, tiles_n, group_m, Kt);
        const int b = it & 1;
        if (it >= 2 && !wait_phase(bar(ACC_EMPTY + b), ((it >> 1) + 1) & 1u, wc)) break;
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
          const uint32_t a_big = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t a_small = a_big + G::BLOCK_BYTES;
          const uint32_t b_big = a_big + G::PAIR_BYTES;
          const uint32_t b_small = b_big + G::BLOCK_BYTES;
#pragma unroll
          for (int j = 0; j < BK / 8; ++j) {
            const uint32_t koff = j * 32;  // 8 tf32 = 32 bytes along K
            const uint64_t ab = smem_desc(a_big + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t as = smem_desc(a_small + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t bb = smem_desc(b_big + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            const uint64_t bs = smem_desc(b_small + koff, 16, G::ATOM_BYTES, G::LAYOUT);
            mma_tf32_pair(acc_tmem, ab, bs, idesc, acc);
            acc = 1;
            mma_tf32_pair(acc_tmem, as, bb, idesc, 1);
            mma_tf32_pair(acc_tmem, ab, bb, idesc, 1);
          }
          mma_commit_pair(bar(EMPTY + s), 0x3);
        }
        if (!stop) mma_commit_pair(bar(ACC_FULL + b), 0x3);
      }
      mma_commit_pair(bar(DRAIN), 0x1);
      wait_phase(bar(DRAIN), 0, wc, false);
    }
  } else {
    const int q = warp & 3;
    // This warp's staging square, past the barriers.
    float* const epi_square =
        reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256) + q * EPI_WARP_FLOATS;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acc_empty_even = map_to_cta(bar(ACC_EMPTY), 0);
    int it = 0;
    for (int u = 0; u < num_units; ++u, ++it) {
      const int b = it & 1;
      const bool ready = wait_phase(bar(ACC_FULL + b), (it >> 1) & 1u, wc, true,
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
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, G::TMEM_COLS);
  }
}

}  // namespace tf32x3

// ---------------------------------------------------------------------------
// Host side.  Configurations: (BK, BN) in {16, 32} x {256, 128, 64}.

namespace {

// Launches a GEMM kernel as a programmatic dependent of the pack kernel
// before it on `stream` (clusters of `cluster` CTAs when > 1): its CTAs are
// scheduled as the packer's retire and set up their barriers and tensor
// memory, then wait for the packed operands (griddepcontrol.wait).  The
// arguments are passed by address in declaration order.
template <class... Args>
cudaError_t launch_after_pack(const void* kernel, dim3 grid, int threads, int smem_bytes,
                              int cluster, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  void* ptrs[] = {static_cast<void*>(&args)...};
  return cudaLaunchKernelExC(&cfg, kernel, ptrs);
}

template <int BK, int BN>
struct Cfg {
  using G = tf32x3::Geometry<BK, BN>;
  static int64_t workspace_bytes_packed(int M, int N, int K) { return workspace(M, N, K); }
  static int64_t workspace(int M, int N, int K) {
    const int64_t mt = (M + tf32x3::BM - 1) / tf32x3::BM;
    const int64_t nt = (N + BN - 1) / BN;
    const int64_t kt = (K + BK - 1) / BK;
    return mt * kt * G::A_PAIR_BYTES + nt * kt * G::B_PAIR_BYTES;
  }
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(tf32x3::tf32x3_gemm_kernel<G>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
  }
  // vec_a / vec_b: the operand is read k-contiguous (A as stored, B stored
  // transposed) with a leading dimension % 4 == 0 from a 16-byte aligned
  // base, so its packer may read float4.
  static cudaError_t launch(const GemmArgs& a, void* workspace, bool vec_a, bool vec_b,
                            bool vec_c, int max_ctas, int fault_inject, cudaStream_t stream) {
    using namespace tf32x3;
    const int mt = (a.M + BM - 1) / BM, nt = (a.N + BN - 1) / BN, kt = (a.K + BK - 1) / BK;
    if (mt > 65535 || nt > 65535 || (mt * BM + 255) / 256 > 65535 ||
        (nt * BN + 255) / 256 > 65535)
      return cudaErrorInvalidValue;
    float* Ap = static_cast<float*>(workspace);
    float* Bp = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         static_cast<int64_t>(mt) * kt * G::A_PAIR_BYTES);
    // A: rows m, k contiguous unless stored transposed.
    if (a.trans_a)
      pack_rc_kernel<G, BM><<<dim3(kt, (mt * BM + 255) / 256), 256, 0, stream>>>(
          a.A, a.lda, Ap, a.M, a.K, kt, mt, a.bounds);
    else
      pack_kc_kernel<G, BM><<<dim3(kt, mt), 256, 0, stream>>>(a.A, a.lda, Ap, a.M, a.K, kt,
                                                              vec_a ? 1 : 0, a.bounds);
    // B: rows n, n contiguous (row-major K x N) unless stored transposed.
    if (a.trans_b)
      pack_kc_kernel<G, BN><<<dim3(kt, nt), 256, 0, stream>>>(a.B, a.ldb, Bp, a.N, a.K, kt,
                                                              vec_b ? 1 : 0, a.bounds);
    else
      pack_rc_kernel<G, BN><<<dim3(kt, (nt * BN + 255) / 256), 256, 0, stream>>>(
          a.B, a.ldb, Bp, a.N, a.K, kt, nt, a.bounds);
    const int tiles = mt * nt;
    // Split tail: the partial tiles follow the packed operands.
    Sched sched{a.full_tiles, a.split, a.kt_per_slice, nullptr, a.sk_ctas, a.sk_iters};
    if (a.split > 1 || a.sk_ctas > 0)
      sched.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                workspace_bytes_packed(a.M, a.N, a.K));
    const int units = a.full_tiles + (tiles - a.full_tiles) * a.split;
    const int grid = persistent_grid(a, units, max_ctas);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // The staged epilogue only for rows of C that are not float4-aligned:
    // otherwise the kernel stays small enough (193 KB) to share an SM with a
    // packer CTA (33 KB), so its CTAs are placed while the packers run
    // (1024^3 back to back 32.7 us, against 34.6 us staged).
    const Epilogue ep = make_epilogue(a, vec_c, tiles, BM, BN, !vec_c);
    e = launch_after_pack(reinterpret_cast<const void*>(tf32x3_gemm_kernel<G>), dim3(grid),
                          THREADS, epilogue_smem(G::SMEM_BYTES, ep), 1, stream, Ap, Bp, ep,
                          kt, mt, nt, a.group_m, sched, fault_inject);
    if (e != cudaSuccess) return e;
    return launch_second_pass(a, sched.partial, BM, BN, kt, vec_c, stream);
  }
};

// CTA-pair configuration (256 x 256 tiles), K depth BK.
template <int BK>
struct CfgPair {
  using G = tf32x3::PairGeometry<BK>;
  using GP = tf32x3::Geometry<BK, 128>;  // packing in 128-row blocks
  static constexpr int ROWS = tf32x3::PAIR_HALF;

  static int64_t workspace(int M, int N, int K) {
    const int64_t mt = (M + 255) / 256, nt = (N + 255) / 256, kt = (K + BK - 1) / BK;
    return (2 * mt + 2 * nt) * kt * G::PAIR_BYTES;
  }
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(tf32x3::tf32x3_pair_kernel<BK>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
  }
  static int max_clusters() {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(tf32x3::THREADS, 1, 1);
    cfg.dynamicSmemBytes = G::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(
                                               tf32x3::tf32x3_pair_kernel<BK>),
                                       &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  }
  static cudaError_t launch(const GemmArgs& a, void* workspace, bool vec_a, bool vec_b,
                            bool vec_c, int max_clusters, int fault_inject, cudaStream_t stream) {
    using namespace tf32x3;
    const int mt = (a.M + PAIR_TILE - 1) / PAIR_TILE, nt = (a.N + PAIR_TILE - 1) / PAIR_TILE;
    const int kt = (a.K + BK - 1) / BK;
    if (2 * mt > 65535 || 2 * nt > 65535) return cudaErrorInvalidValue;
    float* Ap = static_cast<float*>(workspace);
    float* Bp = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         static_cast<int64_t>(2 * mt) * kt * G::PAIR_BYTES);
    if (a.trans_a)
      pack_rc_kernel<GP, ROWS><<<dim3(kt, (2 * mt * ROWS + 255) / 256), 256, 0, stream>>>(
          a.A, a.lda, Ap, a.M, a.K, kt, 2 * mt, a.bounds);
    else
      pack_kc_kernel<GP, ROWS><<<dim3(kt, 2 * mt), 256, 0, stream>>>(a.A, a.lda, Ap, a.M, a.K,
                                                                     kt, vec_a ? 1 : 0, a.bounds);
    if (a.trans_b)
      pack_kc_kernel<GP, ROWS><<<dim3(kt, 2 * nt), 256, 0, stream>>>(a.B, a.ldb, Bp, a.N, a.K,
                                                                     kt, vec_b ? 1 : 0, a.bounds);
    else
      pack_rc_kernel<GP, ROWS><<<dim3(kt, (2 * nt * ROWS + 255) / 256), 256, 0, stream>>>(
          a.B, a.ldb, Bp, a.N, a.K, kt, 2 * nt, a.bounds);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // The packed buffers as 2-D tensors of 1 KB rows (256 floats, no
    // swizzle: the blocks are already in the tensor core's order).
    CUtensorMap map_a, map_b;
    const int64_t rows_a = static_cast<int64_t>(2 * mt) * kt * G::PAIR_ROWS;
    const int64_t rows_b = static_cast<int64_t>(2 * nt) * kt * G::PAIR_ROWS;
    if (!encode_tensor_map_2d(&map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Ap, rows_a, 256, 256,
                              256, G::PAIR_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tensor_map_2d(&map_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Bp, rows_b, 256, 256,
                              256, G::PAIR_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    const int tiles = mt * nt;
    Sched sched{a.full_tiles, a.split, a.kt_per_slice, nullptr, a.sk_ctas, a.sk_iters};
    if (a.split > 1 || a.sk_ctas > 0)
      sched.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                CfgPair::workspace(a.M, a.N, a.K));
    const int units = a.full_tiles + (tiles - a.full_tiles) * a.split;
    const int clusters = persistent_grid(a, units, max_clusters);
    const Epilogue ep = make_epilogue(a, vec_c, tiles, PAIR_TILE, PAIR_TILE, !vec_c);  // as above
    e = launch_after_pack(reinterpret_cast<const void*>(tf32x3_pair_kernel<BK>),
                          dim3(2 * clusters), THREADS, epilogue_smem(G::SMEM_BYTES, ep), 2,
                          stream, map_a, map_b, ep, kt, mt, nt, a.group_m, sched,
                          fault_inject);
    if (e != cudaSuccess) return e;
    return launch_second_pass(a, sched.partial, PAIR_TILE, PAIR_TILE, kt, vec_c, stream);
  }
};

// Split-A configuration (A split inside the GEMM kernel), K depth BK.
template <int BK, int BN>
struct CfgASplit {
  using AG = tf32x3::ASplitGeometry<BK, BN>;
  using G = typename AG::G;

  static int64_t workspace(int M, int N, int K) {
    (void)M;
    const int64_t nt = (N + BN - 1) / BN, kt = (K + BK - 1) / BK;
    return nt * kt * G::B_PAIR_BYTES;
  }
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(tf32x3::tf32x3_asplit_kernel<BK, BN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, AG::SMEM_BYTES);
  }
  static cudaError_t launch(const GemmArgs& a, void* workspace, bool vec_b, bool vec_c,
                            int max_ctas, int fault_inject, cudaStream_t stream) {
    using namespace tf32x3;
    const int mt = (a.M + BM - 1) / BM, nt = (a.N + BN - 1) / BN, kt = (a.K + BK - 1) / BK;
    if (nt > 65535 || (nt * BN + 255) / 256 > 65535) return cudaErrorInvalidValue;
    float* Bp = static_cast<float*>(workspace);
    if (a.trans_b)
      pack_kc_kernel<G, BN><<<dim3(kt, nt), 256, 0, stream>>>(a.B, a.ldb, Bp, a.N, a.K, kt,
                                                              vec_b ? 1 : 0, a.bounds);
    else
      pack_rc_kernel<G, BN><<<dim3(kt, (nt * BN + 255) / 256), 256, 0, stream>>>(
          a.B, a.ldb, Bp, a.N, a.K, kt, nt, a.bounds);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // A (M x K, row pitch lda) in 128 x BK boxes with the swizzle of the
    // MMA's K-major layout; zero fill past M and K.
    CUtensorMap map_a;
    if (!encode_tensor_map_2d(&map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.A, a.M, a.K, a.lda,
                              BK, BM, AG::TMA_SWIZZLE))
      return cudaErrorInvalidValue;
    const int tiles = mt * nt;
    Sched sched{a.full_tiles, a.split, a.kt_per_slice, nullptr, a.sk_ctas, a.sk_iters};
    if (a.split > 1 || a.sk_ctas > 0)
      sched.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                CfgASplit::workspace(a.M, a.N, a.K));
    const int units = a.full_tiles + (tiles - a.full_tiles) * a.split;
    const int grid = persistent_grid(a, units, max_ctas);
    const Epilogue ep = make_epilogue(a, vec_c, tiles, BM, BN, !vec_c);  // as above
    e = launch_after_pack(reinterpret_cast<const void*>(tf32x3_asplit_kernel<BK, BN>),
                          dim3(grid), ASPLIT_THREADS, epilogue_smem(AG::SMEM_BYTES, ep), 1,
                          stream, map_a,
                          static_cast<const float*>(Bp), ep, kt, mt, nt, a.group_m, sched,
                          fault_inject);
    if (e != cudaSuccess) return e;
    return launch_second_pass(a, sched.partial, BM, BN, kt, vec_c, stream);
  }
};

template <class F>
bool dispatch_asplit(int bk, int bn, F&& f) {
  if (bk == 16 && bn == 256) { f(CfgASplit<16, 256>{}); return true; }
  if (bk == 16 && bn == 128) { f(CfgASplit<16, 128>{}); return true; }
  if (bk == 16 && bn == 64) { f(CfgASplit<16, 64>{}); return true; }
  if (bk == 32 && bn == 256) { f(CfgASplit<32, 256>{}); return true; }
  if (bk == 32 && bn == 128) { f(CfgASplit<32, 128>{}); return true; }
  if (bk == 32 && bn == 64) { f(CfgASplit<32, 64>{}); return true; }
  return false;
}

template <class F>
bool dispatch_pair(int bk, F&& f) {
  if (bk == 16) { f(CfgPair<16>{}); return true; }
  if (bk == 32) { f(CfgPair<32>{}); return true; }
  return false;
}

// Calls f.template operator()<BK, BN>() for the runtime choice; false when
// the pair is not built.
template <class F>
bool dispatch(int bk, int bn, F&& f) {
  if (bk == 16 && bn == 256) { f(Cfg<16, 256>{}); return true; }
  if (bk == 16 && bn == 128) { f(Cfg<16, 128>{}); return true; }
  if (bk == 16 && bn == 64) { f(Cfg<16, 64>{}); return true; }
  if (bk == 32 && bn == 256) { f(Cfg<32, 256>{}); return true; }
  if (bk == 32 && bn == 128) { f(Cfg<32, 128>{}); return true; }
  if (bk == 32 && bn == 64) { f(Cfg<32, 64>{}); return true; }
  return false;
}

}  // namespace

bool tf32x3_valid(int bm, int bk, int bn, int split_a) {
  if (split_a) return bm == tf32x3::BM && dispatch_asplit(bk, bn, [](auto) {});
  if (bm == tf32x3::PAIR_TILE) return bn == tf32x3::PAIR_TILE && dispatch_pair(bk, [](auto) {});
  return bm == tf32x3::BM && dispatch(bk, bn, [](auto) {});
}

int64_t tf32x3_workspace_bytes(int M, int N, int K, int bm, int bk, int bn, int split_a) {
  int64_t r = -1;
  if (split_a)
    dispatch_asplit(bk, bn, [&](auto c) { r = decltype(c)::workspace(M, N, K); });
  else if (bm == tf32x3::PAIR_TILE)
    dispatch_pair(bk, [&](auto c) { r = decltype(c)::workspace(M, N, K); });
  else
    dispatch(bk, bn, [&](auto c) { r = decltype(c)::workspace(M, N, K); });
  return r;
}

int tf32x3_smem_bytes(int bm, int bk, int bn, int split_a) {
  int r = -1;
  if (split_a)
    dispatch_asplit(bk, bn, [&](auto c) { r = decltype(c)::AG::SMEM_BYTES; });
  else if (bm == tf32x3::PAIR_TILE)
    dispatch_pair(bk, [&](auto c) { r = decltype(c)::G::SMEM_BYTES; });
  else
    dispatch(bk, bn, [&](auto c) { r = decltype(c)::G::SMEM_BYTES; });
  return r;
}

int tf32x3_stages(int bm, int bk, int bn, int split_a) {
  int r = -1;
  if (split_a)
    dispatch_asplit(bk, bn, [&](auto c) { r = decltype(c)::AG::STAGES; });
  else if (bm == tf32x3::PAIR_TILE)
    dispatch_pair(bk, [&](auto c) { r = decltype(c)::G::STAGES; });
  else
    dispatch(bk, bn, [&](auto c) { r = decltype(c)::G::STAGES; });
  return r;
}

namespace {
std::mutex g_pair_mutex;
int g_pair_clusters[64][2];  // [device][bk == 32]
}  // namespace

int tf32x3_pair_max_clusters(int device, int bk) {
  if (device < 0 || device >= 64 || (bk != 16 && bk != 32)) return 0;
  std::lock_guard<std::mutex> lock(g_pair_mutex);
  int& n = g_pair_clusters[device][bk == 32 ? 1 : 0];
  if (n == 0) {
    cudaError_t e = cudaErrorInvalidValue;
    dispatch_pair(bk, [&](auto c) {
      e = decltype(c)::prepare();
      if (e == cudaSuccess) n = decltype(c)::max_clusters();
    });
    if (e != cudaSuccess) cudaGetLastError();
  }
  return n;
}

int tf32x3_threads(int split_a) {
  return split_a ? tf32x3::ASPLIT_THREADS : tf32x3::THREADS;
}
int tf32x3_bm() { return tf32x3::BM; }

cudaError_t tf32x3_prepare(int device, int bm, int bk, int bn, int split_a) {
  (void)device;
  cudaError_t e = cudaErrorInvalidValue;
  if (split_a)
    dispatch_asplit(bk, bn, [&](auto c) { e = decltype(c)::prepare(); });
  else if (bm == tf32x3::PAIR_TILE)
    dispatch_pair(bk, [&](auto c) { e = decltype(c)::prepare(); });
  else
    dispatch(bk, bn, [&](auto c) { e = decltype(c)::prepare(); });
  return e;
}

cudaError_t launch_tf32x3(const GemmArgs& a, void* workspace, bool vec_a, bool vec_b,
                          bool vec_c, int bm, int bk, int bn, int split_a, int max_ctas,
                          int fault_inject, cudaStream_t stream) {
  cudaError_t e = cudaErrorInvalidValue;
  if (split_a) {
    if (bm != tf32x3::BM || a.trans_a) return e;
    dispatch_asplit(bk, bn, [&](auto c) {
      e = decltype(c)::launch(a, workspace, vec_b, vec_c, max_ctas, fault_inject, stream);
    });
    return e;
  }
  if (bm == tf32x3::PAIR_TILE) {
    dispatch_pair(bk, [&](auto c) {
      e = decltype(c)::launch(a, workspace, vec_a, vec_b, vec_c, max_ctas, fault_inject,
                              stream);
    });
    return e;
  }
  dispatch(bk, bn, [&](auto c) {
    e = decltype(c)::launch(a, workspace, vec_a, vec_b, vec_c, max_ctas, fault_inject, stream);
  });
  return e;
}

// ---------------------------------------------------------------------------
// Static scratch of the allocation-free entry point (mt_sgemm_tf32x3_noalloc):
// the packed copies of A and B live here instead of in memory allocated per
// call.  Every device that loads the library holds this array until the
// process exits.  Calls share it, so calls that overlap on the GPU race on
// it; each call's pack kernels rewrite every byte the call then reads
// (padding included), so nothing has to be cleared between calls.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_noalloc_mutex;
// Device address of the array per device ordinal, kept for the life of the
// process (a cudaDeviceReset that reloads the module is not supported, as
// for the library's other per-device set-up).
void* g_noalloc_ptr[64];
}  // namespace

cudaError_t tf32x3_noalloc_scratch(int device, void** ptr) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[device]) {
    // In host code the array's name is only a stand-in; the device address
    // comes from the runtime, looked up once per device with that device
    // current (the caller's current device).
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[device] = p;
  }
  *ptr = g_noalloc_ptr[device];
  return cudaSuccess;
}

cudaError_t tf32x3_read_and_clear_status(unsigned int* status) {
  cudaError_t e = cudaMemcpyFromSymbol(status, tf32x3::g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(tf32x3::g_status, &zero, sizeof(unsigned int));
}

}  // namespace mt
