// Building blocks of the persistent tcgen05 GEMM kernels (3xTF32 on fp32
// inputs, fp32-accumulating MMA on 16-bit inputs): inline PTX for mbarriers,
// bulk and tensor (TMA) copies, tcgen05 MMA / TMEM, bounded waits, the
// work-unit schedule with its split tail, and the TMEM -> C epilogue store.
#pragma once

#include <cstdint>

#include "device_util.cuh"

namespace mt {
namespace tc {

constexpr uint64_t TIMEOUT_NS = 1000000000ull;  // 1 s per wait

// ---------------------------------------------------------------------------
// mbarriers, copies, fences.
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.b32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Contiguous global -> shared copy (16-byte aligned, size % 16 == 0),
// completing `bytes` transaction bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Tiled tensor copy of one box at coordinates (x, y) of a 2-D tensor map
// (x innermost) into shared memory; the whole box's bytes complete on `bar`,
// elements outside the tensor arrive as zeros.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// The same copy for a CTA pair (cta_group::2): the box lands in this CTA's
// shared memory and its bytes complete on `bar`, which may be the peer's
// barrier (a shared::cluster address from mapa).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int x, int y,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Shared::cluster address of this CTA's shared address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   cluster_addr)
               : "memory");
}

// Orders this thread's generic-proxy writes to shared memory before later
// async-proxy reads of it (TMA stores, tcgen05.mma operand fetches).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 MMA.

// Shared-memory matrix descriptor: start address, leading byte offset,
// stride byte offset (both in bytes, multiples of 16), swizzle `layout`
// (2 = 128-byte, 4 = 64-byte), descriptor version 1.
//   K-major swizzled operand: rows in 8-row atoms; stride = bytes between
//     atoms; leading offset unused (the MMA's K extent lies inside one
//     swizzle row).
//   MN-major swizzled operand: 8 k-rows of one swizzle width of M/N values
//     form an atom; leading = bytes between atoms along M/N, stride = bytes
//     between atoms along K.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t leading_bytes,
                                              uint32_t stride_bytes, uint64_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);           // start address, 16-byte units
  d |= static_cast<uint64_t>((leading_bytes >> 4) & 0x3FFFu) << 16;  // leading byte offset
  d |= static_cast<uint64_t>((stride_bytes >> 4) & 0x3FFFu) << 32;   // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
  d |= layout << 61;                                            // swizzle mode
  return d;
}

// Instruction descriptor: D fp32; A and B of format a_fmt / b_fmt (kind::tf32:
// 2 = tf32; kind::f16: 0 = f16, 1 = bf16); a_mn / b_mn = 1 for an MN-major
// operand; M x N.
__host__ __device__ constexpr uint32_t instr_desc(int m, int n, uint32_t a_fmt,
                                                  uint32_t b_fmt, uint32_t a_mn = 0,
                                                  uint32_t b_mn = 0) {
  return (1u << 4)                                 // D format: f32
         | (a_fmt << 7) | (b_fmt << 10)            // operand formats
         | (a_mn << 15) | (b_mn << 16)             // operand major-ness
         | (static_cast<uint32_t>(n >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);  // M / 16
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// CTA-pair MMA (cta_group::2, issued by the even CTA of the pair): A's rows
// are split between the pair (the first half from this CTA's shared memory,
// the second half from the peer's at the same address), B's columns likewise,
// and each CTA's TMEM receives its half of D's rows, all N columns.
__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_tf32_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on the barrier at `bar`'s offset in every CTA of `cta_mask` once
// every pair MMA this thread issued before it has retired.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// Pair allocation: one warp of each CTA of the pair executes it together;
// the same TMEM columns are allocated in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_addr, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   slot_addr),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

// Arrives on `bar` once every MMA this thread issued before it has retired.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_addr, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   slot_addr),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// Bounded waits.  A CTA's roles share an abort flag in shared memory; the
// kernel's device status word (bit 0) records that a wait expired.
struct WaitCtx {
  volatile int* abort_flag;
  unsigned int* status;
};

// Returns false when the CTA is aborting (another role gave up) or this wait
// itself ran out of time, in which case it raises the abort flag and the
// status word.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                           bool honour_abort = true,
                                           uint64_t limit_ns = TIMEOUT_NS) {
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u) {
      if (honour_abort && *w.abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        *w.abort_flag = 1;
        atomicOr(w.status, 1u);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Work units of the persistent loop: below full_tiles a unit is a whole tile
// (its index in the grouped raster); the tiles after those are split into
// `split` K slices, one unit per slice, whose fp32 partial tiles (dense
// BM x BN, tail tile major, slice minor) are added by a second kernel.
//
// Stream-K (sk_ctas > 0, split = 1): CTA (or cluster) c of the persistent
// grid takes its whole tiles below full_tiles (c, c + grid, ...), then, if c
// < sk_ctas, the run [c*sk_iters/sk_ctas, (c+1)*sk_iters/sk_ctas) of the K
// tiles of the tiles from full_tiles on (tile-major, k ascending), one unit
// per tile the run touches.  A unit that covers its tile whole goes to C;
// a piece goes to partial slot 2c (the run's first tile) or 2c+1 (its
// last), added in k order by the stream-K fix-up kernel.
struct Sched {
  int full_tiles;
  int split;
  int kt_per_slice;
  float* partial;
  int sk_ctas;
  long long sk_iters;
};

struct Unit {
  int tm, tn;    // tile coordinates
  int kt0, kt1;  // K tiles [kt0, kt1)
  int pidx;      // partial tile index, -1 for a whole tile
};

__device__ __forceinline__ Unit unit_of(int u, const Sched& sc, int tiles_m, int tiles_n,
                                        int group_m, int Kt) {
  Unit w;
  int tile = u;
  w.kt0 = 0;
  w.kt1 = Kt;
  w.pidx = -1;
  if (u >= sc.full_tiles) {
    const int v = u - sc.full_tiles;
    tile = sc.full_tiles + v / sc.split;
    w.kt0 = min(Kt, (v % sc.split) * sc.kt_per_slice);
    w.kt1 = min(Kt, w.kt0 + sc.kt_per_slice);
    w.pidx = v;
  }
  grouped_tile(tile, tiles_m, tiles_n, group_m, w.tm, w.tn);
  return w;
}

// Units of CTA (or cluster) c of a persistent grid of `ctas`, in the order
// it runs them: with the split tail, units c, c + ctas, ...; with stream-K,
// its whole tiles, then the tiles its run touches.
__device__ __forceinline__ int units_of(int c, int ctas, const Sched& sc, int num_tiles,
                                        int Kt) {
  if (sc.sk_ctas > 0) {
    const int dp = sc.full_tiles > c ? (sc.full_tiles - 1 - c) / ctas + 1 : 0;
    if (c >= sc.sk_ctas) return dp;
    const long long b = static_cast<long long>(c) * sc.sk_iters / sc.sk_ctas;
    const long long e = static_cast<long long>(c + 1) * sc.sk_iters / sc.sk_ctas;
    return dp + (e > b ? static_cast<int>((e - 1) / Kt - b / Kt + 1) : 0);
  }
  const int num_units = sc.full_tiles + (num_tiles - sc.full_tiles) * sc.split;
  return num_units > c ? (num_units - 1 - c) / ctas + 1 : 0;
}

// Unit j (0 <= j < units_of(c, ...)) of CTA (or cluster) c.
__device__ __forceinline__ Unit unit_at(int j, int c, int ctas, const Sched& sc, int tiles_m,
                                        int tiles_n, int group_m, int Kt) {
  if (sc.sk_ctas > 0) {
    const int dp = sc.full_tiles > c ? (sc.full_tiles - 1 - c) / ctas + 1 : 0;
    if (j >= dp) {
      const int s = j - dp;
      const long long b = static_cast<long long>(c) * sc.sk_iters / sc.sk_ctas;
      const long long e = static_cast<long long>(c + 1) * sc.sk_iters / sc.sk_ctas;
      const long long start = s == 0 ? b : (b / Kt + s) * Kt;
      const long long t_rel = start / Kt;
      const long long end = min(e, (t_rel + 1) * Kt);
      Unit w;
      w.kt0 = static_cast<int>(start - t_rel * Kt);
      w.kt1 = static_cast<int>(end - t_rel * Kt);
      w.pidx = w.kt0 == 0 && w.kt1 == Kt ? -1 : 2 * c + (s == 0 ? 0 : 1);
      grouped_tile(sc.full_tiles + static_cast<int>(t_rel), tiles_m, tiles_n, group_m, w.tm,
                   w.tn);
      return w;
    }
  }
  return unit_of(c + j * ctas, sc, tiles_m, tiles_n, group_m, Kt);
}

// Each epilogue warp's 32 x 32 staging square in shared memory: with a row
// stride of 33 words a warp's row-wise writes (lane l writes row l) and its
// column-wise reads (lane l reads column l) each fall on 32 distinct banks.
constexpr int EPI_STRIDE = 33;
constexpr int EPI_WARP_FLOATS = 32 * EPI_STRIDE;
// The squares of a CTA's four epilogue warps.
constexpr int EPI_STAGE_BYTES = 4 * EPI_WARP_FLOATS * 4;

// The C update of a tile, shared by the epilogues.
struct Epilogue {
  float* C;
  int64_t ldc;
  float alpha, beta;
  int M, N;
  int vec_c;  // 16-byte stores of C allowed (N, ldc % 4 == 0, aligned base)
  const float* bias;  // N floats added to every row (nullptr: none)
  // 1: results go through the epilogue warps' staging squares in shared
  // memory (the kernel was launched with EPI_STAGE_BYTES more of it); 0:
  // each lane stores its own row.
  int staged = 0;
  // Elements of C's view and of the split tail's partial tiles, and the
  // checked build's record (see bounds_ok).
  int64_t c_extent = 0, partial_extent = 0;
  BoundsRecord* bounds = nullptr;
};

// Shared memory to launch a kernel of `smem_bytes` (its staging squares
// included) with: the squares only when the epilogue uses them.
inline int epilogue_smem(int smem_bytes, const Epilogue& ep) {
  return ep.staged ? smem_bytes : smem_bytes - EPI_STAGE_BYTES;
}

// The epilogue of a call: C's view, and the split tail's partial tiles
// (one dense tile_m x bn tile per slice of each split tile).
inline Epilogue make_epilogue(const GemmArgs& a, bool vec_c, int tiles, int tile_m, int bn,
                              bool staged) {
  Epilogue ep{a.C, a.ldc, a.alpha, a.beta, a.M, a.N, vec_c ? 1 : 0, a.bias};
  ep.staged = staged ? 1 : 0;
  ep.c_extent = a.c_extent;
  ep.partial_extent = a.sk_ctas > 0
                          ? 2 * static_cast<int64_t>(a.sk_ctas) * tile_m * bn
                          : static_cast<int64_t>(tiles - a.full_tiles) * a.split * tile_m * bn;
  ep.bounds = a.bounds;
  return ep;
}


// Drains this warp's 32 TMEM lanes -- rows q*32 .. q*32+31 of the BM x BN
// accumulator whose first column of this warp's lanes is TMEM address
// `t_row` -- to C: C = alpha * acc + beta * C (+ bias[col]), masked to
// M x N, C not read when beta == 0; or, for a K slice, to its dense partial
// tile.  With ep.staged each 32-column chunk goes through the warp's
// staging square `stage`: a TMEM load gives lane l row l, the square gives
// lane l column l, so every store writes 32 consecutive floats of one row
// (one 128-byte line when aligned) instead of one float4 (or, unaligned,
// one float) in each of 32 rows.  Measured on GB300, ragged 4097 x 3001 x
// 2053 (rows of C not float4-aligned): bf16 inputs 118.7 -> 69.5 us, 3xTF32
// 236.4 -> 206.8 us; bf16 4096^3 95.2 -> 91.1 us.
//
// TILE_M is the tile's row count (BM for one CTA, 2 * BM for a CTA pair) and
// sub_row0 the first tile row this CTA holds (0, or BM for the odd CTA of a
// pair); partial tiles are dense TILE_M x BN.
template <int BM, int BN, int TILE_M = BM>
__device__ __forceinline__ void store_accumulator(uint32_t t_row, const Unit& w, int q,
                                                  int lane, const Epilogue& ep,
                                                  float* partial, float* stage,
                                                  int sub_row0 = 0) {
  if (ep.staged) {
    const int r0 = sub_row0 + q * 32;      // this warp's first row of the tile
    const int row0 = w.tm * TILE_M + r0;   // ... and of C
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      float v[32];
      tmem_ld32(t_row + ch * 32, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) stage[lane * EPI_STRIDE + i] = v[i];
      __syncwarp();
      // Column `lane` of the chunk, all 32 reads in flight at once.
#pragma unroll
      for (int r = 0; r < 32; ++r) v[r] = stage[r * EPI_STRIDE + lane];
      const int col = w.tn * BN + ch * 32 + lane;  // this lane's column of C
      if (w.pidx >= 0) {
        float* p = partial + static_cast<int64_t>(w.pidx) * (TILE_M * BN) +
                   static_cast<int64_t>(r0) * BN + ch * 32 + lane;
#pragma unroll
        for (int r = 0; r < 32; ++r, p += BN)
          if (bounds_ok(ep.bounds, SITE_PARTIAL, p - partial, 1, ep.partial_extent)) *p = v[r];
      } else if (col < ep.N && (!ep.bias || bounds_ok(ep.bounds, SITE_BIAS, col, 1, ep.N))) {
        const float bias_c = ep.bias ? ep.bias[col] : 0.0f;
        float* cp = ep.C + static_cast<int64_t>(row0) * ep.ldc + col;
        const int rows = min(32, ep.M - row0);
        if (ep.beta == 0.0f) {
#pragma unroll
          for (int r = 0; r < 32; ++r, cp += ep.ldc)
            if (r < rows && bounds_ok(ep.bounds, SITE_C_STORE, cp - ep.C, 1, ep.c_extent))
              *cp = ep.bias ? ep.alpha * v[r] + bias_c : ep.alpha * v[r];
        } else {
          // C is read too: row by row from the square, which is rewritten
          // only after the barrier below.
#pragma unroll 4
          for (int r = 0; r < rows; ++r, cp += ep.ldc) {
            if (!bounds_ok(ep.bounds, SITE_C_STORE, cp - ep.C, 1, ep.c_extent)) continue;
            float o = fmaf(ep.beta, *cp, ep.alpha * stage[r * EPI_STRIDE + lane]);
            if (ep.bias) o += bias_c;
            *cp = o;
          }
        }
      }
      __syncwarp();  // the square is read before the next chunk is written
    }
    return;
  }
  const int row = w.tm * TILE_M + sub_row0 + q * 32 + lane;
  float* c_row = ep.C + static_cast<int64_t>(row) * ep.ldc;
#pragma unroll 1
  for (int ch = 0; ch < BN / 32; ++ch) {
    float v[32];
    tmem_ld32(t_row + ch * 32, v);
    const int col0 = w.tn * BN + ch * 32;
    if (w.pidx >= 0) {
      float* prow = partial + static_cast<int64_t>(w.pidx) * (TILE_M * BN) +
                    (sub_row0 + q * 32 + lane) * BN + ch * 32;
#pragma unroll
      for (int g4 = 0; g4 < 8; ++g4)
        if (bounds_ok(ep.bounds, SITE_PARTIAL, (prow - partial) + 4 * g4, 4, ep.partial_extent))
          *reinterpret_cast<float4*>(prow + 4 * g4) =
              make_float4(v[4 * g4], v[4 * g4 + 1], v[4 * g4 + 2], v[4 * g4 + 3]);
    } else if (row < ep.M) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= ep.alpha;
      if (ep.vec_c) {
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4)
          if (col0 + 4 * g4 < ep.N &&
              bounds_ok(ep.bounds, SITE_C_STORE, (c_row - ep.C) + col0 + 4 * g4, 4,
                        ep.c_extent) &&
              (!ep.bias || bounds_ok(ep.bounds, SITE_BIAS, col0 + 4 * g4, 4, ep.N))) {
            float4* cp = reinterpret_cast<float4*>(c_row + col0 + 4 * g4);
            float4 o = make_float4(v[4 * g4], v[4 * g4 + 1], v[4 * g4 + 2], v[4 * g4 + 3]);
            if (ep.beta != 0.0f) {
              const float4 c0 = *cp;
              o = make_float4(fmaf(ep.beta, c0.x, o.x), fmaf(ep.beta, c0.y, o.y),
                              fmaf(ep.beta, c0.z, o.z), fmaf(ep.beta, c0.w, o.w));
            }
            if (ep.bias) {
              const int c = col0 + 4 * g4;
              o.x += ep.bias[c];
              o.y += ep.bias[c + 1];
              o.z += ep.bias[c + 2];
              o.w += ep.bias[c + 3];
            }
            *cp = o;
          }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i < ep.N &&
              bounds_ok(ep.bounds, SITE_C_STORE, (c_row - ep.C) + col0 + i, 1, ep.c_extent) &&
              (!ep.bias || bounds_ok(ep.bounds, SITE_BIAS, col0 + i, 1, ep.N))) {
            float o = ep.beta != 0.0f ? fmaf(ep.beta, c_row[col0 + i], v[i]) : v[i];
            if (ep.bias) o += ep.bias[col0 + i];
            c_row[col0 + i] = o;
          }
      }
    }
  }
}

}  // namespace tc
}  // namespace mt
