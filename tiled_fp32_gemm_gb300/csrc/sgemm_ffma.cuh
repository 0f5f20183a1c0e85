// CUDA-core fp32 GEMM: tiled, multi-stage, register-tile FFMA kernel.
//
// What it computes is the tiled matmul of "My Triton From Scratch, Part 14:
// Shared Memory Tiles" (section "Staging inside a runtime K loop": an
// accumulator that starts at zero takes the product of each staged A and B
// tile as K advances in steps of BK, then a masked store), with the
// physical choices of "Part 18: Shared Memory Optimization"
// and of the skills page "Optimize Shared Memory Tiling":
//
//  * tile scheduler — one CTA per BM x BN tile of C ("The canonical source
//    pattern": program_id -> tile origin), walked in a grouped raster so a
//    wave shares A and B panels in L2; the tiles past the last full wave are
//    either cut into K slices (split tail) or dealt out as stream-K runs of
//    K tiles across tile boundaries, one segment per tile a run touches,
//    whose pieces a second kernel adds in k order;
//  * masked staging — A[m0+r, k0+c] and B[k0+r, n0+c] are copied into a
//    shared stage, 0.0 where the element lies outside M, N or K ("Zero-filled
//    boundary tiles"); every shared slot is written, so all threads reach the
//    same barriers;
//  * padded shared rows — A rows are padded by the pages' bank rule counted
//    in 16-byte slots (section "Choosing padding instead of hard-coding it");
//    B rows are read as a broadcast and get no padding, as the rule says
//    (section "Why shared-memory banks matter", last paragraphs);
//  * A tiles row-major (As[m][k], a thread reads a float4 of four k of one
//    row) or K-major (As[k][m], a thread reads a float4 of four rows at one
//    k).  The K-major tile is read one k row at a time, so the rule gives
//    it no padding; filled from A stored K x M in 16-byte chunks, or
//    gathered from A stored M x K with 4-byte copies that write 8 k rows at
//    one column at once, for which the rule pads each row by one word
//    (rounded up to a float4).  Only the rows a thread owns change: 4 x 4
//    blocks instead of a stride of LM rows;
//  * K pipeline — STAGES shared stages filled by cp.async with zero fill,
//    one barrier per K tile (Part 18 "What ping-pong changes about
//    synchronization"; skills page step 7: commit, wait_group, then
//    __syncthreads), with STAGES-1 tiles in flight while one is computed.
//    STAGES = 1 is the single-buffer form the pages fall back to (Part 18
//    "One stage versus two stages": copy, barrier, compute, barrier), kept
//    to measure what the pipeline buys;
//  * unrolled register-tile micro-kernel — each thread keeps a TM x TN block
//    of C in registers and, for every k of the fixed-size BK loop (fully
//    unrolled, Part 18 "Unrolling the inner reduction loop"), reads its A
//    values (float4s) and float4s of B and issues TM*TN FMAs; the packed
//    form issues them as fma.rn.f32x2 pairs;
//  * masked epilogue — float4 or scalar stores where row < M and col < N.
//
// Every output is a sequence of fp32 FMAs in increasing k, one per k, so
// the scalar and the packed micro-kernels give bit-identical results.
#pragma once

#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kernels.h"
#include "smem_layout.cuh"

namespace mt {

// KSLICES_ > 1: the CTA's warps form KSLICES_ groups that each cover the
// whole tile for 1/KSLICES_ of every staged K tile's k steps (group g takes
// k steps g*BK/KSLICES_ ...); the groups' sums are added through shared
// memory at the end, group 0's first.  More warps per tile for grids with
// fewer tiles than SMs.
template <int BM_, int BN_, int BK_, int WM_, int WN_, int TM_, int TN_,
          int STAGES_, int MINB_, int KSLICES_ = 1>
struct FfmaTile {
  static constexpr int BM = BM_, BN = BN_, BK = BK_;
  static constexpr int WM = WM_, WN = WN_, TM = TM_, TN = TN_;
  static constexpr int STAGES = STAGES_, MIN_BLOCKS = MINB_;
  static constexpr int KSLICES = KSLICES_;
  static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
  static constexpr int TILE_WARPS = WARPS_M * WARPS_N;  // warps covering the tile once
  static constexpr int THREADS = TILE_WARPS * 32 * KSLICES;
  static_assert(BK % (4 * KSLICES) == 0, "each K slice takes whole float4 steps");
  // Shared memory the slice sums go through (groups 1.. of a sliced tile).
  static constexpr int REDUCE_BYTES = (KSLICES - 1) * BM * BN * 4;
  static constexpr int at_least_reduce(int bytes) {
    return bytes > REDUCE_BYTES ? bytes : REDUCE_BYTES;
  }
  static constexpr int LM = WM / TM;  // lanes of a warp along M
  static constexpr int LN = 32 / LM;  // lanes of a warp along N
  static_assert(BM % WM == 0 && BN % WN == 0, "warp tiles must cover the CTA tile");
  static_assert(WM % TM == 0 && LM * LN == 32 && LN * TN == WN, "lane layout");
  static_assert(TN % 4 == 0 && BK % 4 == 0, "float4 fragments");
  static_assert(LM <= 8, "at most 8 A rows per 8-lane phase");
  // Rows of A that the 8 lanes of one 16-byte access phase read at the same
  // k: lanes are numbered M-fastest, so a phase spans min(LM, 8) rows.
  static constexpr int A_SIMULTANEOUS_ROWS = LM < 8 ? LM : 8;

  static constexpr SmemLayout a_layout(bool pad) {
    return SmemLayout{BM, BK, pad ? vector_row_padding_rule(BK, A_SIMULTANEOUS_ROWS) : 0,
                      STAGES};
  }
  // Every lane of a warp reads the same k row of B: one row at a time, so
  // the rule gives no padding.  A transposed B is written instead 8 k rows
  // at a time at the same column (the staging's lane blocks): the scalar
  // rule asks for one padding word there, rounded up to a float4 so rows
  // stay 16-byte aligned for the reads.
  static constexpr int B_TRANS_PAD = (row_padding_rule(BN, 8) + 3) / 4 * 4;
  static constexpr SmemLayout b_layout(bool pad, bool trans = false) {
    return SmemLayout{BK, BN,
                      trans ? B_TRANS_PAD : (pad ? vector_row_padding_rule(BN, 1) : 0), STAGES};
  }
  static constexpr int smem_bytes(bool pad, bool trans_b = false) {
    return at_least_reduce(a_layout(pad).nbytes() + b_layout(pad, trans_b).nbytes());
  }
  // A staged K-major (As[k][m]): a warp reads one k row at a time, float4s
  // of four consecutive rows of A, so the rule gives no padding.
  static constexpr SmemLayout a_layout_kmajor() {
    return SmemLayout{BK, BM, vector_row_padding_rule(BM, 1), STAGES};
  }
  static constexpr int smem_bytes_kmajor() {
    return at_least_reduce(a_layout_kmajor().nbytes() + b_layout(true).nbytes());
  }
  // A gathered K-major from row-major storage: the copies write 8 k rows at
  // the same column at once, so the scalar rule asks for one padding word,
  // rounded up to a float4 to keep rows 16-byte aligned for the reads.
  static constexpr int A_GATHER_PAD = (row_padding_rule(BM, 8) + 3) / 4 * 4;
  static constexpr SmemLayout a_layout_gather() {
    return SmemLayout{BK, BM, A_GATHER_PAD, STAGES};
  }
  static constexpr int smem_bytes_gather() {
    return at_least_reduce(a_layout_gather().nbytes() + b_layout(true).nbytes());
  }
};

// ---------------------------------------------------------------------------
// Global -> shared staging of one K tile: A (BM x BK) into As[r][c] and B
// (BK x BN) into Bs[kk][n], 0.0 where the element lies outside M, N or K.
//   STAGE_VEC    16-byte chunks along the contiguous dimension (operand not
//                transposed, leading dimension % 4 == 0, 16-byte aligned);
//   STAGE_SCALAR 4-byte elements, threads along the contiguous dimension;
//   STAGE_TRANS  4-byte elements of a transposed operand (A stored K x M, B
//                stored N x K); a warp copies 8 x 4 blocks, 8 lanes along
//                the contiguous dimension, so global reads stay within
//                32-byte sectors and the shared writes land in 32 distinct
//                banks.
//   STAGE_KMAJOR A only: A stored K x M (M % 4 == 0, lda % 4 == 0, 16-byte
//                aligned) copied in 16-byte chunks along M into a K-major
//                tile As[k][m]; the micro-kernel then reads four rows of A
//                with one float4.
//   STAGE_GATHER A only: A stored M x K (any lda and alignment) copied
//                element by element into the same K-major tile; a warp
//                copies 8 x 4 blocks, 8 lanes along K.
enum StageMode {
  STAGE_VEC = 0,
  STAGE_SCALAR = 1,
  STAGE_TRANS = 2,
  STAGE_KMAJOR = 3,
  STAGE_GATHER = 4
};

template <class T, int MODE>
struct AStage;
template <class T, int MODE>
struct BStage;

template <class T>
struct AStage<T, STAGE_VEC> {
  static constexpr int CHUNKS_ROW = T::BK / 4;
  static_assert(T::THREADS % CHUNKS_ROW == 0, "");
  static constexpr int ROWS_STEP = T::THREADS / CHUNKS_ROW;
  static constexpr int ITERS = T::BM / ROWS_STEP;
  static_assert(ITERS * ROWS_STEP == T::BM && ITERS <= 32, "");
  const float* base;  // any valid address, read by nothing (masked chunks)
  const float* src;   // A[(m0 + row) * lda + col]
  int64_t row_step;   // ROWS_STEP * lda
  int row, col, K;
  uint32_t rows_ok;   // bit t: row t of this thread's chunks is inside M
  int64_t extent;     // checked builds: elements of A
  BoundsRecord* rec;

  __device__ AStage(const GemmArgs& a, int m0, int tid)
      : base(a.A), K(a.K), extent(a.a_extent), rec(a.bounds) {
    row = tid / CHUNKS_ROW;
    col = (tid % CHUNKS_ROW) * 4;
    row_step = static_cast<int64_t>(ROWS_STEP) * a.lda;
    src = a.A + static_cast<int64_t>(m0 + row) * a.lda + col;
    rows_ok = 0;
#pragma unroll
    for (int t = 0; t < ITERS; ++t)
      if (m0 + row + t * ROWS_STEP < a.M) rows_ok |= 1u << t;
  }
  template <class L>
  __device__ __forceinline__ void load(float* As, const L& la, int stage, int kt) const {
    const int k0 = kt * T::BK;
    const bool k_ok = k0 + col < K;
#pragma unroll
    for (int t = 0; t < ITERS; ++t) {
      const float* g = src + t * row_step + k0;
      const int so = la.offset(stage, row + t * ROWS_STEP, col);
      const bool ok = k_ok && (rows_ok >> t & 1u) &&
                      bounds_ok(rec, SITE_A_LOAD, g - base, 4, extent);
      if (bounds_ok(rec, SITE_A_SMEM, so, 4, la.size()))
        cp_async_16(smem_u32(As + so), ok ? g : base, ok ? 16u : 0u);
    }
  }
};

template <class T>
struct AStage<T, STAGE_SCALAR> {
  static_assert(T::THREADS % T::BK == 0, "");
  static constexpr int ROWS_STEP = T::THREADS / T::BK;
  static constexpr int ITERS = T::BM / ROWS_STEP;
  static_assert(ITERS <= 32, "");
  const float* base;
  const float* src;
  int64_t row_step;
  int row, col, K;
  uint32_t rows_ok;
  int64_t extent;
  BoundsRecord* rec;

  __device__ AStage(const GemmArgs& a, int m0, int tid)
      : base(a.A), K(a.K), extent(a.a_extent), rec(a.bounds) {
    row = tid / T::BK;
    col = tid % T::BK;
    row_step = static_cast<int64_t>(ROWS_STEP) * a.lda;
    src = a.A + static_cast<int64_t>(m0 + row) * a.lda + col;
    rows_ok = 0;
#pragma unroll
    for (int t = 0; t < ITERS; ++t)
      if (m0 + row + t * ROWS_STEP < a.M) rows_ok |= 1u << t;
  }
  template <class L>
  __device__ __forceinline__ void load(float* As, const L& la, int stage, int kt) const {
    const int k0 = kt * T::BK;
    const bool k_ok = k0 + col < K;
#pragma unroll
    for (int t = 0; t < ITERS; ++t) {
      const float* g = src + t * row_step + k0;
      const int so = la.offset(stage, row + t * ROWS_STEP, col);
      const bool ok = k_ok && (rows_ok >> t & 1u) &&
                      bounds_ok(rec, SITE_A_LOAD, g - base, 1, extent);
      if (bounds_ok(rec, SITE_A_SMEM, so, 1, la.size()))
        cp_async_4(smem_u32(As + so), ok ? g : base, ok ? 4u : 0u);
    }
  }
};

template <class T>
struct AStage<T, STAGE_TRANS> {
  // Lane l copies row 8*rb + l%8, column 4*cb + l/8 of block b = warp +
  // t*NW (rb = b % RB, cb = b / RB) from At[(k0 + column) * lda + m0 + row].
  static constexpr int RB = T::BM / 8, CB = T::BK / 4;
  static constexpr int NW = T::THREADS / 32;
  static constexpr int ITERS = RB * CB / NW;
  static_assert(ITERS * NW == RB * CB, "");
  const float* At;
  int64_t lda;
  int M, K, m0, lr, lc, warp;
  int64_t extent;
  BoundsRecord* rec;

  __device__ AStage(const GemmArgs& a, int m0_, int tid)
      : At(a.A), lda(a.lda), M(a.M), K(a.K), m0(m0_), extent(a.a_extent), rec(a.bounds) {
    lr = tid & 7;
    lc = (tid & 31) >> 3;
    warp = tid >> 5;
  }
  template <class L>
  __device__ __forceinline__ void load(float* As, const L& la, int stage, int kt) const {
    const int k0 = kt * T::BK;
#pragma unroll
    for (int t = 0; t < ITERS; ++t) {
      const int b = warp + t * NW;
      const int r = (b % RB) * 8 + lr, c = (b / RB) * 4 + lc;
      const int64_t go = static_cast<int64_t>(k0 + c) * lda + m0 + r;
      const int so = la.offset(stage, r, c);
      const bool ok = m0 + r < M && k0 + c < K && bounds_ok(rec, SITE_A_LOAD, go, 1, extent);
      if (bounds_ok(rec, SITE_A_SMEM, so, 1, la.size()))
        cp_async_4(smem_u32(As + so), ok ? At + go : At, ok ? 4u : 0u);
    }
  }
};

template <class T>
struct AStage<T, STAGE_KMAJOR> {
  static constexpr int CHUNKS_ROW = T::BM / 4;
  static_assert(T::THREADS % CHUNKS_ROW == 0, "");
  static constexpr int ROWS_STEP = T::THREADS / CHUNKS_ROW;
  static constexpr int ITERS = T::BK / ROWS_STEP;
  static_assert(ITERS * ROWS_STEP == T::BK, "");
  const float* base;
  const float* src;  // At[k * lda + m0 + col], k = this thread's first row
  int64_t lda, row_step;
  int row, col, K;
  bool col_ok;
  int64_t extent;
  BoundsRecord* rec;

  __device__ AStage(const GemmArgs& a, int m0, int tid)
      : base(a.A), lda(a.lda), K(a.K), extent(a.a_extent), rec(a.bounds) {
    row = tid / CHUNKS_ROW;
    col = (tid % CHUNKS_ROW) * 4;
    row_step = static_cast<int64_t>(ROWS_STEP) * a.lda;
    src = a.A + static_cast<int64_t>(row) * a.lda + m0 + col;
    col_ok = m0 + col < a.M;
  }
  template <class L>
  __device__ __forceinline__ void load(float* As, const L& la, int stage, int kt) const {
    const int k0 = kt * T::BK;
#pragma unroll
    for (int t = 0; t < ITERS; ++t) {
      const float* g = src + static_cast<int64_t>(k0) * lda + t * row_step;
      const int so = la.offset(stage, row + t * ROWS_STEP, col);
      const bool ok = col_ok && k0 + row + t * ROWS_STEP < K &&
                      bounds_ok(rec, SITE_A_LOAD, g - base, 4, extent);
      if (bounds_ok(rec, SITE_A_SMEM, so, 4, la.size()))
        cp_async_16(smem_u32(As + so), ok ? g : base, ok ? 16u : 0u);
    }
  }
};

template <class T>
struct AStage<T, STAGE_GATHER> {
  // Lane l copies k = 8*kb + l%8 and m = 4*mb + l/8 of block b = warp +
  // t*NW (kb = b % KB, mb = b / KB) from A[(m0 + m) * lda + k0 + k].  With
  // NW a multiple of KB a thread's k is fixed and its m advances by M_STEP.
  // Eight lanes read 32 consecutive bytes of one row of A; the row stride
  // BM + 4 is 4 (mod 32) words, so a warp's 32 shared writes (8 k x 4 m)
  // land in 32 distinct banks.
  static constexpr int KB = T::BK / 8, MB = T::BM / 4;
  static constexpr int NW = T::THREADS / 32;
  static_assert(T::BK % 8 == 0 && NW % KB == 0, "gather blocks");
  static constexpr int ITERS = KB * MB / NW;
  static constexpr int M_STEP = NW / KB * 4;
  static_assert(ITERS * NW == KB * MB && ITERS <= 32, "");
  const float* base;
  const float* src;  // A[(m0 + m_first) * lda + k_off]
  int64_t row_step;  // M_STEP * lda
  int k_off, m_first, K;
  uint32_t rows_ok;  // bit t: row m0 + m_first + t*M_STEP is inside M
  int64_t extent;
  BoundsRecord* rec;

  __device__ AStage(const GemmArgs& a, int m0, int tid)
      : base(a.A), K(a.K), extent(a.a_extent), rec(a.bounds) {
    const int warp = tid >> 5, lane = tid & 31;
    k_off = (warp % KB) * 8 + (lane & 7);
    m_first = (warp / KB) * 4 + (lane >> 3);
    row_step = static_cast<int64_t>(M_STEP) * a.lda;
    src = a.A + static_cast<int64_t>(m0 + m_first) * a.lda + k_off;
    rows_ok = 0;
#pragma unroll
    for (int t = 0; t < ITERS; ++t)
      if (m0 + m_first + t * M_STEP < a.M) rows_ok |= 1u << t;
  }
  template <class L>
  __device__ __forceinline__ void load(float* As, const L& la, int stage, int kt) const {
    const int k0 = kt * T::BK;
    const bool k_ok = k0 + k_off < K;
#pragma unroll
    for (int t = 0; t < ITERS; ++t) {
      const float* g = src + t * row_step + k0;
      const int so = la.offset(stage, k_off, m_first + t * M_STEP);
      const bool ok = k_ok && (rows_ok >> t & 1u) &&
                      bounds_ok(rec, SITE_A_LOAD, g - base, 1, extent);
      if (bounds_ok(rec, SITE_A_SMEM, so, 1, la.size()))
        cp_async_4(smem_u32(As + so), ok ? g : base, ok ? 4u : 0u);
    }
  }
};

template <class T>
struct BStage<T, STAGE_VEC> {
  static constexpr int CHUNKS_ROW = T::BN / 4;
  static_assert(T::THREADS % CHUNKS_ROW == 0, "");
  static constexpr int ROWS_STEP = T::THREADS / CHUNKS_ROW;
  static constexpr int ITERS = T::BK / ROWS_STEP;
  static_assert(ITERS * ROWS_STEP == T::BK, "");
  const float* base;
  const float* src;   // B[row * ldb + n0 + col]
  int64_t ldb, row_step;
  int row, col, K;
  bool col_ok;
  int64_t extent;
  BoundsRecord* rec;

  __device__ BStage(const GemmArgs& a, int n0, int tid)
      : base(a.B), ldb(a.ldb), K(a.K), extent(a.b_extent), rec(a.bounds) {
    row = tid / CHUNKS_ROW;
    col = (tid % CHUNKS_ROW) * 4;
    row_step = static_cast<int64_t>(ROWS_STEP) * a.ldb;
    src = a.B + static_cast<int64_t>(row) * a.ldb + n0 + col;
    col_ok = n0 + col < a.N;
  }
  template <class L>
  __device__ __forceinline__ void load(float* Bs, const L& lb, int stage, int kt) const {
    const int k0 = kt * T::BK;
#pragma unroll
    for (int t = 0; t < ITERS; ++t) {
      const float* g = src + static_cast<int64_t>(k0) * ldb + t * row_step;
      const int so = lb.offset(stage, row + t * ROWS_STEP, col);
      const bool ok = col_ok && k0 + row + t * ROWS_STEP < K &&
                      bounds_ok(rec, SITE_B_LOAD, g - base, 4, extent);
      if (bounds_ok(rec, SITE_B_SMEM, so, 4, lb.size()))
        cp_async_16(smem_u32(Bs + so), ok ? g : base, ok ? 16u : 0u);
    }
  }
};

template <class T>
struct BStage<T, STAGE_SCALAR> {
  static_assert(T::THREADS % T::BN == 0, "");
  static constexpr int ROWS_STEP = T::THREADS / T::BN;
  static constexpr int ITERS = T::BK / ROWS_STEP;
  const float* base;
  const float* src;
  int64_t ldb, row_step;
  int row, col, K;
  bool col_ok;
  int64_t extent;
  BoundsRecord* rec;

  __device__ BStage(const GemmArgs& a, int n0, int tid)
      : base(a.B), ldb(a.ldb), K(a.K), extent(a.b_extent), rec(a.bounds) {
    row = tid / T::BN;
    col = tid % T::BN;
    row_step = static_cast<int64_t>(ROWS_STEP) * a.ldb;
    src = a.B + static_cast<int64_t>(row) * a.ldb + n0 + col;
    col_ok = n0 + col < a.N;
  }
  template <class L>
  __device__ __forceinline__ void load(float* Bs, const L& lb, int stage, int kt) const {
    const int k0 = kt * T::BK;
#pragma unroll
    for (int t = 0; t < ITERS; ++t) {
      const float* g = src + static_cast<int64_t>(k0) * ldb + t * row_step;
      const int so = lb.offset(stage, row + t * ROWS_STEP, col);
      const bool ok = col_ok && k0 + row + t * ROWS_STEP < K &&
                      bounds_ok(rec, SITE_B_LOAD, g - base, 1, extent);
      if (bounds_ok(rec, SITE_B_SMEM, so, 1, lb.size()))
        cp_async_4(smem_u32(Bs + so), ok ? g : base, ok ? 4u : 0u);
    }
  }
};

template <class T>
struct BStage<T, STAGE_TRANS> {
  // Lane l copies k row 8*kb + l%8, column 4*nb + l/8 of block b = warp +
  // t*NW (kb = b % KB, nb = b / KB) from Bt[(n0 + column) * ldb + k0 + row].
  static constexpr int KB = T::BK / 8, NB = T::BN / 4;
  static constexpr int NW = T::THREADS / 32;
  static constexpr int ITERS = KB * NB / NW;
  static_assert(ITERS * NW == KB * NB, "");
  const float* Bt;
  int64_t ldb;
  int N, K, n0, lk, ln, warp;
  int64_t extent;
  BoundsRecord* rec;

  __device__ BStage(const GemmArgs& a, int n0_, int tid)
      : Bt(a.B), ldb(a.ldb), N(a.N), K(a.K), n0(n0_), extent(a.b_extent), rec(a.bounds) {
    lk = tid & 7;
    ln = (tid & 31) >> 3;
    warp = tid >> 5;
  }
  template <class L>
  __device__ __forceinline__ void load(float* Bs, const L& lb, int stage, int kt) const {
    const int k0 = kt * T::BK;
#pragma unroll
    for (int t = 0; t < ITERS; ++t) {
      const int b = warp + t * NW;
      const int kk = (b % KB) * 8 + lk, n = (b / KB) * 4 + ln;
      const int64_t go = static_cast<int64_t>(n0 + n) * ldb + k0 + kk;
      const int so = lb.offset(stage, kk, n);
      const bool ok = n0 + n < N && k0 + kk < K && bounds_ok(rec, SITE_B_LOAD, go, 1, extent);
      if (bounds_ok(rec, SITE_B_SMEM, so, 1, lb.size()))
        cp_async_4(smem_u32(Bs + so), ok ? Bt + go : Bt, ok ? 4u : 0u);
    }
  }
};

__device__ __forceinline__ float pick(const float4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// A float4 fragment read from a staged region of `size` floats (a checked
// build reads zeros for one outside it and records it).
__device__ __forceinline__ float4 frag4(const float* region, const float* p, int size,
                                        BoundsRecord* rec) {
  if (!bounds_ok(rec, SITE_FRAG, p - region, 4, size)) return make_float4(0.f, 0.f, 0.f, 0.f);
  return *reinterpret_cast<const float4*>(p);
}

// ---------------------------------------------------------------------------
// AMODE, BMODE: StageMode of each operand.  VEC_C: C is written with float4
// stores (N % 4 == 0, ldc % 4 == 0, C 16-byte aligned), else with scalar
// stores.
template <class T, int AMODE, int BMODE, bool PAD, bool PACKED,
          bool VEC_C = (AMODE == STAGE_VEC)>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
    sgemm_ffma_kernel(GemmArgs args) {
  constexpr bool VEC = VEC_C;
  constexpr bool KMAJOR = AMODE == STAGE_KMAJOR || AMODE == STAGE_GATHER;
  static_assert(!KMAJOR || T::TM % 4 == 0, "K-major A reads rows in fours");
  constexpr SmemLayout LA = AMODE == STAGE_GATHER ? T::a_layout_gather()
                            : KMAJOR              ? T::a_layout_kmajor()
                                                  : T::a_layout(PAD);
  constexpr SmemLayout LB = T::b_layout(PAD, BMODE == STAGE_TRANS);
  extern __shared__ float4 smem_f4[];
  float* As = reinterpret_cast<float*>(smem_f4);
  float* Bs = As + LA.size();

  const int M = args.M, N = args.N, K = args.K;
  const int tid = threadIdx.x;
  // Launched as a programmatic dependent of the operand copy before it on
  // the stream: wait until the copies are complete and visible (a no-op
  // when launched without the attribute).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Work unit: a whole tile; one K slice of a tile of the split tail; or a
  // stream-K run of K tiles across tile boundaries, taken as one segment
  // per tile it touches.  A segment's fp32 partial goes to the workspace
  // instead of C unless it covers its tile whole.
  const int ktiles_all = (K + T::BK - 1) / T::BK;
  const int unit = blockIdx.x;
  const bool streamk = args.sk_ctas > 0 && unit >= args.full_tiles;
  const int sk_unit = unit - args.full_tiles;
  int64_t run_begin = 0, run_end = 0, run_at = 0;
  if (streamk) {
    run_begin = static_cast<int64_t>(sk_unit) * args.sk_iters / args.sk_ctas;
    run_end = static_cast<int64_t>(sk_unit + 1) * args.sk_iters / args.sk_ctas;
    run_at = run_begin;
  }
  for (int segment = 0;; ++segment) {
    int tile = unit, kt_begin = 0, kt_end = ktiles_all;
    int64_t partial_slot = -1;  // < 0: the segment's tile goes to C
    if (streamk) {
      if (run_at >= run_end) break;
      const int64_t t_rel = run_at / ktiles_all;
      tile = args.full_tiles + static_cast<int>(t_rel);
      kt_begin = static_cast<int>(run_at - t_rel * ktiles_all);
      kt_end = static_cast<int>(
          min(static_cast<int64_t>(ktiles_all), kt_begin + (run_end - run_at)));
      if (kt_begin > 0 || kt_end < ktiles_all)
        partial_slot = 2 * static_cast<int64_t>(sk_unit) + (run_at == run_begin ? 0 : 1);
      run_at += kt_end - kt_begin;
      if (segment > 0) {
        // The stages and the K-group sums of the previous segment are reused:
        // every copy must have landed and every thread be past its reads.
        cp_async_wait<0>();
        __syncthreads();
      }
    } else {
      if (segment > 0) break;
      if (unit >= args.full_tiles) {
        const int v = unit - args.full_tiles;
        tile = args.full_tiles + v / args.split;
        const int slice = v % args.split;
        kt_begin = min(ktiles_all, slice * args.kt_per_slice);
        kt_end = min(ktiles_all, kt_begin + args.kt_per_slice);
        partial_slot = v;  // slice-major per tile
      }
    }
    const int ktiles = kt_end - kt_begin;
    int tm, tn;
    grouped_tile(tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
    const int m0 = tm * T::BM, n0 = tn * T::BN;

    const AStage<T, AMODE> stage_a(args, m0, tid);
    const BStage<T, BMODE> stage_b(args, n0, tid);

    // Prologue: STAGES-1 tiles in flight.  One commit group per tile (empty
    // groups keep the count uniform when K has fewer tiles).
#pragma unroll
    for (int s = 0; s < T::STAGES - 1; ++s) {
      if (s < ktiles) {
        stage_a.load(As, LA, s, kt_begin + s);
        stage_b.load(Bs, LB, s, kt_begin + s);
      }
      cp_async_commit();
    }

    // Warp `warp` of K group kg (kg = 0 without K slices).
    const int kg = tid / 32 / T::TILE_WARPS;
    const int warp = tid / 32 % T::TILE_WARPS, lane = tid % 32;
    const int wm = warp / T::WARPS_N, wn = warp % T::WARPS_N;
    const int lm = lane % T::LM, ln = lane / T::LM;
    // Thread (lm, ln) of warp (wm, wn) owns rows wm*WM + i*LM + lm (i < TM)
    // and columns wn*WN + g*LN*4 + ln*4 + c (g < TN/4, c < 4).  With A
    // K-major the rows come in fours: wm*WM + (i/4)*LM*4 + lm*4 + i%4.
    const auto row_of = [&](int i) {
      return KMAJOR ? wm * T::WM + (i / 4) * T::LM * 4 + lm * 4 + i % 4
                    : wm * T::WM + i * T::LM + lm;
    };
    // This group's first k step within a staged K tile.
    constexpr int KS_STEPS = T::BK / T::KSLICES;
    const int k_first = kg * KS_STEPS;
    const int a_off = KMAJOR ? LA.offset(0, k_first, wm * T::WM + lm * 4)
                             : LA.offset(0, wm * T::WM + lm, k_first);
    const int b_off = LB.offset(0, k_first, wn * T::WN + ln * 4);

    float2 acc[T::TM][T::TN / 2];
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
#pragma unroll
      for (int j = 0; j < T::TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);

    int stage = 0;
    int load_stage = T::STAGES - 1;
    for (int kt = 0; kt < ktiles; ++kt) {
      if constexpr (T::STAGES == 1) {
        // One stage, no double buffering (the pages' fallback form): copy
        // tile kt, wait for it, barrier, compute, and a second barrier below
        // before the next copy overwrites the stage.  Nothing overlaps the
        // copies.
        stage_a.load(As, LA, 0, kt_begin + kt);
        stage_b.load(Bs, LB, 0, kt_begin + kt);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
      } else {
        // Tile kt has landed for this thread; the barrier makes every
        // thread's copies visible and guarantees that the stage refilled
        // below (read in iteration kt-1) is no longer being read.
        cp_async_wait<T::STAGES - 2>();
        __syncthreads();
        if (kt + T::STAGES - 1 < ktiles) {
          stage_a.load(As, LA, load_stage, kt_begin + kt + T::STAGES - 1);
          stage_b.load(Bs, LB, load_stage, kt_begin + kt + T::STAGES - 1);
        }
        cp_async_commit();
      }

      const float* a_ptr = As + stage * LA.stage_size() + a_off;
      const float* b_ptr = Bs + stage * LB.stage_size() + b_off;
#pragma unroll
      for (int k4 = 0; k4 < KS_STEPS / 4; ++k4) {
        // Row-major A: one float4 of four k per row, used over the next four
        // k.  K-major A: one float4 of four rows per k.
        float4 a[KMAJOR ? 1 : T::TM];
        if constexpr (!KMAJOR) {
#pragma unroll
          for (int i = 0; i < T::TM; ++i)
            a[i] = frag4(As, a_ptr + i * T::LM * LA.row_stride() + k4 * 4, LA.size(), args.bounds);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          float4 ak[KMAJOR ? T::TM / 4 : 1];
          if constexpr (KMAJOR) {
#pragma unroll
            for (int q = 0; q < T::TM / 4; ++q)
              ak[q] = frag4(As, a_ptr + (k4 * 4 + kk) * LA.row_stride() + q * T::LM * 4, LA.size(),
                            args.bounds);
          }
          float4 b[T::TN / 4];
#pragma unroll
          for (int g = 0; g < T::TN / 4; ++g)
            b[g] = frag4(Bs, b_ptr + (k4 * 4 + kk) * LB.row_stride() + g * T::LN * 4, LB.size(),
                         args.bounds);
#pragma unroll
          for (int g = 0; g < T::TN / 4; ++g) {
#pragma unroll
            for (int i = 0; i < T::TM; ++i) {
              const float av = KMAJOR ? pick(ak[i / 4], i % 4) : pick(a[i], kk);
              if constexpr (PACKED) {
                const float2 a2 = make_float2(av, av);
                acc[i][2 * g] = __ffma2_rn(a2, make_float2(b[g].x, b[g].y), acc[i][2 * g]);
                acc[i][2 * g + 1] = __ffma2_rn(a2, make_float2(b[g].z, b[g].w), acc[i][2 * g + 1]);
              } else {
                acc[i][2 * g].x = fmaf(av, b[g].x, acc[i][2 * g].x);
                acc[i][2 * g].y = fmaf(av, b[g].y, acc[i][2 * g].y);
                acc[i][2 * g + 1].x = fmaf(av, b[g].z, acc[i][2 * g + 1].x);
                acc[i][2 * g + 1].y = fmaf(av, b[g].w, acc[i][2 * g + 1].y);
              }
            }
          }
        }
      }
      if constexpr (T::STAGES == 1) __syncthreads();  // every read of the stage is done
      stage = stage + 1 == T::STAGES ? 0 : stage + 1;
      load_stage = load_stage + 1 == T::STAGES ? 0 : load_stage + 1;
    }

    if constexpr (T::KSLICES > 1) {
      // Add the K groups' sums through shared memory (the stages are free once
      // every copy has landed and every thread is past its last read): groups
      // 1.. store theirs, group 0 adds them in group order and goes on alone.
      cp_async_wait<0>();
      __syncthreads();
      float* red = reinterpret_cast<float*>(smem_f4);
      if (kg > 0) {
        float* mine = red + (kg - 1) * (T::BM * T::BN);
#pragma unroll
        for (int i = 0; i < T::TM; ++i) {
          const int r = row_of(i);
#pragma unroll
          for (int g = 0; g < T::TN / 4; ++g) {
            const int c = wn * T::WN + g * T::LN * 4 + ln * 4;
            if (bounds_ok(args.bounds, SITE_SLICE_SUM, (mine - red) + r * T::BN + c, 4,
                          T::REDUCE_BYTES / 4))
              *reinterpret_cast<float4*>(mine + r * T::BN + c) =
                  make_float4(acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x,
                              acc[i][2 * g + 1].y);
          }
        }
      }
      __syncthreads();
      if (kg > 0) continue;  // group 0 finishes the segment
#pragma unroll
      for (int s_ = 1; s_ < T::KSLICES; ++s_) {
        const float* other = red + (s_ - 1) * (T::BM * T::BN);
#pragma unroll
        for (int i = 0; i < T::TM; ++i) {
          const int r = row_of(i);
#pragma unroll
          for (int g = 0; g < T::TN / 4; ++g) {
            const int c = wn * T::WN + g * T::LN * 4 + ln * 4;
            const float4 o = frag4(red, other + r * T::BN + c, T::REDUCE_BYTES / 4, args.bounds);
            acc[i][2 * g].x += o.x;
            acc[i][2 * g].y += o.y;
            acc[i][2 * g + 1].x += o.z;
            acc[i][2 * g + 1].y += o.w;
          }
        }
      }
    }

    if (partial_slot >= 0) {
      // The segment's partial tile, dense BM x BN (rows and columns past M or
      // N hold zeros from the zero-filled staging and are never read back).
      float* P = args.partial + partial_slot * (T::BM * T::BN);
#pragma unroll
      for (int i = 0; i < T::TM; ++i) {
        const int r = row_of(i);
#pragma unroll
        for (int g = 0; g < T::TN / 4; ++g) {
          const int c = wn * T::WN + g * T::LN * 4 + ln * 4;
          if (bounds_ok(args.bounds, SITE_PARTIAL, (P - args.partial) + r * T::BN + c, 4,
                        args.partial_extent))
            *reinterpret_cast<float4*>(P + r * T::BN + c) =
                make_float4(acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x,
                            acc[i][2 * g + 1].y);
        }
      }
      continue;
    }

    // Masked epilogue: C[row, col] = alpha * acc + beta * C[row, col]
    // (+ bias[col]) for row < M, col < N (C is not read when beta == 0;
    // alpha == 1, beta == 0 and no bias store acc unchanged).
    float* C = args.C;
    const float alpha = args.alpha, beta = args.beta;
    const float* bias = args.bias;
#pragma unroll
    for (int i = 0; i < T::TM; ++i) {
      const int row = m0 + row_of(i);
      if (row >= M) continue;
      float* c_row = C + static_cast<int64_t>(row) * args.ldc;
#pragma unroll
      for (int g = 0; g < T::TN / 4; ++g) {
        const int col = n0 + wn * T::WN + g * T::LN * 4 + ln * 4;
        float4 v = make_float4(alpha * acc[i][2 * g].x, alpha * acc[i][2 * g].y,
                               alpha * acc[i][2 * g + 1].x, alpha * acc[i][2 * g + 1].y);
        if constexpr (VEC) {
          // N % 4 == 0, so a float4 group is either wholly inside or outside.
          if (col < N &&
              bounds_ok(args.bounds, SITE_C_STORE, (c_row - C) + col, 4, args.c_extent) &&
              (!bias || bounds_ok(args.bounds, SITE_BIAS, col, 4, N))) {
            float4* cp = reinterpret_cast<float4*>(c_row + col);
            if (beta != 0.0f) {
              const float4 o = *cp;
              v = make_float4(fmaf(beta, o.x, v.x), fmaf(beta, o.y, v.y), fmaf(beta, o.z, v.z),
                              fmaf(beta, o.w, v.w));
            }
            if (bias) {
              v.x += bias[col];
              v.y += bias[col + 1];
              v.z += bias[col + 2];
              v.w += bias[col + 3];
            }
            *cp = v;
          }
        } else {
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (col + e < N &&
                bounds_ok(args.bounds, SITE_C_STORE, (c_row - C) + col + e, 1, args.c_extent) &&
                (!bias || bounds_ok(args.bounds, SITE_BIAS, col + e, 1, N))) {
              float o = beta != 0.0f ? fmaf(beta, c_row[col + e], vv[e]) : vv[e];
              if (bias) o += bias[col + e];
              c_row[col + e] = o;
            }
        }
      }
    }
  }  // segment
}

// Only the kernels a flag asks for are instantiated (the others stay
// nullptr in the entry).
template <class T, bool PACKED, bool WITH_UNPADDED, bool WITH_TRANS = false,
          bool WITH_KMAJOR = false>
FfmaEntry make_entry() {
  FfmaEntry e{};
  e.bm = T::BM;
  e.bn = T::BN;
  e.bk = T::BK;
  e.stages = T::STAGES;
  e.threads = T::THREADS;
  e.kslices = T::KSLICES;
  e.min_blocks = T::MIN_BLOCKS;
  e.wm = T::WM;
  e.wn = T::WN;
  e.tm = T::TM;
  e.tn = T::TN;
  e.packed = PACKED ? 1 : 0;
  e.pad_a = T::a_layout(true).row_padding;
  e.pad_b = T::b_layout(true).row_padding;
  e.smem_bytes[0] = T::smem_bytes(false);
  e.smem_bytes[1] = T::smem_bytes(true);
  e.kern[1][1] = reinterpret_cast<const void*>(
      &sgemm_ffma_kernel<T, STAGE_VEC, STAGE_VEC, true, PACKED>);
  e.kern[0][1] = reinterpret_cast<const void*>(
      &sgemm_ffma_kernel<T, STAGE_SCALAR, STAGE_SCALAR, true, PACKED>);
  if constexpr (WITH_UNPADDED) {
    e.kern[1][0] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_VEC, STAGE_VEC, false, PACKED>);
    e.kern[0][0] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_SCALAR, STAGE_SCALAR, false, PACKED>);
  }
  if constexpr (WITH_KMAJOR) {
    e.smem_bytes_km = T::smem_bytes_kmajor();
    e.smem_bytes_kg = T::smem_bytes_gather();
    e.pad_a_kg = T::A_GATHER_PAD;
    e.kern_kg[1] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_GATHER, STAGE_VEC, true, PACKED, true>);
    e.kern_kg[0] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_GATHER, STAGE_VEC, true, PACKED, false>);
    e.kern_km[1] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_KMAJOR, STAGE_VEC, true, PACKED, true>);
    e.kern_km[0] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_KMAJOR, STAGE_VEC, true, PACKED, false>);
  }
  e.pad_b_t = T::b_layout(true, true).row_padding;
  e.smem_bytes_t = T::smem_bytes(true, true);
  if constexpr (WITH_TRANS) {
    e.kern_t[1][0] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_TRANS, STAGE_SCALAR, true, PACKED>);
    e.kern_t[0][1] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_SCALAR, STAGE_TRANS, true, PACKED>);
    e.kern_t[1][1] = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_TRANS, STAGE_TRANS, true, PACKED>);
    e.kern_vsc = reinterpret_cast<const void*>(
        &sgemm_ffma_kernel<T, STAGE_VEC, STAGE_VEC, true, PACKED, false>);
  }
  return e;
}

}  // namespace mt
