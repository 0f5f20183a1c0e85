// CUDA-core fp32 GEMM: tiled, multi-stage, register-tile FFMA kernel.
//
// What it computes is the tiled matmul of "My Triton From Scratch, Part 14:
// Shared Memory Tiles" (section "Staging inside a runtime K loop": acc =
// zeros; for k_base in range(0, K, BK): acc += dot(A tile, B tile); masked
// store), with the physical choices of "Part 18: Shared Memory Optimization"
// and of the skills page "Optimize Shared Memory Tiling":
//
//  * tile scheduler — one CTA per BM x BN tile of C ("The canonical source
//    pattern": program_id -> tile origin), walked in a grouped raster so a
//    wave shares A and B panels in L2;
//  * masked staging — A[m0+r, k0+c] and B[k0+r, n0+c] are copied into a
//    shared stage, 0.0 where the element lies outside M, N or K ("Zero-filled
//    boundary tiles"); every shared slot is written, so all threads reach the
//    same barriers;
//  * padded shared rows — A rows are padded by the pages' bank rule counted
//    in 16-byte slots (section "Choosing padding instead of hard-coding it");
//    B rows are read as a broadcast and get no padding, as the rule says
//    (section "Why shared-memory banks matter", last paragraphs);
//  * K pipeline — STAGES shared stages filled by cp.async with zero fill,
//    one barrier per K tile (Part 18 "What ping-pong changes about
//    synchronization"; skills page step 7: commit, wait_group, then
//    __syncthreads), with STAGES-1 tiles in flight while one is computed;
//  * unrolled register-tile micro-kernel — each thread keeps a TM x TN block
//    of C in registers and, for every k of the fixed-size BK loop (fully
//    unrolled, Part 18 "Unrolling the inner reduction loop"), reads a float4
//    of A per row and float4s of B and issues TM*TN FMAs; the packed form
//    issues them as fma.rn.f32x2 pairs;
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

template <int BM_, int BN_, int BK_, int WM_, int WN_, int TM_, int TN_,
          int STAGES_, int MINB_>
struct FfmaTile {
  static constexpr int BM = BM_, BN = BN_, BK = BK_;
  static constexpr int WM = WM_, WN = WN_, TM = TM_, TN = TN_;
  static constexpr int STAGES = STAGES_, MIN_BLOCKS = MINB_;
  static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
  static constexpr int THREADS = WARPS_M * WARPS_N * 32;
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
  // the rule gives no padding.
  static constexpr SmemLayout b_layout(bool pad) {
    return SmemLayout{BK, BN, pad ? vector_row_padding_rule(BN, 1) : 0, STAGES};
  }
  static constexpr int smem_bytes(bool pad) {
    return a_layout(pad).nbytes() + b_layout(pad).nbytes();
  }
};

// ---------------------------------------------------------------------------
// Global -> shared staging of one K tile (A: BM x BK, B: BK x BN).
// VEC: 16-byte chunks (needs K % 4 == 0, N % 4 == 0 and 16-byte aligned A, B);
// otherwise 4-byte elements.  Out-of-bounds chunks are zero-filled.
template <class T, bool VEC>
struct Stager;

template <class T>
struct Stager<T, true> {
  static constexpr int A_CHUNKS_ROW = T::BK / 4;
  static constexpr int B_CHUNKS_ROW = T::BN / 4;
  static_assert(T::THREADS % A_CHUNKS_ROW == 0 && T::THREADS % B_CHUNKS_ROW == 0, "");
  static constexpr int A_ROWS_STEP = T::THREADS / A_CHUNKS_ROW;
  static constexpr int B_ROWS_STEP = T::THREADS / B_CHUNKS_ROW;
  static constexpr int A_ITERS = T::BM / A_ROWS_STEP;
  static constexpr int B_ITERS = T::BK / B_ROWS_STEP;
  static_assert(A_ITERS * A_ROWS_STEP == T::BM && B_ITERS * B_ROWS_STEP == T::BK, "");

  const float* a_src;  // A[m0 + a_row, a_col]
  const float* b_src;  // B[b_row, n0 + b_col]
  const float* A;
  const float* B;
  int64_t a_row_step, b_row_step;  // elements between rows a thread copies
  int a_row, a_col, b_row, b_col;
  int M, N, K;
  uint32_t a_rows_ok;  // bit t: row t of this thread's A chunks is inside M
  bool b_col_ok;

  __device__ Stager(const float* A_, const float* B_, int M_, int N_, int K_, int m0, int n0,
                    int tid)
      : A(A_), B(B_), M(M_), N(N_), K(K_) {
    a_row = tid / A_CHUNKS_ROW;
    a_col = (tid % A_CHUNKS_ROW) * 4;
    b_row = tid / B_CHUNKS_ROW;
    b_col = (tid % B_CHUNKS_ROW) * 4;
    a_row_step = static_cast<int64_t>(A_ROWS_STEP) * K;
    b_row_step = static_cast<int64_t>(B_ROWS_STEP) * N;
    a_src = A + static_cast<int64_t>(m0 + a_row) * K + a_col;
    b_src = B + static_cast<int64_t>(b_row) * N + n0 + b_col;
    a_rows_ok = 0;
#pragma unroll
    for (int t = 0; t < A_ITERS; ++t)
      if (m0 + a_row + t * A_ROWS_STEP < M) a_rows_ok |= 1u << t;
    b_col_ok = n0 + b_col < N;
  }

  template <class LA, class LB>
  __device__ __forceinline__ void load(float* As, float* Bs, const LA& la, const LB& lb,
                                       int stage, int kt) const {
    const int k0 = kt * T::BK;
    const bool a_k_ok = k0 + a_col < K;
#pragma unroll
    for (int t = 0; t < A_ITERS; ++t) {
      const bool ok = a_k_ok && (a_rows_ok >> t & 1u);
      const float* src = ok ? a_src + t * a_row_step + k0 : A;
      cp_async_16(smem_u32(As + la.offset(stage, a_row + t * A_ROWS_STEP, a_col)), src,
                  ok ? 16u : 0u);
    }
#pragma unroll
    for (int t = 0; t < B_ITERS; ++t) {
      const int kr = k0 + b_row + t * B_ROWS_STEP;
      const bool ok = b_col_ok && kr < K;
      const float* src = ok ? b_src + static_cast<int64_t>(k0) * N + t * b_row_step : B;
      cp_async_16(smem_u32(Bs + lb.offset(stage, b_row + t * B_ROWS_STEP, b_col)), src,
                  ok ? 16u : 0u);
    }
  }
};

template <class T>
struct Stager<T, false> {
  static_assert(T::THREADS % T::BK == 0 && T::THREADS % T::BN == 0, "");
  static constexpr int A_ROWS_STEP = T::THREADS / T::BK;
  static constexpr int B_ROWS_STEP = T::THREADS / T::BN;
  static constexpr int A_ITERS = T::BM / A_ROWS_STEP;
  static constexpr int B_ITERS = T::BK / B_ROWS_STEP;

  const float* a_src;
  const float* b_src;
  const float* A;
  const float* B;
  int64_t a_row_step, b_row_step;
  int a_row, a_col, b_row, b_col;
  int M, N, K;
  uint32_t a_rows_ok;
  bool b_col_ok;

  __device__ Stager(const float* A_, const float* B_, int M_, int N_, int K_, int m0, int n0,
                    int tid)
      : A(A_), B(B_), M(M_), N(N_), K(K_) {
    a_row = tid / T::BK;
    a_col = tid % T::BK;
    b_row = tid / T::BN;
    b_col = tid % T::BN;
    a_row_step = static_cast<int64_t>(A_ROWS_STEP) * K;
    b_row_step = static_cast<int64_t>(B_ROWS_STEP) * N;
    a_src = A + static_cast<int64_t>(m0 + a_row) * K + a_col;
    b_src = B + static_cast<int64_t>(b_row) * N + n0 + b_col;
    a_rows_ok = 0;
    static_assert(A_ITERS <= 32, "");
#pragma unroll
    for (int t = 0; t < A_ITERS; ++t)
      if (m0 + a_row + t * A_ROWS_STEP < M) a_rows_ok |= 1u << t;
    b_col_ok = n0 + b_col < N;
  }

  template <class LA, class LB>
  __device__ __forceinline__ void load(float* As, float* Bs, const LA& la, const LB& lb,
                                       int stage, int kt) const {
    const int k0 = kt * T::BK;
    const bool a_k_ok = k0 + a_col < K;
#pragma unroll
    for (int t = 0; t < A_ITERS; ++t) {
      const bool ok = a_k_ok && (a_rows_ok >> t & 1u);
      const float* src = ok ? a_src + t * a_row_step + k0 : A;
      cp_async_4(smem_u32(As + la.offset(stage, a_row + t * A_ROWS_STEP, a_col)), src,
                 ok ? 4u : 0u);
    }
#pragma unroll
    for (int t = 0; t < B_ITERS; ++t) {
      const int kr = k0 + b_row + t * B_ROWS_STEP;
      const bool ok = b_col_ok && kr < K;
      const float* src = ok ? b_src + static_cast<int64_t>(k0) * N + t * b_row_step : B;
      cp_async_4(smem_u32(Bs + lb.offset(stage, b_row + t * B_ROWS_STEP, b_col)), src,
                 ok ? 4u : 0u);
    }
  }
};

__device__ __forceinline__ float pick(const float4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// ---------------------------------------------------------------------------
template <class T, bool VEC, bool PAD, bool PACKED>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
    sgemm_ffma_kernel(GemmArgs args) {
  constexpr SmemLayout LA = T::a_layout(PAD);
  constexpr SmemLayout LB = T::b_layout(PAD);
  extern __shared__ float4 smem_f4[];
  float* As = reinterpret_cast<float*>(smem_f4);
  float* Bs = As + LA.size();

  const int M = args.M, N = args.N, K = args.K;
  const int tid = threadIdx.x;

  // Work unit: a whole tile, or one K slice of a tile of the split tail,
  // whose fp32 partial goes to the workspace instead of C.
  const int ktiles_all = (K + T::BK - 1) / T::BK;
  int tile = blockIdx.x, slice = 0, kt_begin = 0, kt_end = ktiles_all;
  const bool partial = static_cast<int>(blockIdx.x) >= args.full_tiles;
  if (partial) {
    const int v = blockIdx.x - args.full_tiles;
    tile = args.full_tiles + v / args.split;
    slice = v % args.split;
    kt_begin = min(ktiles_all, slice * args.kt_per_slice);
    kt_end = min(ktiles_all, kt_begin + args.kt_per_slice);
  }
  const int ktiles = kt_end - kt_begin;
  int tm, tn;
  grouped_tile(tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
  const int m0 = tm * T::BM, n0 = tn * T::BN;

  const Stager<T, VEC> stager(args.A, args.B, M, N, K, m0, n0, tid);

  // Prologue: STAGES-1 tiles in flight.  One commit group per tile (empty
  // groups keep the count uniform when K has fewer tiles).
#pragma unroll
  for (int s = 0; s < T::STAGES - 1; ++s) {
    if (s < ktiles) stager.load(As, Bs, LA, LB, s, kt_begin + s);
    cp_async_commit();
  }

  const int warp = tid / 32, lane = tid % 32;
  const int wm = warp / T::WARPS_N, wn = warp % T::WARPS_N;
  const int lm = lane % T::LM, ln = lane / T::LM;
  // Thread (lm, ln) of warp (wm, wn) owns rows wm*WM + i*LM + lm (i < TM)
  // and columns wn*WN + g*LN*4 + ln*4 + c (g < TN/4, c < 4).
  const int a_off = LA.offset(0, wm * T::WM + lm, 0);
  const int b_off = LB.offset(0, 0, wn * T::WN + ln * 4);

  float2 acc[T::TM][T::TN / 2];
#pragma unroll
  for (int i = 0; i < T::TM; ++i)
#pragma unroll
    for (int j = 0; j < T::TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);

  int stage = 0;
  int load_stage = T::STAGES - 1;
  for (int kt = 0; kt < ktiles; ++kt) {
    // Tile kt has landed for this thread; the barrier makes every thread's
    // copies visible and guarantees that the stage refilled below (read in
    // iteration kt-1) is no longer being read.
    cp_async_wait<T::STAGES - 2>();
    __syncthreads();
    if (kt + T::STAGES - 1 < ktiles)
      stager.load(As, Bs, LA, LB, load_stage, kt_begin + kt + T::STAGES - 1);
    cp_async_commit();

    const float* a_ptr = As + stage * LA.stage_size() + a_off;
    const float* b_ptr = Bs + stage * LB.stage_size() + b_off;
#pragma unroll
    for (int k4 = 0; k4 < T::BK / 4; ++k4) {
      float4 a[T::TM];
#pragma unroll
      for (int i = 0; i < T::TM; ++i)
        a[i] = *reinterpret_cast<const float4*>(a_ptr + i * T::LM * LA.row_stride() + k4 * 4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float4 b[T::TN / 4];
#pragma unroll
        for (int g = 0; g < T::TN / 4; ++g)
          b[g] = *reinterpret_cast<const float4*>(b_ptr + (k4 * 4 + kk) * LB.row_stride() +
                                                  g * T::LN * 4);
#pragma unroll
        for (int i = 0; i < T::TM; ++i) {
          const float av = pick(a[i], kk);
#pragma unroll
          for (int g = 0; g < T::TN / 4; ++g) {
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
    stage = stage + 1 == T::STAGES ? 0 : stage + 1;
    load_stage = load_stage + 1 == T::STAGES ? 0 : load_stage + 1;
  }

  if (partial) {
    // The slice's partial tile, dense BM x BN (rows and columns past M or N
    // hold zeros from the zero-filled staging and are never read back).
    float* P = args.partial +
               (static_cast<int64_t>(tile - args.full_tiles) * args.split + slice) *
                   (T::BM * T::BN);
#pragma unroll
    for (int i = 0; i < T::TM; ++i) {
      const int r = wm * T::WM + i * T::LM + lm;
#pragma unroll
      for (int g = 0; g < T::TN / 4; ++g) {
        const int c = wn * T::WN + g * T::LN * 4 + ln * 4;
        *reinterpret_cast<float4*>(P + r * T::BN + c) =
            make_float4(acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x,
                        acc[i][2 * g + 1].y);
      }
    }
    return;
  }

  // Masked epilogue: C[row, col] for row < M, col < N.
  float* C = args.C;
#pragma unroll
  for (int i = 0; i < T::TM; ++i) {
    const int row = m0 + wm * T::WM + i * T::LM + lm;
    if (row >= M) continue;
    float* c_row = C + static_cast<int64_t>(row) * N;
#pragma unroll
    for (int g = 0; g < T::TN / 4; ++g) {
      const int col = n0 + wn * T::WN + g * T::LN * 4 + ln * 4;
      const float4 v = make_float4(acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x,
                                   acc[i][2 * g + 1].y);
      if constexpr (VEC) {
        // N % 4 == 0, so a float4 group is either wholly inside or outside.
        if (col < N) *reinterpret_cast<float4*>(c_row + col) = v;
      } else {
        if (col + 0 < N) c_row[col + 0] = v.x;
        if (col + 1 < N) c_row[col + 1] = v.y;
        if (col + 2 < N) c_row[col + 2] = v.z;
        if (col + 3 < N) c_row[col + 3] = v.w;
      }
    }
  }
}

template <class T, bool PACKED, bool WITH_UNPADDED>
FfmaEntry make_entry() {
  FfmaEntry e{};
  e.bm = T::BM;
  e.bn = T::BN;
  e.bk = T::BK;
  e.stages = T::STAGES;
  e.threads = T::THREADS;
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
  e.kern[1][1] = reinterpret_cast<const void*>(&sgemm_ffma_kernel<T, true, true, PACKED>);
  e.kern[0][1] = reinterpret_cast<const void*>(&sgemm_ffma_kernel<T, false, true, PACKED>);
  if (WITH_UNPADDED) {
    e.kern[1][0] = reinterpret_cast<const void*>(&sgemm_ffma_kernel<T, true, false, PACKED>);
    e.kern[0][0] = reinterpret_cast<const void*>(&sgemm_ffma_kernel<T, false, false, PACKED>);
  }
  return e;
}

}  // namespace mt
