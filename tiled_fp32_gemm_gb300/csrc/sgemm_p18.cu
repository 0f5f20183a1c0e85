// One-warp tiled GEMM restating the kernel of "My Triton From Scratch,
// Part 18: Shared Memory Optimization" — a deliberately plain kernel for
// parity and for measuring the bank rule, not for speed.
//
// Tile BM=4, BN=8, BK=16 with one warp (the one-warp layout the page
// describes, section "What Version 18 does not do"); each lane owns one
// output of the 4 x 8 tile.  Per K tile:
//   * K tiles alternate between two stages (section "One stage versus two
//     stages");
//   * both tiles are copied cooperatively, thread t taking elements t, t+32,
//     ... ("Part 14: Shared Memory Tiles", section "Cooperative copy
//     mapping"), with 0.0 where the element lies outside M, N or K
//     ("Zero-filled boundary tiles"), synchronously;
//   * one __syncthreads, then the fixed-size dot loop, unrolled (Part 18,
//     "Unrolling the inner reduction loop"); the trailing barrier is not
//     needed because the next tile goes to the other stage (section "What
//     ping-pong changes about synchronization").
// STAGES = 1 is the form the page falls back to when its double-buffer
// matcher declines (section "Why a conservative matcher matters"): every K
// tile overwrites the same storage, so a second barrier after the dot loop
// protects it from the next tile's copies.  Both forms run the same FMA
// chain, so their results are bit-identical.
// A rows are read by four output rows at once at the same k, so the A tile
// gets the rule's padding (16 columns, 4 rows -> one word, stride 17); B is
// read as a broadcast and is not padded (section "Why shared-memory banks
// matter").  pad=false keeps stride 16 to measure the conflict it removes.
// Leading dimensions, transposed storage and alpha/beta only change how the
// copies index A and B and how the result is written.
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kernels.h"
#include "smem_layout.cuh"

namespace mt {

namespace {
constexpr int P18_BM = 4, P18_BN = 8, P18_BK = 16, P18_THREADS = 32;

constexpr SmemLayout p18_a_layout(bool pad, int stages) {
  // The four output rows of a tile read A at the same k at once.
  return SmemLayout{P18_BM, P18_BK, pad ? row_padding_rule(P18_BK, P18_BM) : 0, stages};
}
constexpr SmemLayout p18_b_layout(int stages) { return SmemLayout{P18_BK, P18_BN, 0, stages}; }
}  // namespace

// op(A)[i][k] or op(B)[k][j] from its storage, 0.0 outside rows x cols
// (and, in a checked build, outside the `extent` elements of the storage).
__device__ __forceinline__ float fetch_operand(const float* base, int64_t ld, int trans, int i,
                                               int j, int rows, int cols, int64_t extent,
                                               BoundsRecord* rec) {
  if (i >= rows || j >= cols) return 0.0f;
  const int64_t o = trans ? static_cast<int64_t>(j) * ld + i : static_cast<int64_t>(i) * ld + j;
  return bounds_ok(rec, SITE_P18, o, 1, extent) ? base[o] : 0.0f;
}

template <bool PAD, int STAGES>
__global__ void __launch_bounds__(P18_THREADS) sgemm_p18_kernel(GemmArgs args) {
  static_assert(STAGES == 1 || STAGES == 2, "one stage or a ping-pong pair");
  constexpr SmemLayout LA = p18_a_layout(PAD, STAGES);
  constexpr SmemLayout LB = p18_b_layout(STAGES);
  // Both staged operands: A's stages, then B's.
  __shared__ float staged[LA.size() + LB.size()];
  float* a_tiles = staged;
  float* b_tiles = staged + LA.size();

  const int lane = threadIdx.x;
  const int m0 = (blockIdx.x / args.tiles_n) * P18_BM;
  const int n0 = (blockIdx.x % args.tiles_n) * P18_BN;
  // This lane's output: row r, column c of the 4 x 8 tile.
  const int r = lane / P18_BN, c = lane % P18_BN;
  // Elements of the A tile (64) and of the B tile (128) this lane copies:
  // lane, lane + 32, ... in row-major order of the tile.
  constexpr int A_PER_LANE = P18_BM * P18_BK / P18_THREADS;
  constexpr int B_PER_LANE = P18_BK * P18_BN / P18_THREADS;

  const int k_tiles = (args.K + P18_BK - 1) / P18_BK;
  float acc = 0.0f;
  for (int kt = 0; kt < k_tiles; ++kt) {
    const int buf = STAGES == 2 ? kt & 1 : 0;  // stage of this K tile: tiles alternate
    const int k0 = kt * P18_BK;
#pragma unroll
    for (int e = 0; e < A_PER_LANE; ++e) {
      const int slot = e * P18_THREADS + lane;
      const int ar = slot / P18_BK, ak = slot % P18_BK;
      const float v = fetch_operand(args.A, args.lda, args.trans_a, m0 + ar, k0 + ak, args.M,
                                    args.K, args.a_extent, args.bounds);
      if (bounds_ok(args.bounds, SITE_P18, LA.offset(buf, ar, ak), 1, LA.size()))
        a_tiles[LA.offset(buf, ar, ak)] = v;
    }
#pragma unroll
    for (int e = 0; e < B_PER_LANE; ++e) {
      const int slot = e * P18_THREADS + lane;
      const int bk = slot / P18_BN, bn = slot % P18_BN;
      const float v = fetch_operand(args.B, args.ldb, args.trans_b, k0 + bk, n0 + bn, args.K,
                                    args.N, args.b_extent, args.bounds);
      if (bounds_ok(args.bounds, SITE_P18, LB.offset(buf, bk, bn), 1, LB.size()))
        b_tiles[LB.offset(buf, bk, bn)] = v;
    }
    __syncthreads();
    // Scalar shared reads, one per operand and k (volatile keeps the
    // compiler from merging a row's A reads into wider loads, which would
    // change the access pattern the padding rule is about).
    const volatile float* av = a_tiles;
    const volatile float* bv = b_tiles;
#pragma unroll
    for (int kk = 0; kk < P18_BK; ++kk) {
      if (MT_BOUNDS_CHECK && (!bounds_ok(args.bounds, SITE_P18, LA.offset(buf, r, kk), 1,
                                         LA.size()) ||
                              !bounds_ok(args.bounds, SITE_P18, LB.offset(buf, kk, c), 1,
                                         LB.size())))
        continue;
      acc = fmaf(av[LA.offset(buf, r, kk)], bv[LB.offset(buf, kk, c)], acc);
    }
    if (STAGES == 1) __syncthreads();  // the next tile's copies overwrite this stage
  }
  const int row = m0 + r, col = n0 + c;
  if (row < args.M && col < args.N &&
      bounds_ok(args.bounds, SITE_P18, static_cast<int64_t>(row) * args.ldc + col, 1,
                args.c_extent) &&
      (!args.bias || bounds_ok(args.bounds, SITE_BIAS, col, 1, args.N))) {
    float* out = args.C + static_cast<int64_t>(row) * args.ldc + col;
    const float v = args.alpha * acc;
    float o = args.beta != 0.0f ? fmaf(args.beta, *out, v) : v;
    if (args.bias) o += args.bias[col];
    *out = o;
  }
}

cudaError_t launch_p18(const GemmArgs& a, bool pad, int stages, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(a.tiles_m) * a.tiles_n);
  if (stages == 1) {
    if (pad)
      sgemm_p18_kernel<true, 1><<<grid, P18_THREADS, 0, stream>>>(a);
    else
      sgemm_p18_kernel<false, 1><<<grid, P18_THREADS, 0, stream>>>(a);
  } else {
    if (pad)
      sgemm_p18_kernel<true, 2><<<grid, P18_THREADS, 0, stream>>>(a);
    else
      sgemm_p18_kernel<false, 2><<<grid, P18_THREADS, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

int p18_pad_a(bool pad) { return p18_a_layout(pad, 2).row_padding; }
int p18_smem_bytes(bool pad, int stages) {
  return p18_a_layout(pad, stages).nbytes() + p18_b_layout(stages).nbytes();
}

}  // namespace mt
