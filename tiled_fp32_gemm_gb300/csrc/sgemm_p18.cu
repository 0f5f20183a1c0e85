// One-warp tiled GEMM restating the kernel of "My Triton From Scratch,
// Part 18: Shared Memory Optimization" — a deliberately plain kernel for
// parity and for measuring the bank rule, not for speed.
//
// Tile BM=4, BN=8, BK=16 with one warp (the one-warp layout the page
// describes, section "What Version 18 does not do"); each thread owns one
// output (tile_i, tile_j).  Per K tile:
//   * the stage is (k_base / BK) & 1 (section "One stage versus two stages");
//   * both tiles are copied cooperatively, thread t taking elements t, t+32,
//     ... ("Part 14: Shared Memory Tiles", section "Cooperative copy
//     mapping"), with 0.0 where the element lies outside M, N or K
//     ("Zero-filled boundary tiles"), synchronously;
//   * one __syncthreads, then the fixed-size dot loop, unrolled (Part 18,
//     "Unrolling the inner reduction loop"); the trailing barrier is not
//     needed because the next tile goes to the other stage (section "What
//     ping-pong changes about synchronization").
// A rows are read by four output rows at once at the same k, so the A tile
// gets the rule's padding (16 columns, 4 rows -> one word, stride 17); B is
// read as a broadcast and is not padded (section "Why shared-memory banks
// matter").  pad=false keeps stride 16 to measure the conflict it removes.
// Leading dimensions, transposed storage and alpha/beta only change how the
// copies index A and B and how the result is written.
#include <cuda_runtime.h>

#include "kernels.h"
#include "smem_layout.cuh"

namespace mt {

namespace {
constexpr int P18_BM = 4, P18_BN = 8, P18_BK = 16, P18_THREADS = 32;

constexpr SmemLayout p18_a_layout(bool pad) {
  // Four output rows (tile_i = 0..3) read A at the same dot_k.
  return SmemLayout{P18_BM, P18_BK, pad ? row_padding_rule(P18_BK, P18_BM) : 0, 2};
}
constexpr SmemLayout p18_b_layout() { return SmemLayout{P18_BK, P18_BN, 0, 2}; }
}  // namespace

template <bool PAD>
__global__ void __launch_bounds__(P18_THREADS) sgemm_p18_kernel(GemmArgs args) {
  constexpr SmemLayout LA = p18_a_layout(PAD);
  constexpr SmemLayout LB = p18_b_layout();
  __shared__ float dot_lhs[LA.size()];
  __shared__ float dot_rhs[LB.size()];

  const int M = args.M, N = args.N, K = args.K;
  const int tile = blockIdx.x;
  const int block_m = (tile / args.tiles_n) * P18_BM;
  const int block_n = (tile % args.tiles_n) * P18_BN;
  const int tid = threadIdx.x;
  const int tile_i = tid / P18_BN, tile_j = tid % P18_BN;

  float accumulator = 0.0f;
  for (int k_base = 0; k_base < K; k_base += P18_BK) {
    const int dot_stage = (k_base / P18_BK) & 1;
    for (int index = tid; index < P18_BM * P18_BK; index += P18_THREADS) {
      const int row = index / P18_BK, column = index % P18_BK;
      const int global_row = block_m + row, global_column = k_base + column;
      // op(A)[global_row][global_column], stored row-major or transposed.
      dot_lhs[LA.offset(dot_stage, row, column)] =
          global_row < M && global_column < K
              ? args.A[args.trans_a ? static_cast<int64_t>(global_column) * args.lda + global_row
                                    : static_cast<int64_t>(global_row) * args.lda + global_column]
              : 0.0f;
    }
    for (int index = tid; index < P18_BK * P18_BN; index += P18_THREADS) {
      const int row = index / P18_BN, column = index % P18_BN;
      const int global_row = k_base + row, global_column = block_n + column;
      dot_rhs[LB.offset(dot_stage, row, column)] =
          global_row < K && global_column < N
              ? args.B[args.trans_b ? static_cast<int64_t>(global_column) * args.ldb + global_row
                                    : static_cast<int64_t>(global_row) * args.ldb + global_column]
              : 0.0f;
    }
    __syncthreads();
    // One 4-byte shared load per operand and k, as the page's generated loop
    // reads them (volatile keeps the compiler from merging the A reads of a
    // row into wider loads, which would change the access pattern the
    // padding rule is about).
    const volatile float* lhs = dot_lhs;
    const volatile float* rhs = dot_rhs;
#pragma unroll
    for (int dot_k = 0; dot_k < P18_BK; ++dot_k)
      accumulator = fmaf(lhs[LA.offset(dot_stage, tile_i, dot_k)],
                         rhs[LB.offset(dot_stage, dot_k, tile_j)], accumulator);
  }
  const int out_row = block_m + tile_i, out_col = block_n + tile_j;
  if (out_row < M && out_col < N) {
    float* c = args.C + static_cast<int64_t>(out_row) * args.ldc + out_col;
    const float v = args.alpha * accumulator;
    *c = args.beta != 0.0f ? fmaf(args.beta, *c, v) : v;
  }
}

cudaError_t launch_p18(const GemmArgs& a, bool pad, cudaStream_t stream) {
  const int64_t grid = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  if (pad)
    sgemm_p18_kernel<true><<<static_cast<unsigned>(grid), P18_THREADS, 0, stream>>>(a);
  else
    sgemm_p18_kernel<false><<<static_cast<unsigned>(grid), P18_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

int p18_pad_a(bool pad) { return p18_a_layout(pad).row_padding; }
int p18_smem_bytes(bool pad) { return p18_a_layout(pad).nbytes() + p18_b_layout().nbytes(); }

}  // namespace mt
