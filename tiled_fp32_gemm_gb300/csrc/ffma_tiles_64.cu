// FFMA configurations for grids too small to fill the GPU with 128 x 128
// tiles (see sgemm_ffma.cuh).
#include "sgemm_ffma.cuh"

namespace mt {

// 64 x 128, BK 32, 2 stages: 4 warps of 32 x 64, 8 x 8 per thread, 3 CTAs
// per SM (at most 168 registers a thread).
using Tile64x128 = FfmaTile<64, 128, 32, 32, 64, 8, 8, 2, 3>;
// 64 x 64: 4 warps of 32 x 32, 8 x 4 per thread, 4 CTAs per SM.
using Tile64x64 = FfmaTile<64, 64, 32, 32, 32, 8, 4, 3, 4>;
// 64 x 128 with two K groups of 4 warps (8 warps, 1 CTA per SM), BK 32, 3
// stages: each group takes 16 of the 32 k steps of every staged tile.
using Tile64x128ks2 = FfmaTile<64, 128, 32, 32, 64, 8, 8, 3, 1, 2>;

int ffma_entries_64(FfmaEntry* out) {
  out[0] = make_entry<Tile64x128, true, false, false, true>();
  out[1] = make_entry<Tile64x64, true, false, true, true>();
  out[2] = make_entry<Tile64x128ks2, true, false, false, true>();
  return 3;
}

}  // namespace mt
