// The 128 x 128 FFMA tile with a K depth of 32 and 3 stages (see
// sgemm_ffma.cuh): 4 warps of 64 x 64, 8 x 16 per thread, 2 CTAs per SM,
// with every staging form (padded and unpadded row-major A, transposed
// operands, and A staged K-major).  The automatic plans take it for
// row-major A tiles; with A staged K-major they take the K-depth-16,
// 4-stage tile of ffma_tiles_k16.cu.
#include "sgemm_ffma.cuh"

namespace mt {

using Tile128x128w64 = FfmaTile<128, 128, 32, 64, 64, 8, 16, 3, 2>;

int ffma_entries_128(FfmaEntry* out) {
  out[0] = make_entry<Tile128x128w64, true, true, true, true>();
  return 1;
}

}  // namespace mt
