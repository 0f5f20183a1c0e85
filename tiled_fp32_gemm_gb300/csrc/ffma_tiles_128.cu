// The default FFMA configuration (see sgemm_ffma.cuh): 128 x 128 tiles, 4
// warps of 64 x 64, 8 x 16 per thread, 3 stages, 2 CTAs per SM, with every
// staging form (padded and unpadded row-major A, transposed operands, and
// A staged K-major).
#include "sgemm_ffma.cuh"

namespace mt {

using Tile128x128w64 = FfmaTile<128, 128, 32, 64, 64, 8, 16, 3, 2>;

int ffma_entries_128(FfmaEntry* out) {
  out[0] = make_entry<Tile128x128w64, true, true, true, true>();
  return 1;
}

}  // namespace mt
