// FFMA configurations with tiles other than 128 x 128 (see sgemm_ffma.cuh).
#include "sgemm_ffma.cuh"

namespace mt {

// 8 warps of 64 x 64, 8 x 16 per thread, 1 CTA per SM.
using Tile128x256 = FfmaTile<128, 256, 32, 64, 64, 8, 16, 3, 1>;
using Tile256x128 = FfmaTile<256, 128, 32, 64, 64, 8, 16, 3, 1>;
// 4 warps of 32 x 32, 8 x 4 per thread, 4 CTAs per SM (small grids).
using Tile64x64 = FfmaTile<64, 64, 32, 32, 32, 8, 4, 3, 4>;

int ffma_entries_other(FfmaEntry* out) {
  int n = 0;
  out[n++] = make_entry<Tile128x256, true, false>();
  out[n++] = make_entry<Tile256x128, true, false>();
  out[n++] = make_entry<Tile64x64, true, false, true>();
  return n;
}

}  // namespace mt
