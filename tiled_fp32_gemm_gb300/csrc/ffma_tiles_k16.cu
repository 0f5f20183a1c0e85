// The automatic FFMA configuration for large grids with A staged K-major
// (see sgemm_ffma.cuh): 128 x 128 tiles with a K depth of 16 and 4 stages, 4
// warps of 64 x 64, 8 x 16 per thread, 2 CTAs per SM.  On GB300 it measured
// 0.5 % faster than K depth 32 with 3 stages at 4096^3 and 8192^3 (66.8
// against 66.4 and 70.8 against 70.4 TFLOP/s) with half the shared memory.
// Only the K-major kernels are built: row-major A tiles use the K depth 32
// tile.
#include "sgemm_ffma.cuh"

namespace mt {

using Tile128x128k16km = FfmaTile<128, 128, 16, 64, 64, 8, 16, 4, 2>;

int ffma_entries_k16(FfmaEntry* out) {
  out[0] = make_entry<Tile128x128k16km, true, false, false, true>();
  return 1;
}

}  // namespace mt
