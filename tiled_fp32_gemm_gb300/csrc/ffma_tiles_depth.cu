// The automatic large-grid FFMA tile (128 x 128, K depth 16, 4 warps of
// 64 x 64, 8 x 16 per thread, 2 CTAs per SM) with shallower K pipelines, to
// measure what the pipeline buys (see sgemm_ffma.cuh): one stage (no
// double buffering, two barriers per K tile), two stages (one tile copied
// while one is computed) and three.  Selected by their stage count; the
// automatic choice keeps the 4-stage tile.  Every depth runs the same FMA
// chain, so the results are bit-identical.
#include "sgemm_ffma.cuh"

namespace mt {

using Tile128x128k16s1 = FfmaTile<128, 128, 16, 64, 64, 8, 16, 1, 2>;
using Tile128x128k16s2 = FfmaTile<128, 128, 16, 64, 64, 8, 16, 2, 2>;
using Tile128x128k16s3 = FfmaTile<128, 128, 16, 64, 64, 8, 16, 3, 2>;

int ffma_entries_depth(FfmaEntry* out) {
  out[0] = make_entry<Tile128x128k16s1, true, false, false, true>();
  out[1] = make_entry<Tile128x128k16s2, true, false, false, true>();
  out[2] = make_entry<Tile128x128k16s3, true, false, false, true>();
  return 3;
}

}  // namespace mt
