// Alternative FFMA configurations, selectable by their tile parameters and
// kept for measurement (see sgemm_ffma.cuh); the automatic choice does not
// use them.
#include "sgemm_ffma.cuh"

namespace mt {

// 8 warps of 32 x 64, 8 x 8 per thread, 3 stages, 2 CTAs per SM.
using Tile128x128 = FfmaTile<128, 128, 32, 32, 64, 8, 8, 3, 2>;
// The same with 4 stages (1 CTA per SM).
using Tile128x128s4 = FfmaTile<128, 128, 32, 32, 64, 8, 8, 4, 1>;
// 8 warps of 64 x 32 (8 lanes along M), 8 x 8 per thread.
using Tile128x128w64x32 = FfmaTile<128, 128, 32, 64, 32, 8, 8, 3, 2>;
// K depth 16, 4 stages.
using Tile128x128k16 = FfmaTile<128, 128, 16, 32, 64, 8, 8, 4, 2>;
// 8 warps of 64 x 64, 8 x 16 per thread, 1 CTA per SM.
using Tile128x256 = FfmaTile<128, 256, 32, 64, 64, 8, 16, 3, 1>;
using Tile256x128 = FfmaTile<256, 128, 32, 64, 64, 8, 16, 3, 1>;

int ffma_entries_alt(FfmaEntry* out) {
  int n = 0;
  // Table order matters: the first entry that matches the caller's
  // choices wins, so each tile's preferred warp layout comes first.
  out[n++] = make_entry<Tile128x128, true, true>();
  out[n++] = make_entry<Tile128x128, false, false>();
  out[n++] = make_entry<Tile128x128s4, true, false>();
  out[n++] = make_entry<Tile128x128w64x32, true, false>();
  out[n++] = make_entry<Tile128x128k16, true, false>();
  out[n++] = make_entry<Tile128x256, true, false>();
  out[n++] = make_entry<Tile256x128, true, false>();
  return n;
}

}  // namespace mt
