// Registry of the FFMA tile configurations built into the library.  The
// kernels themselves are in sgemm_ffma.cuh; each ffma_tiles_*.cu instantiates
// a few configurations (separate translation units build in parallel).
#include "kernels.h"

namespace mt {

int ffma_entries_128(FfmaEntry* out);
int ffma_entries_other(FfmaEntry* out);

const FfmaEntry* ffma_entries(int* count) {
  static FfmaEntry entries[32];
  static const int n = [] {
    int k = ffma_entries_128(entries);
    k += ffma_entries_other(entries + k);
    return k;
  }();
  *count = n;
  return entries;
}

}  // namespace mt
