// Registry of the FFMA tile configurations built into the library.  The
// kernels themselves are in sgemm_ffma.cuh; each ffma_tiles_*.cu instantiates
// a few configurations (separate translation units build in parallel).
#include "device_util.cuh"
#include "kernels.h"

namespace mt {

// One CTA per split tile: C[tile] = sum over slices s = 0, 1, ... of the
// slice partials, added in that order.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(GemmArgs a, int bm, int bn,
                                                           int vec_c) {
  int tm, tn;
  grouped_tile(a.full_tiles + blockIdx.x, a.tiles_m, a.tiles_n, a.group_m, tm, tn);
  const int block = bm * bn;
  const float4* P = reinterpret_cast<const float4*>(
      a.partial + static_cast<int64_t>(blockIdx.x) * a.split * block);
  for (int e4 = threadIdx.x; e4 < block / 4; e4 += blockDim.x) {
    const int r = (e4 * 4) / bn, c = (e4 * 4) % bn;
    const int row = tm * bm + r, col = tn * bn + c;
    if (row >= a.M || col >= a.N) continue;
    float4 s = P[e4];
    for (int sl = 1; sl < a.split; ++sl) {
      const float4 v = P[static_cast<int64_t>(sl) * (block / 4) + e4];
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    float* c_row = a.C + static_cast<int64_t>(row) * a.N;
    if (vec_c) {
      *reinterpret_cast<float4*>(c_row + col) = s;
    } else {
      c_row[col] = s.x;
      if (col + 1 < a.N) c_row[col + 1] = s.y;
      if (col + 2 < a.N) c_row[col + 2] = s.z;
      if (col + 3 < a.N) c_row[col + 3] = s.w;
    }
  }
}

cudaError_t launch_splitk_reduce(const GemmArgs& a, int bm, int bn, bool vec_c,
                                 cudaStream_t stream) {
  const int tail = a.tiles_m * a.tiles_n - a.full_tiles;
  if (tail <= 0) return cudaSuccess;
  splitk_reduce_kernel<<<tail, 256, 0, stream>>>(a, bm, bn, vec_c ? 1 : 0);
  return cudaGetLastError();
}

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
