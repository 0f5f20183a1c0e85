// Registry of the FFMA tile configurations built into the library (the
// kernels themselves are in sgemm_ffma.cuh; each ffma_tiles_*.cu instantiates
// a few configurations, so the translation units build in parallel), and the
// helper kernels of the path: the K-slice reduce (shared by every variant's
// split tail), the C scaling of empty products, and the operand copy.
#include <algorithm>

#include "device_util.cuh"
#include "kernels.h"

namespace mt {

// C[row][col..col+3] = alpha * s + beta * C (+ bias), masked to M x N: the
// epilogue of the second-pass kernels that add partial tiles.
__device__ __forceinline__ void store_sum4(const GemmArgs& a, int row, int col, float4 s,
                                           int vec_c) {
  float* c_row = a.C + static_cast<int64_t>(row) * a.ldc;
  const float v[4] = {a.alpha * s.x, a.alpha * s.y, a.alpha * s.z, a.alpha * s.w};
  if (vec_c) {
    if (!bounds_ok(a.bounds, SITE_C_STORE, (c_row - a.C) + col, 4, a.c_extent) ||
        (a.bias && !bounds_ok(a.bounds, SITE_BIAS, col, 4, a.N)))
      return;
    float4* cp = reinterpret_cast<float4*>(c_row + col);
    float4 o = make_float4(v[0], v[1], v[2], v[3]);
    if (a.beta != 0.0f) {
      const float4 c0 = *cp;
      o = make_float4(fmaf(a.beta, c0.x, v[0]), fmaf(a.beta, c0.y, v[1]),
                      fmaf(a.beta, c0.z, v[2]), fmaf(a.beta, c0.w, v[3]));
    }
    if (a.bias) {
      o.x += a.bias[col];
      o.y += a.bias[col + 1];
      o.z += a.bias[col + 2];
      o.w += a.bias[col + 3];
    }
    *cp = o;
  } else {
    for (int e = 0; e < 4; ++e)
      if (col + e < a.N &&
          bounds_ok(a.bounds, SITE_C_STORE, (c_row - a.C) + col + e, 1, a.c_extent) &&
          (!a.bias || bounds_ok(a.bounds, SITE_BIAS, col + e, 1, a.N))) {
        float o = a.beta != 0.0f ? fmaf(a.beta, c_row[col + e], v[e]) : v[e];
        if (a.bias) o += a.bias[col + e];
        c_row[col + e] = o;
      }
  }
}

// C[tile] = alpha * (sum over slices s = 0, 1, ... of the slice partials,
// added in that order) + beta * C[tile] (+ bias[col]), masked to M x N.
// Each split tile is cut into `pieces` CTAs of up to 1024 float4 (4 per
// thread), so a small tail still spreads over the GPU.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(GemmArgs a, int bm, int bn,
                                                           int pieces, int vec_c) {
  // Launched as a programmatic dependent of the GEMM kernel before it on the
  // stream: wait until that kernel has finished and its partial tiles are
  // visible (a no-op when launched without the attribute).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x / pieces, piece = blockIdx.x % pieces;
  int tm, tn;
  grouped_tile(a.full_tiles + t, a.tiles_m, a.tiles_n, a.group_m, tm, tn);
  const int block4 = bm * bn / 4;
  const int per_piece = (block4 + pieces - 1) / pieces;
  const int e_begin = piece * per_piece;
  const int e_end = min(block4, e_begin + per_piece);
  const int64_t tile_off = static_cast<int64_t>(t) * a.split * block4;  // in float4s
  const float4* P = reinterpret_cast<const float4*>(a.partial) + tile_off;
  // A thread's (at most) four float4 of the piece are read slice by slice,
  // four independent loads at a time.
  float4 s[4];
  for (int sl = 0; sl < a.split; ++sl) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e4 = e_begin + threadIdx.x + q * 256;
      if (e4 >= e_end) continue;
      const int64_t e = static_cast<int64_t>(sl) * block4 + e4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (bounds_ok(a.bounds, SITE_PARTIAL, (tile_off + e) * 4, 4, a.partial_extent)) v = P[e];
      if (sl == 0) {
        s[q] = v;
      } else {
        s[q].x += v.x;
        s[q].y += v.y;
        s[q].z += v.z;
        s[q].w += v.w;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e4 = e_begin + threadIdx.x + q * 256;
    if (e4 >= e_end) continue;
    const int r = (e4 * 4) / bn, c = (e4 * 4) % bn;
    const int row = tm * bm + r, col = tn * bn + c;
    if (row < a.M && col < a.N) store_sum4(a, row, col, s[q], vec_c);
  }
}

// The stream-K fix-up (see launch_streamk_fixup): tile t of the stream-K
// tiles is cut into `pieces` CTAs like the split-K reduce.  The units whose
// runs overlap the tile's K tiles [t*ktiles, (t+1)*ktiles) are consecutive;
// their pieces are added in unit order, which is k order, so the result
// does not depend on scheduling.  The slots of those units are worked out
// once per CTA, up to 256 at a time, into shared memory.
__global__ void __launch_bounds__(256) streamk_fixup_kernel(GemmArgs a, int bm, int bn,
                                                           int pieces, int ktiles, int vec_c) {
  __shared__ long long slot_of[256];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x / pieces, piece = blockIdx.x % pieces;
  const int64_t first = static_cast<int64_t>(t) * ktiles, last = first + ktiles;
  const int c0 = streamk_unit_of(first, a.sk_iters, a.sk_ctas);
  const int c1 = streamk_unit_of(last - 1, a.sk_iters, a.sk_ctas);
  if (c0 == c1) return;  // one run covered the tile whole: already in C
  int tm, tn;
  grouped_tile(a.full_tiles + t, a.tiles_m, a.tiles_n, a.group_m, tm, tn);
  const int block4 = bm * bn / 4;
  const int per_piece = (block4 + pieces - 1) / pieces;
  const int e_begin = piece * per_piece;
  const int e_end = min(block4, e_begin + per_piece);
  const float4* P = reinterpret_cast<const float4*>(a.partial);
  // Each thread sums at most this many float4 of the piece.
  constexpr int kMaxPerThread = 4;
  float4 s[kMaxPerThread];
#pragma unroll
  for (int q = 0; q < kMaxPerThread; ++q) s[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = c0; base <= c1; base += 256) {
    const int n = min(256, c1 - base + 1);
    __syncthreads();  // the previous chunk's slots are no longer read
    if (static_cast<int>(threadIdx.x) < n) {
      const int u = base + threadIdx.x;
      const int64_t b = static_cast<int64_t>(u) * a.sk_iters / a.sk_ctas;
      const int64_t e = static_cast<int64_t>(u + 1) * a.sk_iters / a.sk_ctas;
      // An empty run has no piece; the tile is the first of u's run unless
      // the run began before it.
      slot_of[threadIdx.x] = e <= b ? -1 : 2 * static_cast<int64_t>(u) + (b < first ? 1 : 0);
    }
    __syncthreads();
    // Piece by piece in k order, the thread's float4 four independent loads
    // at a time.  The sum starts from zero: adding the first piece to +0.0
    // leaves it unchanged, except that -0.0 becomes +0.0, as it does in any
    // fp32 sum.
    for (int j = 0; j < n; ++j) {
      const long long slot = slot_of[j];
      if (slot < 0) continue;
#pragma unroll
      for (int q = 0; q < kMaxPerThread; ++q) {
        const int e4 = e_begin + threadIdx.x + q * 256;
        if (e4 >= e_end) continue;
        const int64_t at = slot * block4 + e4;
        if (!bounds_ok(a.bounds, SITE_PARTIAL, at * 4, 4, a.partial_extent)) continue;
        const float4 v = P[at];
        s[q].x += v.x;
        s[q].y += v.y;
        s[q].z += v.z;
        s[q].w += v.w;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kMaxPerThread; ++q) {
    const int e4 = e_begin + threadIdx.x + q * 256;
    if (e4 >= e_end) continue;
    const int r = (e4 * 4) / bn, c = (e4 * 4) % bn;
    const int row = tm * bm + r, col = tn * bn + c;
    if (row < a.M && col < a.N) store_sum4(a, row, col, s[q], vec_c);
  }
}

cudaError_t launch_splitk_reduce(const GemmArgs& a, int bm, int bn, bool vec_c,
                                 cudaStream_t stream) {
  const int tail = a.tiles_m * a.tiles_n - a.full_tiles;
  if (tail <= 0) return cudaSuccess;
  // Pieces of at most 1024 float4: four per thread of 256.
  const int pieces = std::max(1, (bm * bn / 4 + 1023) / 1024);
  GemmArgs r = a;
  // Callers that did not state the partial buffer's extent (the tensor-core
  // paths) have exactly one dense bm x bn tile per slice of each split tile.
  if (r.partial_extent == 0)
    r.partial_extent = static_cast<int64_t>(tail) * a.split * bm * bn;
  // Programmatic stream serialization: the reduce grid is launched while the
  // GEMM kernel finishes and waits for it inside (griddepcontrol.wait), so
  // its launch latency overlaps the GEMM's last CTAs.  Measured on GB300:
  // bf16 4096^3 98.0 -> 94.9 us, FFMA 512 x 512 x 4096 65.2 -> 62.1 us,
  // 3xTF32 4096^3 459 -> 455 us; results bit-identical.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(tail * pieces));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int vc = vec_c ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, r, bm, bn, pieces, vc);
}

cudaError_t launch_streamk_fixup(const GemmArgs& a, int bm, int bn, int ktiles, bool vec_c,
                                 cudaStream_t stream) {
  if (a.sk_ctas <= 0 || a.sk_iters <= 0 || ktiles <= 0) return cudaSuccess;
  const int64_t tiles = a.sk_iters / ktiles;
  // Pieces of at most 1024 float4: four per thread of 256.
  const int pieces = std::max(1, (bm * bn / 4 + 1023) / 1024);
  if (tiles <= 0 || tiles * pieces > INT32_MAX) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * pieces));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int vc = vec_c ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, streamk_fixup_kernel, a, bm, bn, pieces, ktiles, vc);
}

cudaError_t launch_second_pass(const GemmArgs& a, float* partial, int bm, int bn, int ktiles,
                               bool vec_c, cudaStream_t stream) {
  GemmArgs r = a;
  r.partial = partial;
  if (a.sk_ctas > 0) {
    // Two dense bm x bn slots per stream-K unit (callers that stated a larger
    // extent keep theirs).
    const int64_t slots = 2 * static_cast<int64_t>(a.sk_ctas) * bm * bn;
    if (r.partial_extent < slots) r.partial_extent = slots;
    return launch_streamk_fixup(r, bm, bn, ktiles, vec_c, stream);
  }
  if (a.split > 1) return launch_splitk_reduce(r, bm, bn, vec_c, stream);
  return cudaSuccess;
}

// C = beta * C (+ bias[col]) on an M x N view (C not read when beta is 0).
__global__ void __launch_bounds__(256) scale_c_kernel(float* C, int M, int N, int64_t ldc,
                                                     float beta, const float* bias,
                                                     BoundsRecord* rec) {
  const int64_t total = static_cast<int64_t>(M) * N;
  const int64_t extent = view_extent(M, N, ldc);
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = e / N, j = e % N;
    if (!bounds_ok(rec, SITE_C_STORE, i * ldc + j, 1, extent) ||
        (bias && !bounds_ok(rec, SITE_BIAS, j, 1, N)))
      continue;
    float* c = C + i * ldc + j;
    float v = beta != 0.0f ? beta * *c : 0.0f;
    if (bias) v += bias[j];
    *c = v;
  }
}

cudaError_t launch_scale_c(float* C, int M, int N, int64_t ldc, float beta,
                           const float* bias, cudaStream_t stream, BoundsRecord* bounds) {
  const int64_t total = static_cast<int64_t>(M) * N;
  if (total <= 0) return cudaSuccess;
  const int64_t blocks = (total + 255) / 256;
  scale_c_kernel<<<static_cast<unsigned>(blocks < 65536 ? blocks : 65536), 256, 0, stream>>>(
      C, M, N, ldc, beta, bias, bounds);
  return cudaGetLastError();
}

// out[r * ldo + c] = op(src)[r][c] for r < R, c < cols, and 0.0 for
// cols <= c < ldo, with op(src)[r][c] = TRANS ? src[c * ld + r] : src[r * ld + c].
// 64 x 64 tiles of out through shared memory (a 65-word row stride: the
// transposed read of a column touches 32 distinct banks), so global reads
// and writes are both row-contiguous; each thread has 16 loads in flight.
// 1-D grid of tiles_r * tiles_c CTAs, 256 threads.
template <bool TRANS>
__global__ void __launch_bounds__(256) prep_operand_kernel(const float* __restrict__ src,
                                                           int64_t ld, float* __restrict__ out,
                                                           int64_t ldo, int R, int cols,
                                                           int tiles_c, BoundsRecord* rec) {
  const int64_t src_extent = TRANS ? view_extent(cols, R, ld) : view_extent(R, cols, ld);
  const int64_t out_extent = static_cast<int64_t>(R) * ldo;
  // No early griddepcontrol.launch_dependents here: the GEMM launched after
  // the copy would then be placed while the copy's CTAs hold every SM, and
  // its CTAs (up to three per SM) crowd onto fewer SMs.  Measured on GB300:
  // 1024^3 51 -> 123 us with the trigger at the top of this kernel.
  __shared__ float t[64][65];
  const int r0 = static_cast<int>(blockIdx.x / tiles_c) * 64;
  const int c0 = static_cast<int>(blockIdx.x % tiles_c) * 64;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
  for (int i = ty; i < 64; i += 8) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int x = tx + 32 * h;
      if constexpr (TRANS) {
        // Source row c0 + i holds column c0 + i of op(src): t[c][r].
        const int c = c0 + i, r = r0 + x;
        const int64_t o = static_cast<int64_t>(c) * ld + r;
        t[i][x] = c < cols && r < R && bounds_ok(rec, SITE_PREP_SRC, o, 1, src_extent) ? src[o]
                                                                                       : 0.0f;
      } else {
        const int r = r0 + i, c = c0 + x;
        const int64_t o = static_cast<int64_t>(r) * ld + c;
        t[i][x] = r < R && c < cols && bounds_ok(rec, SITE_PREP_SRC, o, 1, src_extent) ? src[o]
                                                                                       : 0.0f;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = ty; i < 64; i += 8) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int x = tx + 32 * h;
      const int r = r0 + i, c = c0 + x;
      if (r < R && c < ldo &&
          bounds_ok(rec, SITE_PREP_DST, static_cast<int64_t>(r) * ldo + c, 1, out_extent))
        out[static_cast<int64_t>(r) * ldo + c] = TRANS ? t[x][i] : t[i][x];
    }
  }
}

cudaError_t launch_prep_operand(const float* src, int64_t ld, bool trans, float* out,
                                int64_t ldo, int R, int cols, cudaStream_t stream,
                                BoundsRecord* bounds) {
  if (R <= 0 || ldo <= 0) return cudaSuccess;
  const int64_t tiles_r = (R + 63) / 64, tiles_c = (ldo + 63) / 64;
  if (tiles_c > INT32_MAX || tiles_r * tiles_c > INT32_MAX) return cudaErrorInvalidValue;
  const unsigned grid = static_cast<unsigned>(tiles_r * tiles_c);
  if (trans)
    prep_operand_kernel<true><<<grid, 256, 0, stream>>>(src, ld, out, ldo, R, cols,
                                                        static_cast<int>(tiles_c), bounds);
  else
    prep_operand_kernel<false><<<grid, 256, 0, stream>>>(src, ld, out, ldo, R, cols,
                                                         static_cast<int>(tiles_c), bounds);
  return cudaGetLastError();
}

int ffma_entries_128(FfmaEntry* out);
int ffma_entries_alt(FfmaEntry* out);
int ffma_entries_k16(FfmaEntry* out);
int ffma_entries_64(FfmaEntry* out);
int ffma_entries_depth(FfmaEntry* out);

const FfmaEntry* ffma_entries(int* count) {
  // Each tile unit fills at most kUnitMax entries into a scratch block;
  // only whole units that fit are kept, so the table never overruns.
  constexpr int kCapacity = 32, kUnitMax = 8;
  static FfmaEntry entries[kCapacity];
  static const int n = [] {
    int (*const units[])(FfmaEntry*) = {ffma_entries_128, ffma_entries_alt, ffma_entries_64,
                                        ffma_entries_k16, ffma_entries_depth};
    int k = 0;
    for (auto unit : units) {
      FfmaEntry scratch[kUnitMax] = {};
      const int got = unit(scratch);
      for (int i = 0; i < got && i < kUnitMax && k < kCapacity; ++i) entries[k++] = scratch[i];
    }
    return k;
  }();
  *count = n;
  return entries;
}

}  // namespace mt
