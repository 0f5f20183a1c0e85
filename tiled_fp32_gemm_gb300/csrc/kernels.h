// Internal interface between the host dispatcher (api.cu) and the kernel
// translation units.  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mt {

// Record of the accesses a checked build (compiled with MT_BOUNDS_CHECK=1)
// found outside their buffers: how many, and the first one's site, element
// offset and the buffer's extent in elements.  Those accesses are skipped
// (a copy becomes a zero fill, a load reads 0, a store is dropped), so a
// checked kernel never touches memory outside its buffers.
struct BoundsRecord {
  unsigned int count;
  int site;
  long long offset;
  long long extent;
};

// Access sites a checked build names in BoundsRecord::site.
enum BoundsSite {
  SITE_A_LOAD = 1,      // global read of A by the staging copies
  SITE_B_LOAD = 2,      // global read of B by the staging copies
  SITE_A_SMEM = 3,      // shared write of a staged A tile
  SITE_B_SMEM = 4,      // shared write of a staged B tile
  SITE_FRAG = 5,        // shared read of an A or B fragment by the micro-kernel
  SITE_C_STORE = 6,     // global read or write of C
  SITE_PARTIAL = 7,     // global read or write of a K-slice partial tile
  SITE_BIAS = 8,        // global read of the bias row
  SITE_SLICE_SUM = 9,   // shared read or write of a K group's sum
  SITE_PREP_SRC = 10,   // global read of an operand by the copy kernel
  SITE_PREP_DST = 11,   // global write of an operand copy
  SITE_P18 = 12         // any access of the one-warp kernel
};

// One compiled FFMA tile configuration and its kernel instantiations.
struct FfmaEntry {
  int bm, bn, bk, stages, threads, min_blocks;
  int kslices;         // K groups of warps inside a CTA (1 = none)
  int wm, wn, tm, tn;  // warp tile and per-thread tile
  int packed;          // 1: fma.rn.f32x2 micro-kernel, 0: scalar fma
  int pad_a, pad_b;    // padding words per shared row under the rule
  int smem_bytes[2];   // [pad] dynamic shared memory per CTA
  const void* kern[2][2];  // [vec][pad], untransposed operands; nullptr when not built
  // Transposed operands (4-byte staging, padded rows): [trans_a][trans_b],
  // [0][0] unused; nullptr when not built.
  const void* kern_t[2][2];
  int pad_b_t, smem_bytes_t;  // B padding and shared memory when B is transposed
  // 16-byte staging of A and B with scalar stores of C (padded rows);
  // nullptr when not built.
  const void* kern_vsc;
  // A staged K-major from A stored K x M (16-byte chunks), B as kern[1][1];
  // [vec_c].  smem_bytes_km: its dynamic shared memory.
  const void* kern_km[2];
  int smem_bytes_km;
  // A gathered K-major from row-major storage (4-byte copies), B as
  // kern[1][1]; [vec_c].  pad_a_kg: padding words of its K-major A rows.
  const void* kern_kg[2];
  int smem_bytes_kg, pad_a_kg;
};

// Copies op(src) (R x cols, op = transpose when trans) into row-major `out`
// with row pitch ldo >= cols, zero-filling columns cols..ldo-1: the layout
// the 16-byte staging reads, for operands it cannot read as stored.
cudaError_t launch_prep_operand(const float* src, int64_t ld, bool trans, float* out,
                                int64_t ldo, int R, int cols, cudaStream_t stream,
                                BoundsRecord* bounds = nullptr);

// C = beta * C (+ bias[col] when bias is not null) over an M x N view with
// row stride ldc (C is not read when beta is 0).  The whole product when
// alpha == 0 or K == 0.
cudaError_t launch_scale_c(float* C, int M, int N, int64_t ldc, float beta,
                           const float* bias, cudaStream_t stream,
                           BoundsRecord* bounds = nullptr);

// All FFMA configurations built into the library (null-terminated count).
const FfmaEntry* ffma_entries(int* count);

// Arguments every GEMM kernel receives:
//   C = alpha * op(A) * op(B) + beta * C   (beta == 0: C is not read)
// op(A)[i][k] = trans_a ? A[k*lda + i] : A[i*lda + k],
// op(B)[k][j] = trans_b ? B[j*ldb + k] : B[k*ldb + j], C[i][j] at C[i*ldc + j].
struct GemmArgs {
  const float* A;
  const float* B;
  float* C;
  int M, N, K;
  int tiles_m, tiles_n;
  int group_m;
  int64_t lda, ldb, ldc;
  float alpha, beta;
  int trans_a, trans_b;
  // N floats added to every row of C after alpha * op(A) * op(B) + beta * C
  // (nullptr: none).
  const float* bias;
  // Split-K tail (FFMA kernel): work units below full_tiles are whole tiles
  // (tile = unit, in grouped raster order); the remaining tiles are cut
  // into `split` K slices of kt_per_slice K tiles each, one unit per slice,
  // and each slice writes its fp32 partial tile to `partial` (dense
  // BM x BN blocks, slice-major per tile).  full_tiles = all tiles and
  // split = 1 when nothing is split.
  int full_tiles;
  int split;
  int kt_per_slice;
  float* partial;
  // Stream-K (FFMA kernel; sk_ctas > 0, split = 1): the tiles from
  // full_tiles on hold sk_iters K tiles in all (tile-major, k ascending);
  // unit full_tiles + c (c < sk_ctas) takes the contiguous run
  // [c*sk_iters/sk_ctas, (c+1)*sk_iters/sk_ctas) across tile boundaries.
  // A tile the run covers whole goes to C; a piece of a tile goes to
  // `partial` as a dense BM x BN block: slot 2c for the run's first tile,
  // 2c+1 for its last.  launch_streamk_fixup adds the pieces of each tile in
  // k order.
  int sk_ctas;
  int64_t sk_iters;
  // Elements from A, B, C, partial up to the last element the product
  // addresses (checked builds test every access against them), and the
  // checked build's record (nullptr otherwise).
  int64_t a_extent, b_extent, c_extent, partial_extent;
  BoundsRecord* bounds;
};

// Elements a rows x cols view with row pitch ld spans (0 if empty).
__host__ __device__ inline int64_t view_extent(int64_t rows, int64_t cols, int64_t ld) {
  return rows > 0 && cols > 0 ? (rows - 1) * ld + cols : 0;
}

// Sums the K-slice partials of the split tiles (in slice order, so the
// result does not depend on scheduling) and writes them to C with the
// edge masks (alpha, beta, bias applied).  bm*bn/4096 CTAs (at least one)
// per split tile, launched as a programmatic dependent of the GEMM kernel
// before it on `stream`.  A zero a.partial_extent is taken as one dense
// bm x bn tile per slice of each split tile.
cudaError_t launch_splitk_reduce(const GemmArgs& a, int bm, int bn, bool vec_c,
                                 cudaStream_t stream);

// Stream-K fix-up: for every stream-K tile that no single unit covered,
// adds its pieces (the partial slots of the units whose runs overlap it, in
// unit order, which is k order) and writes the sum to C with the edge masks
// (alpha, beta, bias applied); tiles a unit covered whole were written by
// the GEMM kernel and are skipped.  ktiles: K tiles per tile.  Launched as
// a programmatic dependent of the GEMM kernel before it on `stream`.
cudaError_t launch_streamk_fixup(const GemmArgs& a, int bm, int bn, int ktiles, bool vec_c,
                                 cudaStream_t stream);

// The second pass of a call whose GEMM kernel wrote partial tiles to
// `partial` (bm x bn each, ktiles K tiles per tile): the stream-K fix-up when
// a.sk_ctas > 0, the split-K reduce when a.split > 1, else nothing.
cudaError_t launch_second_pass(const GemmArgs& a, float* partial, int bm, int bn, int ktiles,
                               bool vec_c, cudaStream_t stream);

// CTAs (clusters, for CTA pairs) of a persistent grid with at most max_ctas
// resident: every unit gets one when they fit; with stream-K, the whole
// tiles' full waves or, without any, the stream-K units.
inline int persistent_grid(const GemmArgs& a, int units, int max_ctas) {
  if (a.sk_ctas > 0) return a.full_tiles > 0 ? max_ctas : a.sk_ctas;
  return units < max_ctas ? units : max_ctas;
}

// First unit of the stream-K split whose run holds stream-K iteration x:
// the largest c with c * iters / ctas <= x (runs may be empty when there
// are fewer iterations than units; the one returned is not).
__host__ __device__ inline int streamk_unit_of(int64_t x, int64_t iters, int ctas) {
  int64_t c = x * ctas / iters;  // c * iters / ctas <= x by construction, or one past
  while (c + 1 < ctas && (c + 1) * iters / ctas <= x) ++c;
  while (c > 0 && c * iters / ctas > x) --c;
  return static_cast<int>(c);
}

// The one-warp kernel restating the pages' Version 18 (BM=4, BN=8, BK=16,
// two stages, synchronous staging, padded A).  pad selects the rule's
// padding (true) or an unpadded A tile (false); stages = 1 selects the
// single-stage form with two barriers per K tile, else 2.
cudaError_t launch_p18(const GemmArgs& a, bool pad, int stages, cudaStream_t stream);
int p18_pad_a(bool pad);
int p18_smem_bytes(bool pad, int stages);

// tcgen05 3xTF32 variant (sgemm_tf32x3.cu): persistent kernel over tiles of
// 128 x bn (bm = 128; bn = 256, 128 or 64) or, on CTA pairs, of 256 x 256
// (bm = 256, bn = 256), with a K depth bk of 16 or 32 per stage.  A call
// needs a device workspace of tf32x3_workspace_bytes(M, N, K, bm, bk, bn)
// bytes (the packed, split, swizzled copies of A and B); launch_tf32x3 runs
// the two pack kernels and the GEMM on at most max_ctas CTAs (one per SM;
// bm = 256: clusters of two).
// split_a = 1: the split-A kernel (bm = 128, bk = 32, A not transposed with
// a 16-byte aligned base and lda % 4 == 0): A is split inside the GEMM
// kernel and only B is packed.
bool tf32x3_valid(int bm, int bk, int bn, int split_a);
int64_t tf32x3_workspace_bytes(int M, int N, int K, int bm, int bk, int bn, int split_a);
int tf32x3_smem_bytes(int bm, int bk, int bn, int split_a);
int tf32x3_stages(int bm, int bk, int bn, int split_a);
int tf32x3_threads(int split_a);
int tf32x3_bm();
cudaError_t tf32x3_prepare(int device, int bm, int bk, int bn, int split_a);
// Clusters of two of the pair kernel resident at once on `device` (the
// current device); 0 if the query fails.  Sets its shared-memory limit.
int tf32x3_pair_max_clusters(int device, int bk);
// vec_a / vec_b: that operand may be read with float4 by its packer (read
// k-contiguous, leading dimension % 4 == 0, 16-byte aligned); vec_c: C may
// be written with float4.  fault_inject = 1: the copy threads issue nothing
// (tests the bounded waits).
cudaError_t launch_tf32x3(const GemmArgs& a, void* workspace, bool vec_a, bool vec_b,
                          bool vec_c, int bm, int bk, int bn, int split_a, int max_ctas,
                          int fault_inject, cudaStream_t stream);
// Size of the static scratch the allocation-free tf32x3 entry point uses,
// and its device address on `device` (looked up once per device; the device
// must be current).
constexpr int64_t kNoAllocScratchBytes = int64_t(32) << 20;  // 32 MiB
cudaError_t tf32x3_noalloc_scratch(int device, void** ptr);
// Reads and zeroes the device status word of the tf32x3 kernels
// (bit 0: a bounded wait expired).  Synchronous.
cudaError_t tf32x3_read_and_clear_status(unsigned int* status);

// ---------------------------------------------------------------------------
// TMA tensor maps (tensor_map.cu).  A 2-D map of a rows x cols matrix of
// elem_bytes-byte elements with row pitch ld elements, boxes of box_cols x
// box_rows, zero fill outside the matrix.  false when the driver's encoder
// is unavailable or rejects the arguments.
bool tensor_map_encoder_available();
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, int elem_bytes,
                          const void* base, int64_t rows, int64_t cols, int64_t ld,
                          int box_cols, int box_rows, CUtensorMapSwizzle swizzle);

// ---------------------------------------------------------------------------
// tcgen05 kind::f16 kernel on 16-bit inputs (gemm_f16.cu).  GemmArgs carries
// the sizes, leading dimensions, transposes, alpha/beta, C and the split
// tail; its A and B are unused (the 16-bit operands come here).
struct F16Operands {
  const void* A;
  const void* B;
  int dtype;  // 1 = fp16, 2 = bf16
};

// Workspace of one call: padded copies of operands TMA cannot read in place
// (row pitch not a multiple of 16 bytes or base not 16-byte aligned), then
// the split tail's partial tiles.
struct F16Layout {
  int64_t repack_a_bytes, repack_b_bytes;
  int64_t partial_offset;
  int64_t workspace_bytes;
};

// Tiles: bm = 128 (one CTA per tile, bn = 256 or 128) or bm = 256 (a CTA
// pair per 256 x 256 tile, bn = 256).
F16Layout f16tc_layout(const GemmArgs& a, const F16Operands& f, int tile_m, int bn);
bool f16tc_valid(int bm, int bn);
int f16tc_smem_bytes(int bm, int bn);
int f16tc_stages(int bm, int bn);
int f16tc_threads();
int f16tc_bm();
int f16tc_bk();
cudaError_t f16tc_prepare(int bm, int bn);
// Clusters of two CTAs of the pair kernel resident at once on `device` (the
// current device); 0 if the query fails.  Sets the kernel's shared-memory
// limit on first use.
int f16tc_pair_max_clusters(int device);
// Whether the driver's tensor-map encoder could be looked up.
bool f16tc_encoder_available();
// max_ctas: CTAs of the persistent grid at most (bm = 256: clusters of two).
cudaError_t launch_f16tc(const GemmArgs& a, const F16Operands& f, void* workspace, bool vec_c,
                         int bm, int bn, int max_ctas, int fault_inject, cudaStream_t stream);
cudaError_t f16tc_read_and_clear_status(unsigned int* status);

}  // namespace mt
