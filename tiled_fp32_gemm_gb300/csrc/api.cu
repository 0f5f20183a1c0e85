// Host side of the C ABI: argument checks, variant and tile selection,
// shared-memory budget, launch, and the pure-host layout helpers.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_set>

#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kernels.h"
#include "mt_sgemm.h"
#include "smem_layout.cuh"

namespace {

constexpr int kMaxDevices = 64;
// K depth of the 3xTF32 kernel when the caller does not choose: 16 for
// 256-wide tiles (a 4-stage ring instead of 2), 32 for narrower tiles (3 or
// 4 stages, half the barrier round trips) — the faster of the two on GB300.
int tf32x3_default_bk(int bn) { return bn == 256 ? 16 : 32; }

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;  // max dynamic shared memory per block with opt-in
  bool valid = false;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
// Kernels whose dynamic shared-memory limit was raised, per device.
std::unordered_set<const void*> g_attr_done[kMaxDevices];
cudaMemPool_t g_pools[kMaxDevices];

mt_status current_device(int* dev, DeviceInfo* info) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
    cudaGetLastError();
    return MT_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& di = g_devices[d];
  if (!di.valid) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) !=
            cudaSuccess) {
      cudaGetLastError();
      return MT_ERR_NO_DEVICE;
    }
    di.valid = true;
  }
  *dev = d;
  *info = di;
  return MT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
  if (a_bytes <= 0 || b_bytes <= 0 || !a || !b) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Row pitch (floats) of an operand copied for the FFMA kernel's 16-byte
// staging: whole 128-byte lines, so every staged row segment starts on a
// line (a pitch rounded only to 16 bytes left the ragged case's rows 16 or
// 112 bytes off a line, each 512-byte segment touching five lines).
int64_t copy_pitch(int64_t cols) { return ceil_div(std::max<int64_t>(cols, 1), 32) * 32; }

// One product: C = alpha * op(A) * op(B) + beta * C (see GemmArgs).  A and
// B hold fp32 values (dtype 0) or 16-bit ones (MT_DTYPE_F16 / MT_DTYPE_BF16).
struct Problem {
  const void* A;
  const void* B;
  float* C;
  int64_t M, N, K;
  int64_t lda, ldb, ldc;
  float alpha, beta;
  int trans_a, trans_b;
  int dtype;
  const float* bias;  // N floats added to every row of C (nullptr: none)
};

int ab_bytes(const Problem& P) { return P.dtype ? 2 : 4; }

// The packed row-major product C = A*B (a leading dimension of at least 1
// keeps empty operands valid).
Problem packed_problem(const void* A, const void* B, float* C, int64_t M, int64_t N,
                       int64_t K, int dtype = 0) {
  const int64_t lda = K > 0 ? K : 1, ldn = N > 0 ? N : 1;
  return Problem{A, B, C, M, N, K, lda, ldn, ldn, 1.0f, 0.0f, 0, 0, dtype};
}

// Everything a launch needs beyond the plan the caller can see.
struct Launch {
  mt_plan plan;
  int entry = -1;  // FFMA table index
  const void* kern = nullptr;
  int tiles_m = 0, tiles_n = 0, group_m = 8;
  bool pad = true;
  int fault_inject = 0;
  int max_ctas = 0;  // persistent kernels: CTAs to launch at most
  // FFMA split-K and stream-K (see GemmArgs).
  int full_tiles = 0, split = 1, kt_per_slice = 0;
  int sk_ctas = 0;
  int64_t sk_iters = 0;
  // 3xTF32: float4 reads of A / B by their packers; A split inside the
  // GEMM kernel instead of packed.
  bool vec_a = false, vec_b = false;
  int split_a = 0;
  // FFMA: operands copied into zero-padded row-major scratch first (row
  // pitches ldo_a = copy_pitch(K), ldo_b = copy_pitch(N)); workspace
  // layout [copy of A][copy of B][split-K partials].
  bool prep_a = false, prep_b = false;
  int64_t ldo_a = 0, ldo_b = 0, prep_b_offset = 0, partial_offset = 0;
  // FFMA with A staged K-major: A is read as a K x M matrix (stored so, or
  // copied so into scratch with pitch ldo_a = copy_pitch(M) when
  // prep_a_kmajor), or gathered from row-major storage (a_gather).
  bool a_kmajor = false, prep_a_kmajor = false, a_gather = false;
};

mt_status check_dims(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
    return MT_ERR_INVALID_ARG;
  // Every operand must be addressable with 64-bit byte offsets.
  const int64_t lim = (INT64_MAX / 4) >> 1;
  if ((M && N > lim / M) || (M && K > lim / M) || (K && N > lim / K)) return MT_ERR_INVALID_ARG;
  return MT_OK;
}

// Bytes from the first to one past the last element of a rows x cols view
// with row stride ld and elements of `elem` bytes.
int64_t extent_bytes(int64_t rows, int64_t cols, int64_t ld, int elem = 4) {
  return rows > 0 && cols > 0 ? ((rows - 1) * ld + cols) * elem : 0;
}

// Leading dimensions: each stored row must hold its logical row.
mt_status check_lds(const Problem& P) {
  const int64_t lim = INT64_MAX / 16;
  if (P.lda < std::max<int64_t>(1, P.trans_a ? P.M : P.K) ||
      P.ldb < std::max<int64_t>(1, P.trans_b ? P.K : P.N) || P.ldc < std::max<int64_t>(1, P.N) ||
      P.lda > lim || P.ldb > lim || P.ldc > lim)
    return MT_ERR_INVALID_ARG;
  if ((P.trans_a ? P.K : P.M) > 0 && P.lda > lim / std::max<int64_t>(1, P.trans_a ? P.K : P.M))
    return MT_ERR_INVALID_ARG;
  if ((P.trans_b ? P.N : P.K) > 0 && P.ldb > lim / std::max<int64_t>(1, P.trans_b ? P.N : P.K))
    return MT_ERR_INVALID_ARG;
  if (P.M > 0 && P.ldc > lim / P.M) return MT_ERR_INVALID_ARG;
  return MT_OK;
}

// Whether A and B are read at all (BLAS: not when alpha == 0 or K == 0).
bool reads_ab(const Problem& P) { return P.K > 0 && P.alpha != 0.0f; }

mt_status check_problem(const Problem& P) {
  mt_status st = check_dims(P.M, P.N, P.K);
  if (st != MT_OK) return st;
  if (P.trans_a < 0 || P.trans_a > 1 || P.trans_b < 0 || P.trans_b > 1) return MT_ERR_INVALID_ARG;
  st = check_lds(P);
  if (st != MT_OK) return st;
  if (P.M == 0 || P.N == 0) return MT_OK;
  if (!P.C || !aligned4(P.C)) return MT_ERR_INVALID_ARG;
  const int e = ab_bytes(P);
  const uintptr_t amask = static_cast<uintptr_t>(e - 1);
  if (reads_ab(P) && (!P.A || !P.B || (reinterpret_cast<uintptr_t>(P.A) & amask) ||
                      (reinterpret_cast<uintptr_t>(P.B) & amask)))
    return MT_ERR_INVALID_ARG;
  const int64_t c_bytes = extent_bytes(P.M, P.N, P.ldc);
  if (reads_ab(P)) {
    const int64_t a_bytes = P.trans_a ? extent_bytes(P.K, P.M, P.lda, e)
                                      : extent_bytes(P.M, P.K, P.lda, e);
    const int64_t b_bytes = P.trans_b ? extent_bytes(P.N, P.K, P.ldb, e)
                                      : extent_bytes(P.K, P.N, P.ldb, e);
    if (overlaps(P.C, c_bytes, P.A, a_bytes) || overlaps(P.C, c_bytes, P.B, b_bytes))
      return MT_ERR_ALIAS;
  }
  if (P.bias) {
    // Read by every row's epilogue while C is written.
    if (!aligned4(P.bias)) return MT_ERR_INVALID_ARG;
    if (overlaps(P.C, c_bytes, P.bias, P.N * 4)) return MT_ERR_ALIAS;
  }
  return MT_OK;
}


// Chooses the FFMA table entry.  Explicit choices (tile, stages, warp tile,
// micro-kernel form) must all match one entry; the first match in table
// order wins, so each tile's default warp layout comes first.  Otherwise
// the choice is automatic.
int pick_ffma(const mt_config* cfg, int64_t M, int64_t N, int64_t K, int sms, bool kmajor) {
  // Stream-K runs need one group of warps per tile: no K-grouped tile then.
  const bool kgroups_ok = !(cfg && cfg->schedule == 2);
  int count = 0;
  const mt::FfmaEntry* e = mt::ffma_entries(&count);
  const bool explicit_tile = cfg && (cfg->bm || cfg->bn || cfg->bk || cfg->stages || cfg->wm ||
                                     cfg->wn || cfg->tm || cfg->tn);
  const int want_packed = cfg && cfg->fma ? (cfg->fma == 2 ? 1 : 0) : 1;
  if (explicit_tile || (cfg && cfg->fma)) {
    for (int i = 0; i < count; ++i) {
      if (cfg->bm && e[i].bm != cfg->bm) continue;
      if (cfg->bn && e[i].bn != cfg->bn) continue;
      if (cfg->bk && e[i].bk != cfg->bk) continue;
      if (cfg->stages && e[i].stages != cfg->stages) continue;
      if (cfg->wm && e[i].wm != cfg->wm) continue;
      if (cfg->wn && e[i].wn != cfg->wn) continue;
      if (cfg->tm && e[i].tm != cfg->tm) continue;
      if (cfg->tn && e[i].tn != cfg->tn) continue;
      if (e[i].packed != want_packed) continue;
      if (!explicit_tile && !(e[i].bm == 128 && e[i].bn == 128 && e[i].stages == 3)) continue;
      return i;
    }
    return -1;
  }
  // Automatic.  Row-major A: 128x128 tiles when they fill every SM twice
  // over, else 64x64 tiles for more CTAs.  K-major A: 128x128 tiles from
  // three full waves (2 CTAs per SM) up, else 64x128 tiles (3 CTAs per SM)
  // when there are at least half as many as SMs, else 64x64.  Measured on
  // GB300 (K-major A): 4097 x 3001 x 2053 54.7 TFLOP/s on 64x128 tiles
  // against 49.3 on 128x128, 65536 x 128 x 4096 60.7 against 53.5, 1024^3
  // 38.4 against 33.5 on 64x64.  Fewer 64x128 tiles than that with K >=
  // 2048: 64x128 tiles with two K groups of warps per CTA (512 x 512 x 4096
  // 62 us against 82 on 64x64; with K = 768 it lost, 44 us against 31).
  int big = -1, big_km = -1, mid = -1, small = -1, sliced = -1;
  for (int i = 0; i < count; ++i) {
    if (!e[i].packed) continue;
    if (big < 0 && e[i].bm == 128 && e[i].bn == 128 && e[i].bk == 32 && e[i].stages == 3)
      big = i;
    // K-major A: the K depth 16 tile (0.5 % faster at 4096^3 and 8192^3).
    if (big_km < 0 && e[i].bm == 128 && e[i].bn == 128 && e[i].bk == 16 && e[i].wm == 64 &&
        e[i].kern_km[0])
      big_km = i;
    if (mid < 0 && e[i].bm == 64 && e[i].bn == 128 && e[i].kslices == 1 && e[i].kern_km[0])
      mid = i;
    if (sliced < 0 && e[i].kslices > 1 && e[i].kern_km[0]) sliced = i;
    if (small < 0 && e[i].bm == 64 && e[i].bn == 64) small = i;
  }
  const int64_t tiles_big = ceil_div(M, 128) * ceil_div(N, 128);
  if (!kmajor) {
    if (tiles_big >= 2 * static_cast<int64_t>(sms) || small < 0) return big;
    return small;
  }
  if (big_km >= 0) big = big_km;
  if (tiles_big >= 6 * static_cast<int64_t>(sms) || (mid < 0 && small < 0)) return big;
  if (mid >= 0 && 2 * ceil_div(M, 64) * ceil_div(N, 128) >= static_cast<int64_t>(sms)) return mid;
  if (sliced >= 0 && K >= 2048 && kgroups_ok) return sliced;
  return small >= 0 ? small : big;
}

// Tile width of a persistent tensor-core kernel: the widest tile wins
// unless padding N up to it, or too few tiles for the SMs, costs more than
// its higher per-tile efficiency (`weight`, relative to the first width).
int pick_tile_bn(int64_t M, int64_t N, int sms, const int* widths, const double* weight,
                 int count) {
  int best = widths[0];
  double best_score = -1.0;
  for (int i = 0; i < count; ++i) {
    const int bn = widths[i];
    const int64_t nt = ceil_div(N, bn);
    const double used = static_cast<double>(N) / static_cast<double>(nt * bn);
    const int64_t tiles = ceil_div(M, 128) * nt;
    const double waves = static_cast<double>(tiles) / sms;
    const double fill = waves >= 1.0 ? waves / static_cast<double>(ceil_div(tiles, sms))
                                     : waves;
    const double score = used * fill * weight[i];
    if (score > best_score + 1e-9) {
      best_score = score;
      best = bn;
    }
  }
  return best;
}

// 3xTF32: per-tile throughput relative to 256-wide tiles measured at 8192^3
// and 4096^3 on GB300 (narrower tiles re-read A from shared memory for
// fewer columns).
int pick_tf32x3_bn(int64_t M, int64_t N, int sms) {
  static const int widths[3] = {256, 128, 64};
  static const double weight[3] = {1.0, 0.7, 0.4};
  return pick_tile_bn(M, N, sms, widths, weight, 3);
}

// 16-bit kernel: 256- or 128-wide tiles.
int pick_f16_bn(int64_t M, int64_t N, int sms) {
  static const int widths[2] = {256, 128};
  static const double weight[2] = {1.0, 0.8};
  return pick_tile_bn(M, N, sms, widths, weight, 2);
}

// Split tail of a persistent kernel: when `tiles` leave a last round on at
// most half of the `ctas` CTAs, those tiles are cut into K slices that run
// on the idle ones (at most 4, every slice non-empty and at least 2 K tiles
// long) and are added by a second kernel.  Outputs the whole tiles and the
// slice count (1: no split).  slices = 0: as many slices as fit the idle
// CTAs (at most 4); else that many (fewer if K is short).
void split_tail(int64_t tiles, int64_t ctas, int64_t ktiles, bool allowed, int64_t* full,
                int64_t* split, int slices = 0) {
  *full = tiles;
  *split = 1;
  if (!allowed || tiles <= ctas) return;
  const int64_t rem = tiles % ctas;
  if (rem == 0 || 2 * rem > ctas) return;
  int64_t s = slices > 0 ? slices : std::min<int64_t>(ctas / rem, 4);
  while (s > 1 && ((s - 1) * ceil_div(ktiles, s) >= ktiles || ktiles / s < 2)) --s;
  if (s > 1) {
    *full = tiles - rem;
    *split = s;
  }
}

mt::GemmArgs make_args(const Problem& P, const Launch& L);

#if MT_BOUNDS_CHECK
// The checked build's record of out-of-range accesses; kernels get its
// device address through GemmArgs::bounds (looked up once per device).
__device__ mt::BoundsRecord g_bounds;
mt::BoundsRecord* g_bounds_ptr[kMaxDevices];
#endif

// The record the current device's kernels write to: nullptr in normal
// builds (and if the lookup fails).
mt::BoundsRecord* bounds_record() {
#if MT_BOUNDS_CHECK
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_bounds_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bounds) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_bounds_ptr[d] = static_cast<mt::BoundsRecord*>(p);
  }
  return g_bounds_ptr[d];
#else
  return nullptr;
#endif
}

// The automatic 16-bit plan takes CTA pairs (256 x 256 tiles) when 256-wide
// tiles are chosen and there are at least as many pair tiles as resident
// clusters: on GB300 pairs run 8192^3 bf16 at 1.19x and 4096^3 at 1.10x the
// single-CTA 128 x 256 tiles, but are slower with fewer tiles than clusters
// (1024^3: 0.79x).
bool auto_pair(int64_t M, int64_t N, int bn, int sms, int pair_clusters) {
  if (bn != 256) return false;
  const int64_t clusters = pair_clusters > 0 ? pair_clusters : std::max(1, sms / 2);
  return ceil_div(M, 256) * ceil_div(N, 256) >= clusters;
}

// Small grid of a persistent tensor-core kernel: fewer tiles than half the
// resident CTAs (clusters) are cut into K slices, so more of them work (at
// most 4 slices, as many as fit, each at least 1024 deep; the slices are
// added by the second kernel).  Measured on GB300: 512 x 512 x 4096 with
// bf16 inputs 27.3 -> 22.2 us and 3xTF32 98.0 -> 45.8 us in four slices;
// 1024^3 bf16 lost in two slices of 512 (15.0 -> 18.1 us).  Leaves *full
// and *split alone otherwise.
void split_small_grid(int64_t tiles, int64_t max_ctas, int64_t K, int bk, int64_t* full,
                      int64_t* split) {
  if (tiles <= 0 || 2 * tiles > max_ctas) return;
  const int64_t ktiles = ceil_div(K, bk);
  int64_t s = std::min<int64_t>(4, max_ctas / tiles);
  while (s > 1 && ((s - 1) * ceil_div(ktiles, s) >= ktiles || K / s < 1024)) --s;
  if (s > 1) {
    *full = 0;
    *split = s;
  }
}

// Stream-K plan of a persistent tensor-core kernel (schedule 2) over
// `tiles` tiles of `ktiles` K tiles on `max_ctas` resident CTAs (clusters):
// the full waves stay whole tiles; the tiles past them are dealt out as
// contiguous runs of K tiles, at least two per run.  Sets the launch's
// stream-K fields; false when there is nothing to deal out.
bool plan_persistent_streamk(int64_t tiles, int64_t ktiles, int max_ctas, Launch* L) {
  const int64_t G = std::max(1, max_ctas);
  const int64_t rem = tiles % G;
  if (rem == 0 || ktiles <= 0) return false;
  L->full_tiles = static_cast<int>(tiles - rem);
  L->split = 1;
  L->sk_iters = rem * ktiles;
  L->sk_ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(G, L->sk_iters / 2)));
  return true;
}

// The 16-bit kernels (MT_VARIANT_TC16): 128 x BN tiles on one CTA, or 256 x
// 256 tiles on a CTA pair (bm = 256); BK = 64, persistent with a split
// tail; operands TMA cannot read in place are copied first.  pair_clusters:
// clusters of two resident at once (0: half the SMs).
mt_status plan_f16(const Problem& P, const mt_config* cfg, int64_t smem_limit, int sms,
                   int pair_clusters, Launch* L) {
  if (P.dtype != MT_DTYPE_F16 && P.dtype != MT_DTYPE_BF16) return MT_ERR_INVALID_ARG;
  if (cfg && cfg->variant != MT_VARIANT_FFMA && cfg->variant != MT_VARIANT_TC16)
    return MT_ERR_UNSUPPORTED;
  if (cfg && (cfg->wm || cfg->wn || cfg->tm || cfg->tn || cfg->fma || cfg->no_pad ||
              cfg->split_k > 1 || cfg->pack_a))
    return MT_ERR_UNSUPPORTED;
  const int64_t M = P.M, N = P.N, K = P.K;
  const int bk = mt::f16tc_bk();
  const int want_bm = cfg ? cfg->bm : 0;
  const int bn = cfg && cfg->bn ? cfg->bn
                 : want_bm == 256 ? 256 : pick_f16_bn(M, N, sms > 0 ? sms : 1);
  const int bm = want_bm ? want_bm
                         : auto_pair(M, N, bn, sms, pair_clusters) ? 256 : mt::f16tc_bm();
  if (!mt::f16tc_valid(bm, bn)) return MT_ERR_UNSUPPORTED;
  const int stages = mt::f16tc_stages(bm, bn);
  if (cfg && ((cfg->bk && cfg->bk != bk) || (cfg->stages && cfg->stages != stages)))
    return MT_ERR_UNSUPPORTED;
  const bool pair = bm == 256;
  L->fault_inject = cfg ? cfg->fault_inject : 0;
  if (cfg && cfg->group_m) L->group_m = cfg->group_m;
  mt_plan& p = L->plan;
  std::memset(&p, 0, sizeof(p));
  p.variant = MT_VARIANT_TC16;
  p.bm = bm; p.bn = bn; p.bk = bk; p.stages = stages;
  p.threads = mt::f16tc_threads();
  p.vec_c = N % 4 == 0 && P.ldc % 4 == 0 && aligned16(P.C);
  p.smem_bytes = mt::f16tc_smem_bytes(bm, bn);
  const int64_t tiles_m = ceil_div(M, bm), tiles_n = ceil_div(N, bn);
  if (tiles_m * tiles_n > INT32_MAX / 8) return MT_ERR_UNSUPPORTED;
  L->tiles_m = static_cast<int>(tiles_m);
  L->tiles_n = static_cast<int>(tiles_n);
  const int64_t tiles = tiles_m * tiles_n;
  // Persistent: one CTA per SM, or one cluster of two per two SMs.
  if (pair) L->max_ctas = pair_clusters > 0 ? pair_clusters : std::max(1, sms / 2);
  else L->max_ctas = sms > 0 ? sms : 1;
  int64_t full = tiles, split = 1;
  const bool streamk = cfg && cfg->schedule == 2 && cfg->split_k != 1;
  if (!streamk && !(cfg && cfg->split_k == 1)) {
    split_tail(tiles, std::min<int64_t>(tiles, L->max_ctas), ceil_div(K, bk), true, &full,
               &split);
    split_small_grid(tiles, L->max_ctas, K, bk, &full, &split);
  }
  L->full_tiles = static_cast<int>(full);
  L->split = static_cast<int>(split);
  L->kt_per_slice = static_cast<int>(ceil_div(ceil_div(K, bk), split));
  if (streamk) plan_persistent_streamk(tiles, ceil_div(K, bk), L->max_ctas, L);
  p.split_k = L->split;
  p.stream_k = L->sk_ctas;
  p.grid = (L->sk_ctas > 0 ? (L->full_tiles > 0 ? L->max_ctas : L->sk_ctas)
                           : std::min<int64_t>(full + (tiles - full) * split, L->max_ctas)) *
           (pair ? 2 : 1);
  const mt::F16Layout lay =
      mt::f16tc_layout(make_args(P, *L), mt::F16Operands{P.A, P.B, P.dtype}, bm, bn);
  p.vec_ab = lay.repack_a_bytes == 0 && lay.repack_b_bytes == 0;
  p.workspace_bytes = lay.workspace_bytes;
  if (p.smem_bytes > smem_limit) return MT_ERR_SMEM_BUDGET;
  return MT_OK;
}

// Pointers are only inspected for alignment here (NULL counts as aligned);
// check_problem checks them against the sizes.
// dev: the current device (-1 without one), asked for the resident-cluster
// count of the CTA-pair kernels.
// The 3xTF32 plan (called by plan_call after the common checks): A packed or
// split in the kernel, tile, K depth, CTA pairs, split tail and workspace.
mt_status plan_tf32x3(const Problem& P, const mt_config* cfg, int64_t smem_limit, int sms,
                      int dev, Launch* L) {
  const int64_t M = P.M, N = P.N, K = P.K;
  mt_plan& p = L->plan;
  const int want_bm = cfg ? cfg->bm : 0;
  // A split inside the GEMM kernel instead of packed (one CTA per tile):
  // for up to 1024 columns or products up to 2048^3, where packing A costs
  // more than it saves; A must be readable by TMA as stored.  Measured on
  // GB300 against packing: 65536 x 128 x 4096 2.3x, 65536 x 256 x 4096
  // 1.9x, 16384 x 512 x 4096 1.3x, 8192 x 1024 x 4096 1.1x, 2048^3 1.07x;
  // 4096 x 2048 x 4096 0.97x and 4096^3 0.73x (packing stays there).
  const bool a_tma_ok = !P.trans_a && P.lda % 4 == 0 && aligned16(P.A);
  const int want_pack = cfg ? cfg->pack_a : 0;
  const int split_a =
      want_pack == 2 ? 1
      : want_pack == 1 ? 0
      : (a_tma_ok && want_bm != 256 && (N <= 1024 || M * N * K <= (int64_t(1) << 33))) ? 1
                                                                                       : 0;
  if (split_a && (want_bm == 256 || !a_tma_ok)) return MT_ERR_UNSUPPORTED;
  const int bn = cfg && cfg->bn ? cfg->bn
                 : want_bm == 256 ? 256 : pick_tf32x3_bn(M, N, sms > 0 ? sms : 1);
  // CTA pairs (256 x 256 tiles, K depth 16 unless asked) when the pair
  // tiles fill the resident clusters, as for 16-bit inputs.
  const int pair_clusters16 = dev >= 0 ? mt::tf32x3_pair_max_clusters(dev, 16) : 0;
  const int bm = want_bm ? want_bm
                 : !split_a && auto_pair(M, N, bn, sms, pair_clusters16) ? 256
                                                                          : mt::tf32x3_bm();
  const bool pair = bm == 256;
  // Split-A: K depth 16 for 256-wide tiles (4 stages instead of 2), 32
  // for narrower ones (fewer, longer stages measured faster).
  const int bk = cfg && cfg->bk ? cfg->bk
                 : split_a ? (bn == 256 ? 16 : 32) : pair ? 16 : tf32x3_default_bk(bn);
  if (!mt::tf32x3_valid(bm, bk, bn, split_a)) return MT_ERR_UNSUPPORTED;
  const int stages = mt::tf32x3_stages(bm, bk, bn, split_a);
  if (cfg && ((cfg->stages && cfg->stages != stages) || cfg->fma || cfg->no_pad))
    return MT_ERR_UNSUPPORTED;
  p.bm = bm; p.bn = bn; p.bk = bk; p.stages = stages;
  p.threads = mt::tf32x3_threads(split_a);
  p.pack_a = split_a ? 2 : 1;
  L->split_a = split_a;
  p.pad_a = 0; p.pad_b = 0;  // swizzled tiles: the tensor core's layout, no padding
  // A packer reads float4 when it walks k-contiguous rows (A as stored,
  // B stored transposed) that are whole float4s from an aligned base.
  L->vec_a = !P.trans_a && K % 4 == 0 && P.lda % 4 == 0 && aligned16(P.A);
  L->vec_b = P.trans_b && K % 4 == 0 && P.ldb % 4 == 0 && aligned16(P.B);
  p.vec_ab = L->vec_a;
  p.vec_c = N % 4 == 0 && P.ldc % 4 == 0 && aligned16(P.C);
  p.smem_bytes = mt::tf32x3_smem_bytes(bm, bk, bn, split_a);
  L->tiles_m = static_cast<int>(ceil_div(M, bm));
  L->tiles_n = static_cast<int>(ceil_div(N, bn));
  // Pack grids: up to 65535 blocks of rows per operand.
  const int64_t blocks_m = pair ? 2 * L->tiles_m : L->tiles_m;
  const int64_t blocks_n = pair ? 2 * L->tiles_n : L->tiles_n;
  if (blocks_m > 65535 || blocks_n > 65535 ||
      ceil_div(static_cast<int64_t>(L->tiles_n) * bn, 256) > 65535 ||
      ceil_div(static_cast<int64_t>(L->tiles_m) * bm, 256) > 65535)
    return MT_ERR_UNSUPPORTED;
  // Persistent: one CTA per SM, or one cluster of two per two SMs.
  const int64_t tiles = static_cast<int64_t>(L->tiles_m) * L->tiles_n;
  if (pair) {
    const int pc = dev >= 0 ? mt::tf32x3_pair_max_clusters(dev, bk) : 0;
    L->max_ctas = pc > 0 ? pc : std::max(1, sms / 2);
  } else {
    L->max_ctas = sms > 0 ? sms : 1;
  }
  // Split tail (split_k = 1 turns it off).
  const int64_t ctas = std::min<int64_t>(tiles, L->max_ctas);
  const int64_t ktiles = ceil_div(K, bk);
  int64_t full = tiles, split = 1;
  const bool streamk = cfg && cfg->schedule == 2 && cfg->split_k != 1;
  if (!streamk && !(cfg && cfg->split_k == 1)) {
    split_tail(tiles, ctas, ktiles, true, &full, &split);
    split_small_grid(tiles, L->max_ctas, K, bk, &full, &split);
  }
  L->full_tiles = static_cast<int>(full);
  L->split = static_cast<int>(split);
  L->kt_per_slice = static_cast<int>(ceil_div(ktiles, split));
  if (streamk) plan_persistent_streamk(tiles, ktiles, L->max_ctas, L);
  p.split_k = L->split;
  p.stream_k = L->sk_ctas;
  const int64_t units = full + (tiles - full) * split;
  p.grid = (L->sk_ctas > 0 ? (L->full_tiles > 0 ? L->max_ctas : L->sk_ctas)
                           : std::min<int64_t>(units, L->max_ctas)) *
           (pair ? 2 : 1);
  p.workspace_bytes = mt::tf32x3_workspace_bytes(static_cast<int>(M), static_cast<int>(N),
                                                 static_cast<int>(K), bm, bk, bn, split_a) +
                      (L->sk_ctas > 0 ? 2 * static_cast<int64_t>(L->sk_ctas)
                                      : (tiles - full) * split) *
                          bm * bn * 4;
  if (p.smem_bytes > smem_limit) return MT_ERR_SMEM_BUDGET;
  return MT_OK;
}

// The FFMA plan (called by plan_call after the common checks): the tile,
// A's layout and source, operand copies, K slices, workspace and shared
// memory.
mt_status plan_ffma(const Problem& P, const mt_config* cfg, int64_t smem_limit, int sms,
                    bool pad, bool trans, Launch* L) {
  const int64_t M = P.M, N = P.N, K = P.K;
  mt_plan& p = L->plan;

  int count = 0;
  const mt::FfmaEntry* e = mt::ffma_entries(&count);
  // A staged K-major (pack_a 3-5, and automatically when padding is on
  // and B can be staged in 16-byte chunks, as stored or, for products with
  // 512 rows or more, from a copy): the micro-kernel then reads four rows of
  // A with one float4 per k, which measured 9-12 % faster on GB300 than
  // row-major A tiles (4096^3 67.4 against 59.9 TFLOP/s with A given K x M).
  const int want_pack = cfg ? cfg->pack_a : 0;
  const bool b_vec = !P.trans_b && N % 4 == 0 && P.ldb % 4 == 0 && aligned16(P.B);
  const bool kmajor = want_pack >= 3 || (want_pack == 0 && pad && (b_vec || M >= 512));
  const int i = pick_ffma(cfg, M, N, K, sms > 0 ? sms : 1, kmajor);
  if (i < 0) return MT_ERR_UNSUPPORTED;
  const mt::FfmaEntry& E = e[i];
  // Operands the 16-byte staging cannot read as stored (transposed, rows
  // not whole float4s, unaligned base) are copied once into zero-padded
  // row-major scratch when the product repays the pass (2^30 multiply-adds
  // or more), or when asked (pack_a = 1; pack_a = 2 stages them as stored).
  // The copy is exact and the zero padding multiplies zero-filled rows of
  // the other operand, so the result is the same FMA chain.
  const bool a_vec = !P.trans_a && K % 4 == 0 && P.lda % 4 == 0 && aligned16(P.A);
  const bool c_vec = N % 4 == 0 && P.ldc % 4 == 0 && aligned16(P.C);
  const auto round256 = [](int64_t b) { return (b + 255) / 256 * 256; };
  if (kmajor && !(pad && E.kern_km[0] && E.kern_kg[0])) {
    if (want_pack >= 3) return MT_ERR_UNSUPPORTED;
  } else if (kmajor) {
    // The K-major A tile comes straight from A stored K x M when its rows
    // are whole float4s; otherwise from a K x M copy (pack_a = 5, or
    // automatically for A stored K x M, and for A stored M x K when N >=
    // 1024 and the product has 2^30 multiply-adds or more: the transposing
    // pass costs about 70 / N of the product), else gathered element by
    // element from A stored M x K inside the GEMM kernel (pack_a = 4, about
    // 9 % slower than a K-major source on 4096^3).  Measured on GB300 at
    // 1024^3 (64 x 128 tiles): 52.7 us from the copy against 55.2 gathered;
    // at N = 128 (65536 x 128 x 4096) the copy loses, 40 against 61 TFLOP/s.
    // B as the 16-byte staging reads it, copied first when it cannot be read
    // as stored.
    const bool direct = P.trans_a && M % 4 == 0 && P.lda % 4 == 0 && aligned16(P.A);
    if (want_pack == 4 && P.trans_a) return MT_ERR_UNSUPPORTED;
    // For A stored M x K the automatic copy is capped at 2 GiB of workspace
    // (A^T is as large as A): a larger A is gathered, which needs none.  A
    // stored K x M that cannot be read as stored is always copied (the
    // gather reads A stored M x K only).
    const int64_t copy_bytes = K * copy_pitch(M) * 4;
    const bool copy = want_pack == 5 ||
                      (want_pack != 4 && !direct &&
                       (P.trans_a ||
                        (copy_bytes <= (int64_t(2) << 30) && N >= 1024 &&
                         static_cast<double>(M) * N * K >= 1073741824.0)));
    L->a_kmajor = true;
    L->prep_a_kmajor = copy;
    L->a_gather = !direct && !copy;
    L->prep_b = !b_vec;
    L->ldo_a = copy_pitch(M);
    L->ldo_b = copy_pitch(N);
    L->kern = L->a_gather ? E.kern_kg[c_vec ? 1 : 0] : E.kern_km[c_vec ? 1 : 0];
    p.vec_ab = L->a_gather ? 0 : 1;
    p.vec_c = c_vec ? 1 : 0;
    p.pack_a = L->a_gather ? 4 : copy ? 5 : 3;
    p.pad_a = L->a_gather ? E.pad_a_kg : 0;
    p.pad_b = E.pad_b;
    p.smem_bytes = L->a_gather ? E.smem_bytes_kg : E.smem_bytes_km;
    L->prep_b_offset = L->prep_a_kmajor ? round256(K * L->ldo_a * 4) : 0;
  }
  const bool prep = !L->a_kmajor && pad && E.kern_vsc && (!a_vec || !b_vec) &&
                    (want_pack == 1 ||
                     (want_pack == 0 && static_cast<double>(M) * N * K >= 1073741824.0));
  if (!L->a_kmajor) {
    L->prep_a = prep && !a_vec;
    L->prep_b = prep && !b_vec;
  }
  const bool a_ok = a_vec || L->prep_a, b_ok = b_vec || L->prep_b;
  const bool b_staged_trans = P.trans_b && !L->prep_b;
  const void* kern = nullptr;
  if (L->a_kmajor) {
    kern = L->kern;
  } else if (a_ok && b_ok) {
    // 16-byte staging of both; float4 or scalar stores of C.
    kern = c_vec ? E.kern[1][pad ? 1 : 0] : (pad ? E.kern_vsc : E.kern[0][0]);
    p.vec_ab = c_vec || pad ? 1 : 0;
    p.vec_c = c_vec ? 1 : 0;
  } else if (trans) {
    kern = pad ? E.kern_t[P.trans_a][P.trans_b] : nullptr;
    p.vec_ab = 0;
    p.vec_c = 0;
  } else {
    kern = E.kern[0][pad ? 1 : 0];
    p.vec_ab = 0;
    p.vec_c = 0;
  }
  if (!kern) return MT_ERR_UNSUPPORTED;
  // A kernel that stages an operand in 16-byte chunks must get it 16-byte
  // readable (as stored, or from its copy); anything else is a planning
  // error, refused before a launch could read misaligned memory.
  if (L->a_kmajor ? !(b_vec || L->prep_b) ||
                        !(L->a_gather || L->prep_a_kmajor ||
                          (P.trans_a && M % 4 == 0 && P.lda % 4 == 0 && aligned16(P.A)))
                  : p.vec_ab && !(a_ok && b_ok))
    return MT_ERR_UNSUPPORTED;
  p.bm = E.bm; p.bn = E.bn; p.bk = E.bk; p.stages = E.stages; p.threads = E.threads;
  p.fma = E.packed ? 2 : 1;
  p.wm = E.wm; p.wn = E.wn; p.tm = E.tm; p.tn = E.tn;
  if (!L->a_kmajor) {
    p.pack_a = prep ? 1 : 0;
    p.pad_a = pad ? E.pad_a : 0;
    p.pad_b = b_staged_trans ? E.pad_b_t : (pad ? E.pad_b : 0);
    p.smem_bytes = b_staged_trans ? E.smem_bytes_t : E.smem_bytes[pad ? 1 : 0];
  }
  L->entry = i;
  L->kern = kern;
  // Raster groups of 16 tile rows: a wave of 304 CTAs then spans about 16 x
  // 19 tiles, close to square, so it touches fewer A and B panels than with
  // groups of 8 (38 columns).  Measured on GB300 with 128 x 128 tiles, the
  // time unchanged: DRAM read 333 -> 284 MB at 4096^3, 3.30 -> 3.23 GB at
  // 8192^3 (32 rows: 499 MB and 4.72 GB).
  if (!(cfg && cfg->group_m)) L->group_m = 16;
  L->tiles_m = static_cast<int>(ceil_div(M, E.bm));
  L->tiles_n = static_cast<int>(ceil_div(N, E.bn));
  const int64_t tiles = static_cast<int64_t>(L->tiles_m) * L->tiles_n;
  if (tiles > INT32_MAX / 4) return MT_ERR_UNSUPPORTED;
  // Split-K: the tiles of the split part are cut along K into slices whose
  // partial tiles add up in a second kernel (see GemmArgs).  An explicit
  // split_k splits every tile; the automatic splits are below.
  const int64_t ktiles = ceil_div(K, E.bk);
  int64_t full = tiles, split = 1;
  if (cfg && cfg->split_k > 1) {
    full = 0;
    split = std::min<int64_t>(cfg->split_k, ktiles > 0 ? ktiles : 1);
  } else if (!(cfg && cfg->split_k == 1)) {
    // split_k = 1 turns both off.  Fewer tiles than SMs are cut into up to
    // 4 K slices of at least 512 (512 x 512 x 4096: 2.7x).  With K-major A,
    // a last wave under half full is cut into K slices (the CTAs of whole
    // tiles come first, so the slices make up the last wave; 4097 x 3001 x
    // 2053 and 65536 x 128 x 4096 1.04x, 2048 x 2048 x 8192 1.15x).
    const int64_t n_sm = std::max(sms, 1);
    if (tiles < n_sm) {
      int64_t sk = std::min<int64_t>(4, n_sm / std::max<int64_t>(tiles, 1));
      while (sk > 1 && (K / sk < 512 || (sk - 1) * ceil_div(ktiles, sk) >= ktiles)) --sk;
      if (sk > 1) {
        full = 0;
        split = sk;
      }
    } else if (L->a_kmajor) {
      // Four slices, even when the idle CTAs would only take two at once:
      // the slices then run as two short rounds that even out where the
      // whole tiles ended.  Measured on GB300 (against as many slices as fit
      // the idle CTAs): 4096^3 2052 -> 1984 us, 4097 x 3001 x 2053 854 ->
      // 848 us; 8192^3, 2048 x 2048 x 8192 and 65536 x 128 x 4096 unchanged
      // (three slices gained nothing at 4096^3, six less than four).
      split_tail(tiles, n_sm * E.min_blocks, ktiles, true, &full, &split, 4);
    }
  }
  if (split <= 1) {
    split = 1;
    full = tiles;
  }
  // Stream-K (schedule 2): the tiles past the last whole wave of resident
  // CTAs (all of them when there is less than one wave) are not cut into
  // equal K slices but spread evenly, K tile by K tile, over one wave of
  // units, each taking a contiguous run across tile boundaries; a second
  // kernel adds the pieces of the tiles no run covered whole.
  const int schedule = cfg ? cfg->schedule : 0;
  // Automatically, where 64 x 128 tiles with A staged K-major (the tile of
  // grids under six waves of 128 x 128 tiles) would cut a partial last wave
  // into K slices, they take stream-K instead: measured on GB300 against
  // the split tail, 4097 x 3001 x 2053 809.6 against 819.8 us, 65536 x 128 x
  // 4096 equal.  128 x 128 tiles keep the split tail (4096^3 equal, 8192^3
  // 0.2 % faster with it); plans the split tail leaves whole stay whole.
  const bool auto_streamk = schedule == 0 && L->a_kmajor && E.bm == 64 && E.bn == 128 &&
                            E.kslices == 1 && !(cfg && cfg->split_k > 0) && split > 1 &&
                            full > 0;
  if (schedule == 2 || auto_streamk) {
    if (E.kslices != 1 || (cfg && cfg->split_k > 1)) return MT_ERR_UNSUPPORTED;
    split = 1;
    full = tiles;
    if (!(cfg && cfg->split_k == 1) && ktiles > 0) {
      const int64_t slots = static_cast<int64_t>(std::max(sms, 1)) * E.min_blocks;
      const int64_t rem = tiles % slots;
      if (rem != 0) {
        full = tiles - rem;
        L->sk_iters = rem * ktiles;
        // Every unit takes at least two K tiles.
        L->sk_ctas = static_cast<int>(std::max<int64_t>(
            1, std::min<int64_t>(slots, L->sk_iters / 2)));
      }
    }
  }
  L->full_tiles = static_cast<int>(full);
  L->split = static_cast<int>(split);
  L->kt_per_slice = static_cast<int>(ceil_div(ktiles, split));
  p.split_k = L->split;
  p.stream_k = L->sk_ctas;
  p.grid = L->sk_ctas > 0 ? full + L->sk_ctas : full + (tiles - full) * split;
  if (!L->a_kmajor) {
    L->ldo_a = copy_pitch(K);
    L->ldo_b = copy_pitch(N);
    L->prep_b_offset = L->prep_a ? round256(M * L->ldo_a * 4) : 0;
  }
  L->partial_offset = L->prep_b_offset + (L->prep_b ? round256(K * L->ldo_b * 4) : 0);
  p.workspace_bytes = L->partial_offset + (L->sk_ctas > 0 ? 2 * int64_t(L->sk_ctas)
                                                          : (tiles - full) * split) *
                                             E.bm * E.bn * 4;
  // The budget check comes before anything is launched ("Part 18", section
  // "Shared-memory budget checks include stages and padding").
  if (p.smem_bytes > smem_limit) return MT_ERR_SMEM_BUDGET;
  return MT_OK;
}

// The fp32 variant of a call made without a configuration: MT_SGEMM_VARIANT
// = "ffma" (or unset or empty), "tf32x3" or "p18"; -1 for any other value.
int default_variant() {
  const char* v = std::getenv("MT_SGEMM_VARIANT");
  if (!v || !*v || std::strcmp(v, "ffma") == 0) return MT_VARIANT_FFMA;
  if (std::strcmp(v, "tf32x3") == 0) return MT_VARIANT_TF32X3;
  if (std::strcmp(v, "p18") == 0) return MT_VARIANT_P18;
  return -1;
}

mt_status plan_call(const Problem& P, const mt_config* cfg, int64_t smem_limit, int sms,
                    Launch* L, int dev = -1) {
  const int64_t M = P.M, N = P.N, K = P.K;
  mt_status st = check_dims(M, N, K);
  if (st != MT_OK) return st;
  st = check_lds(P);
  if (st != MT_OK) return st;
  const int variant = cfg ? cfg->variant : P.dtype ? MT_VARIANT_TC16 : default_variant();
  if (variant < 0) return MT_ERR_INVALID_ARG;  // MT_SGEMM_VARIANT names no variant
  if (cfg && (cfg->bm < 0 || cfg->bn < 0 || cfg->bk < 0 || cfg->stages < 0 ||
              cfg->no_pad < 0 || cfg->no_pad > 1 || cfg->split_k < 0 || cfg->fma < 0 ||
              cfg->fma > 2 || cfg->fault_inject < 0 || cfg->fault_inject > 1 || cfg->wm < 0 ||
              cfg->wn < 0 || cfg->tm < 0 || cfg->tn < 0 || cfg->pack_a < 0 ||
              cfg->pack_a > 5 || cfg->group_m < 0 || cfg->schedule < 0 ||
              cfg->schedule > 2))
    return MT_ERR_INVALID_ARG;
  // The one-warp kernel has one schedule: a CTA per tile.
  if (cfg && cfg->schedule && !P.dtype && variant == MT_VARIANT_P18) return MT_ERR_UNSUPPORTED;
  if (P.dtype)
    return plan_f16(P, cfg, smem_limit, sms, dev >= 0 ? mt::f16tc_pair_max_clusters(dev) : 0,
                    L);
  if (variant == MT_VARIANT_TC16) return MT_ERR_UNSUPPORTED;  // 16-bit inputs only
  if (cfg && (cfg->wm || cfg->wn || cfg->tm || cfg->tn) && variant != MT_VARIANT_FFMA)
    return MT_ERR_UNSUPPORTED;
  if (cfg && cfg->pack_a && variant != MT_VARIANT_TF32X3 && variant != MT_VARIANT_FFMA)
    return MT_ERR_UNSUPPORTED;
  if (cfg && cfg->pack_a >= 3 && variant != MT_VARIANT_FFMA) return MT_ERR_UNSUPPORTED;
  if (cfg && cfg->fault_inject && variant != MT_VARIANT_TF32X3) return MT_ERR_UNSUPPORTED;
  // 3xTF32 splits only its tail by itself (split_k = 1 turns that off).
  if (cfg && cfg->split_k > 1 && variant != MT_VARIANT_FFMA) return MT_ERR_UNSUPPORTED;
  const bool pad = !(cfg && cfg->no_pad);
  const bool trans = P.trans_a || P.trans_b;
  L->fault_inject = cfg ? cfg->fault_inject : 0;
  if (cfg && cfg->group_m) L->group_m = cfg->group_m;
  mt_plan& p = L->plan;
  std::memset(&p, 0, sizeof(p));
  p.variant = variant;
  p.split_k = 1;
  // 16-byte staging of both operands and 16-byte stores of C: untransposed
  // operands whose rows are whole float4s (K, N and every leading dimension
  // multiples of 4) from 16-byte aligned bases.
  p.vec_ab = !trans && K % 4 == 0 && N % 4 == 0 && P.lda % 4 == 0 && P.ldb % 4 == 0 &&
             P.ldc % 4 == 0 && aligned16(P.A) && aligned16(P.B) && aligned16(P.C);
  p.vec_c = p.vec_ab;
  L->pad = pad;

  if (variant == MT_VARIANT_P18) {
    if (cfg && ((cfg->bm && cfg->bm != 4) || (cfg->bn && cfg->bn != 8) ||
                (cfg->bk && cfg->bk != 16) || (cfg->stages && cfg->stages > 2) || cfg->fma))
      return MT_ERR_UNSUPPORTED;
    // Two stages (Version 18's ping-pong) unless one is asked for.
    p.bm = 4; p.bn = 8; p.bk = 16; p.stages = cfg && cfg->stages == 1 ? 1 : 2; p.threads = 32;
    p.pad_a = mt::p18_pad_a(pad);
    p.pad_b = 0;
    p.vec_ab = 0; p.vec_c = 0;
    p.smem_bytes = 0;  // static shared memory only
    L->tiles_m = static_cast<int>(ceil_div(M, 4));
    L->tiles_n = static_cast<int>(ceil_div(N, 8));
    p.grid = static_cast<int64_t>(L->tiles_m) * L->tiles_n;
    if (p.grid > INT32_MAX) return MT_ERR_UNSUPPORTED;
    return MT_OK;
  }
  if (variant == MT_VARIANT_TF32X3) return plan_tf32x3(P, cfg, smem_limit, sms, dev, L);
  if (variant != MT_VARIANT_FFMA) return MT_ERR_INVALID_ARG;
  return plan_ffma(P, cfg, smem_limit, sms, pad, trans, L);
}

mt_status set_smem_attr(int dev, const Launch& L) {
  if (L.entry < 0 || L.plan.smem_bytes <= 48 * 1024) return MT_OK;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_attr_done[dev].count(L.kern)) return MT_OK;
  if (cudaFuncSetAttribute(L.kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(L.plan.smem_bytes)) != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_LAUNCH;
  }
  g_attr_done[dev].insert(L.kern);
  return MT_OK;
}

mt_status pool_for(int dev, cudaMemPool_t* pool) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_pools[dev]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p = nullptr;
    if (cudaMemPoolCreate(&p, &props) != cudaSuccess) {
      cudaGetLastError();
      return MT_ERR_CUDA;
    }
    // Keep freed blocks for the next call instead of returning them to the
    // driver at every synchronisation.
    uint64_t keep = UINT64_MAX;
    cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
    g_pools[dev] = p;
  }
  *pool = g_pools[dev];
  return MT_OK;
}

// [device][configuration]: shared-memory attribute of the 3xTF32 kernel applied.
std::atomic<uint8_t> g_tf32x3_ready[kMaxDevices][16];

// [split_a][bk == 32][128 x 256, 128 x 128, 128 x 64, pair 256 x 256]
int tf32x3_cfg_index(int bm, int bk, int bn, int split_a) {
  return (split_a ? 8 : 0) + (bk == 32 ? 4 : 0) +
         (bm == 256 ? 3 : bn == 256 ? 0 : bn == 128 ? 1 : 2);
}

mt_status prepare_tf32x3(int dev, int bm, int bk, int bn, int split_a) {
  std::atomic<uint8_t>& ready = g_tf32x3_ready[dev][tf32x3_cfg_index(bm, bk, bn, split_a)];
  if (!ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!ready.load(std::memory_order_relaxed)) {
      if (mt::tf32x3_prepare(dev, bm, bk, bn, split_a) != cudaSuccess) {
        cudaGetLastError();
        return MT_ERR_LAUNCH;
      }
      ready.store(1, std::memory_order_release);
    }
  }
  return MT_OK;
}

mt::GemmArgs make_args(const Problem& P, const Launch& L) {
  mt::GemmArgs a{};
  a.A = P.dtype ? nullptr : static_cast<const float*>(P.A);
  a.B = P.dtype ? nullptr : static_cast<const float*>(P.B);
  a.C = P.C;
  a.M = static_cast<int>(P.M);
  a.N = static_cast<int>(P.N);
  a.K = static_cast<int>(P.K);
  a.tiles_m = L.tiles_m;
  a.tiles_n = L.tiles_n;
  a.group_m = L.group_m;
  a.lda = P.lda;
  a.ldb = P.ldb;
  a.ldc = P.ldc;
  a.alpha = P.alpha;
  a.beta = P.beta;
  a.bias = P.bias;
  a.trans_a = P.trans_a;
  a.trans_b = P.trans_b;
  a.full_tiles = L.full_tiles;
  a.split = L.split;
  a.kt_per_slice = L.kt_per_slice;
  a.sk_ctas = L.sk_ctas;
  a.sk_iters = L.sk_iters;
  a.partial = nullptr;
  a.a_extent = P.trans_a ? mt::view_extent(P.K, P.M, P.lda) : mt::view_extent(P.M, P.K, P.lda);
  a.b_extent = P.trans_b ? mt::view_extent(P.N, P.K, P.ldb) : mt::view_extent(P.K, P.N, P.ldb);
  a.c_extent = mt::view_extent(P.M, P.N, P.ldc);
  a.partial_extent = 0;
  a.bounds = bounds_record();
#if MT_BOUNDS_CHECK
  // Test hook of the checked build only: C is declared one element shorter
  // than it is, so the store of its last element counts as outside and is
  // skipped (no access leaves the real buffer).
  if (std::getenv("MT_CHECKED_SHRINK_C_EXTENT")) a.c_extent -= 1;
#endif
  return a;
}

mt_status run_tf32x3(int dev, const mt::GemmArgs& args, const Launch& L, cudaStream_t stream) {
  mt_status st0 = prepare_tf32x3(dev, L.plan.bm, L.plan.bk, L.plan.bn, L.split_a);
  if (st0 != MT_OK) return st0;
  cudaMemPool_t pool = nullptr;
  mt_status st = pool_for(dev, &pool);
  if (st != MT_OK) return st;
  void* ws = nullptr;
  if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(L.plan.workspace_bytes), pool, stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_CUDA;
  }
  const cudaError_t e =
      mt::launch_tf32x3(args, ws, L.vec_a, L.vec_b, L.plan.vec_c != 0, L.plan.bm, L.plan.bk,
                        L.plan.bn, L.split_a, L.max_ctas, L.fault_inject, stream);
  cudaFreeAsync(ws, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_LAUNCH;
  }
  return MT_OK;
}

// [device][128 x 256, 128 x 128, pair]: shared-memory attribute of the
// 16-bit kernels applied.
std::atomic<uint8_t> g_f16_ready[kMaxDevices][3];

mt_status run_f16(int dev, const Problem& P, const mt::GemmArgs& args, const Launch& L,
                  cudaStream_t stream) {
  if (!mt::f16tc_encoder_available()) return MT_ERR_CUDA;
  std::atomic<uint8_t>& ready =
      g_f16_ready[dev][L.plan.bm == 256 ? 2 : L.plan.bn == 128 ? 1 : 0];
  if (!ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!ready.load(std::memory_order_relaxed)) {
      if (mt::f16tc_prepare(L.plan.bm, L.plan.bn) != cudaSuccess) {
        cudaGetLastError();
        return MT_ERR_LAUNCH;
      }
      ready.store(1, std::memory_order_release);
    }
  }
  void* ws = nullptr;
  if (L.plan.workspace_bytes > 0) {
    cudaMemPool_t pool = nullptr;
    mt_status st = pool_for(dev, &pool);
    if (st != MT_OK) return st;
    if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(L.plan.workspace_bytes), pool,
                                stream) != cudaSuccess) {
      cudaGetLastError();
      return MT_ERR_CUDA;
    }
  }
  const cudaError_t e =
      mt::launch_f16tc(args, mt::F16Operands{P.A, P.B, P.dtype}, ws, L.plan.vec_c != 0,
                       L.plan.bm, L.plan.bn, L.max_ctas, L.fault_inject, stream);
  if (ws) cudaFreeAsync(ws, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_LAUNCH;
  }
  return MT_OK;
}

mt_status run(const Problem& P, cudaStream_t stream, const mt_config* cfg) {
  mt_status st = check_problem(P);
  if (st != MT_OK) return st;
  if (P.M == 0 || P.N == 0) return MT_OK;
  int dev = 0;
  DeviceInfo info;
  st = current_device(&dev, &info);
  if (st != MT_OK) return st;
  Launch L;
  st = plan_call(P, cfg, info.smem_optin, info.sms, &L, dev);
  if (st != MT_OK) return st;
  if (!reads_ab(P)) {
    // No product to form (K == 0: the accumulator's zeros; alpha == 0):
    // C = beta * C (+ bias), A and B untouched.
    if (mt::launch_scale_c(P.C, static_cast<int>(P.M), static_cast<int>(P.N), P.ldc, P.beta,
                           P.bias, stream, bounds_record()) != cudaSuccess) {
      cudaGetLastError();
      return MT_ERR_LAUNCH;
    }
    return MT_OK;
  }
  mt::GemmArgs args = make_args(P, L);
  if (P.dtype) return run_f16(dev, P, args, L, stream);
  if (L.plan.variant == MT_VARIANT_TF32X3) return run_tf32x3(dev, args, L, stream);
  if (L.plan.variant == MT_VARIANT_P18) {
    if (mt::launch_p18(args, L.pad, L.plan.stages, stream) != cudaSuccess) return MT_ERR_LAUNCH;
    return MT_OK;
  }
  st = set_smem_attr(dev, L);
  if (st != MT_OK) return st;
  void* ws = nullptr;
  cudaMemPool_t pool = nullptr;
  bool ok = true;
  if (L.plan.workspace_bytes > 0) {
    st = pool_for(dev, &pool);
    if (st != MT_OK) return st;
    if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(L.plan.workspace_bytes), pool,
                                stream) != cudaSuccess) {
      cudaGetLastError();
      return MT_ERR_CUDA;
    }
    char* base = static_cast<char*>(ws);
    if (L.split > 1 || L.sk_ctas > 0) {
      args.partial = reinterpret_cast<float*>(base + L.partial_offset);
      args.partial_extent = (L.plan.workspace_bytes - L.partial_offset) / 4;
    }
    // Operands copied into the layout the 16-byte staging reads.
    if (L.prep_a) {
      float* a = reinterpret_cast<float*>(base);
      ok = mt::launch_prep_operand(static_cast<const float*>(P.A), P.lda, P.trans_a != 0, a,
                                   L.ldo_a, static_cast<int>(P.M), static_cast<int>(P.K),
                                   stream, args.bounds) == cudaSuccess;
      args.A = a;
      args.lda = L.ldo_a;
      args.trans_a = 0;
      args.a_extent = P.M * L.ldo_a;
    }
    if (L.prep_a_kmajor) {
      // A^T (K x M) into scratch: a transposing copy of A stored M x K, a
      // plain one of A stored K x M.
      float* a = reinterpret_cast<float*>(base);
      ok = mt::launch_prep_operand(static_cast<const float*>(P.A), P.lda, P.trans_a == 0, a,
                                   L.ldo_a, static_cast<int>(P.K), static_cast<int>(P.M),
                                   stream, args.bounds) == cudaSuccess;
      args.A = a;
      args.lda = L.ldo_a;
      args.trans_a = 1;
      args.a_extent = P.K * L.ldo_a;
    }
    if (ok && L.prep_b) {
      float* b = reinterpret_cast<float*>(base + L.prep_b_offset);
      ok = mt::launch_prep_operand(static_cast<const float*>(P.B), P.ldb, P.trans_b != 0, b,
                                   L.ldo_b, static_cast<int>(P.K), static_cast<int>(P.N),
                                   stream, args.bounds) == cudaSuccess;
      args.B = b;
      args.ldb = L.ldo_b;
      args.trans_b = 0;
      args.b_extent = P.K * L.ldo_b;
    }
  }
  void* params[] = {&args};
  // After an operand copy the GEMM is launched as its programmatic
  // dependent: its CTAs are scheduled as the copy's CTAs retire and wait
  // inside (griddepcontrol.wait) for the copy to complete, so the launch
  // latency overlaps the copy.
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(static_cast<unsigned>(L.plan.grid));
  lc.blockDim = dim3(static_cast<unsigned>(L.plan.threads));
  lc.dynamicSmemBytes = static_cast<size_t>(L.plan.smem_bytes);
  lc.stream = stream;
  lc.attrs = attr;
  lc.numAttrs = (L.prep_a || L.prep_a_kmajor || L.prep_b) ? 1 : 0;
  ok = ok && cudaLaunchKernelExC(&lc, L.kern, params) == cudaSuccess;
  // The split tail's reduce or the stream-K fix-up, when the plan has one.
  ok = ok && mt::launch_second_pass(args, args.partial, L.plan.bm, L.plan.bn,
                                    static_cast<int>(ceil_div(P.K, L.plan.bk)),
                                    L.plan.vec_c != 0, stream) == cudaSuccess;
  if (ws) cudaFreeAsync(ws, stream);
  if (!ok) {
    cudaGetLastError();
    return MT_ERR_LAUNCH;
  }
  return MT_OK;
}

// Copy streams of the host-buffer entry point, per device (created once,
// non-blocking).  Concurrent calls share them: their copies serialise, the
// events keep each call's order.
struct HostStreams {
  cudaStream_t h2d = nullptr, d2h = nullptr;
};
HostStreams g_host_streams[kMaxDevices];

mt_status host_streams(int dev, HostStreams* out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  HostStreams& h = g_host_streams[dev];
  if (!h.h2d) {
    cudaStream_t a = nullptr, b = nullptr;
    if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
      if (a) cudaStreamDestroy(a);
      cudaGetLastError();
      return MT_ERR_CUDA;
    }
    h.h2d = a;
    h.d2h = b;
  }
  *out = h;
  return MT_OK;
}

// Row blocks of the host entry point's copy/compute pipeline.  A block must
// still fill the GPU one and a half times over (at least 1.5 x 304 tiles of
// 128 x 128), and its rows start on a multiple of 256, so its A and C rows
// stay 16-byte aligned; at most kMaxHostBlocks blocks.  One block (no
// pipeline) when M is too small for two such blocks.  Measured on GB300:
// 4096^3 as two blocks 2.75 ms against 3.08 as one (three-wave minimum).
constexpr int kMaxHostBlocks = 4;

int64_t host_block_rows(int64_t M, int64_t N, int64_t K) {
  (void)K;
  const int64_t tile_cols = std::max<int64_t>(1, ceil_div(N, 128));
  const int64_t min_rows = ceil_div(ceil_div(3 * 304 / 2, tile_cols) * 128, 256) * 256;
  const int64_t rows = std::max(min_rows, ceil_div(ceil_div(M, kMaxHostBlocks), 256) * 256);
  return rows * 2 <= M ? rows : M;
}

// The host-buffer pipeline behind mt_sgemm_host (sync) and
// mt_sgemm_host_async.  A and B's device copies are allocated on the
// copy-in stream, so a call's copies in do not queue behind the products of
// an earlier call on `stream`; C's copy comes from `stream` and goes back to
// the pool from the copy-out stream after its last copy out.  `stream` waits
// for the last copy out, so the call is complete once `stream` is.
mt_status host_pipeline(const float* A, const float* B, float* C, int64_t M, int64_t N,
                        int64_t K, cudaStream_t stream, const mt_config* cfg, bool sync) {
  mt_status st0 = check_dims(M, N, K);
  if (st0 != MT_OK) return st0;
  if (M == 0 || N == 0) return MT_OK;
  if (!C || (K > 0 && (!A || !B))) return MT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceInfo info;
  mt_status st = current_device(&dev, &info);
  if (st != MT_OK) return st;
  cudaMemPool_t pool = nullptr;
  st = pool_for(dev, &pool);
  if (st != MT_OK) return st;
  HostStreams hs;
  st = host_streams(dev, &hs);
  if (st != MT_OK) return st;
  const size_t a_bytes = static_cast<size_t>(M * K) * 4, b_bytes = static_cast<size_t>(K * N) * 4,
               c_bytes = static_cast<size_t>(M * N) * 4;
  float *dA = nullptr, *dB = nullptr, *dC = nullptr;
  bool ok = true;
  const int64_t rows = host_block_rows(M, N, K);
  const int64_t blocks = ceil_div(M, rows);
  cudaEvent_t ev[2 * kMaxHostBlocks + 3] = {};
  const int nev = static_cast<int>(2 * blocks + 3);
  for (int i = 0; i < nev && ok; ++i)
    ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
  cudaEvent_t ev_calloc = ev[0], ev_done = ev[1], ev_in_done = ev[2];
  // 256-byte aligned pool blocks keep the 16-byte staging path available.
  if (ok && a_bytes)
    ok = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dA), a_bytes, pool, hs.h2d) ==
         cudaSuccess;
  if (ok && b_bytes)
    ok = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dB), b_bytes, pool, hs.h2d) ==
         cudaSuccess;
  if (ok)
    ok = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dC), c_bytes, pool, stream) ==
         cudaSuccess;
  // C's buffer was allocated on the caller's stream; the copy-out stream
  // writes from it.
  if (ok) ok = cudaEventRecord(ev_calloc, stream) == cudaSuccess &&
               cudaStreamWaitEvent(hs.d2h, ev_calloc, 0) == cudaSuccess;
  if (ok && b_bytes)
    ok = cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, hs.h2d) == cudaSuccess;
  // Row blocks of A and C: block i's copy in, product and copy out run on
  // the copy-in stream, the caller's stream and the copy-out stream, so the
  // copies of neighbouring blocks overlap the product of this one.
  for (int64_t i = 0; i < blocks && ok && st == MT_OK; ++i) {
    const int64_t r0 = i * rows, nr = std::min(rows, M - r0);
    cudaEvent_t ev_in = ev[3 + 2 * i], ev_out = ev[4 + 2 * i];
    // Block i of A (and, before block 0, all of B) is on the device ...
    if (K > 0)
      ok = cudaMemcpyAsync(dA + r0 * K, A + r0 * K, static_cast<size_t>(nr * K) * 4,
                           cudaMemcpyHostToDevice, hs.h2d) == cudaSuccess;
    ok = ok && cudaEventRecord(ev_in, hs.h2d) == cudaSuccess &&
         cudaStreamWaitEvent(stream, ev_in, 0) == cudaSuccess;
    if (!ok) break;
    // ... its product runs on the caller's stream ...
    st = run(packed_problem(K > 0 ? dA + r0 * K : nullptr, dB, dC + r0 * N, nr, N, K), stream,
             cfg);
    if (st != MT_OK) break;
    // ... and its rows of C go back while the next block computes.
    ok = cudaEventRecord(ev_out, stream) == cudaSuccess &&
         cudaStreamWaitEvent(hs.d2h, ev_out, 0) == cudaSuccess &&
         cudaMemcpyAsync(C + r0 * N, dC + r0 * N, static_cast<size_t>(nr * N) * 4,
                         cudaMemcpyDeviceToHost, hs.d2h) == cudaSuccess;
  }
  // A and B go back to the pool after the last product (the copies in all
  // precede it, and a failed loop may have left some in flight: the caller's
  // stream waits for the copy-in stream first); C after the last copy out.
  // The caller's stream then waits for the copy-out stream, so the whole
  // call is complete once it is.
  bool drained = ev_in_done && cudaEventRecord(ev_in_done, hs.h2d) == cudaSuccess &&
                 cudaStreamWaitEvent(stream, ev_in_done, 0) == cudaSuccess;
  if (!drained) cudaStreamSynchronize(hs.h2d);
  if (dA) cudaFreeAsync(dA, stream);
  if (dB) cudaFreeAsync(dB, stream);
  if (dC) {
    // The copy-out stream frees C once its copies (and, through ev_calloc,
    // the allocation) are ordered before.
    if (ev_calloc && cudaEventRecord(ev_calloc, stream) == cudaSuccess &&
        cudaStreamWaitEvent(hs.d2h, ev_calloc, 0) == cudaSuccess) {
      cudaFreeAsync(dC, hs.d2h);
    } else {
      cudaStreamSynchronize(hs.d2h);
      cudaFreeAsync(dC, stream);
    }
  }
  drained = ev_done && cudaEventRecord(ev_done, hs.d2h) == cudaSuccess &&
            cudaStreamWaitEvent(stream, ev_done, 0) == cudaSuccess;
  if (!drained) cudaStreamSynchronize(hs.d2h);
  // Events may be destroyed while work still waits on them (their release
  // is deferred until they complete).
  for (int i = 0; i < nev; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  const bool synced = !sync || cudaStreamSynchronize(stream) == cudaSuccess;
  if (!ok || !synced) {
    cudaGetLastError();
    return st != MT_OK ? st : MT_ERR_CUDA;
  }
  return st;
}

}  // namespace

extern "C" {

mt_status mt_sgemm(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
                   cudaStream_t stream) {
  return run(packed_problem(A, B, C, M, N, K), stream, nullptr);
}

mt_status mt_sgemm_ex(const float* A, const float* B, float* C, int64_t M, int64_t N,
                      int64_t K, cudaStream_t stream, const mt_config* cfg) {
  return run(packed_problem(A, B, C, M, N, K), stream, cfg);
}

mt_status mt_sgemm_general(int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                           float alpha, const float* A, int64_t lda, const float* B,
                           int64_t ldb, float beta, float* C, int64_t ldc, cudaStream_t stream,
                           const mt_config* cfg) {
  return run(Problem{A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, trans_a, trans_b}, stream,
             cfg);
}

mt_status mt_sgemm_general_bias(int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                float alpha, const float* A, int64_t lda, const float* B,
                                int64_t ldb, float beta, const float* bias, float* C,
                                int64_t ldc, cudaStream_t stream, const mt_config* cfg) {
  Problem P{A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, trans_a, trans_b};
  P.bias = bias;
  return run(P, stream, cfg);
}

mt_status mt_sgemm_host(const float* A, const float* B, float* C, int64_t M, int64_t N,
                        int64_t K, cudaStream_t stream, const mt_config* cfg) {
  return host_pipeline(A, B, C, M, N, K, stream, cfg, true);
}

mt_status mt_sgemm_host_async(const float* A, const float* B, float* C, int64_t M, int64_t N,
                              int64_t K, cudaStream_t stream, const mt_config* cfg) {
  return host_pipeline(A, B, C, M, N, K, stream, cfg, false);
}

mt_status mt_sgemm_tf32x3_noalloc(const float* A, const float* B, float* C, int64_t M,
                                  int64_t N, int64_t K, cudaStream_t stream) {
  static_assert(MT_NOALLOC_SCRATCH_BYTES == mt::kNoAllocScratchBytes, "scratch size");
  const Problem P = packed_problem(A, B, C, M, N, K);
  mt_status st = check_problem(P);
  if (st != MT_OK) return st;
  if (M == 0 || N == 0) return MT_OK;
  int dev = 0;
  DeviceInfo info;
  st = current_device(&dev, &info);
  if (st != MT_OK) return st;
  mt_config cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.variant = MT_VARIANT_TF32X3;
  Launch L;
  st = plan_call(P, &cfg, info.smem_optin, info.sms, &L, dev);
  if (st != MT_OK) return st;
  if (K == 0) {
    // Empty reduction: zeros, written without any scratch.
    if (cudaMemsetAsync(C, 0, static_cast<size_t>(M * N) * 4, stream) != cudaSuccess) {
      cudaGetLastError();
      return MT_ERR_LAUNCH;
    }
    return MT_OK;
  }
  if (L.plan.workspace_bytes > MT_NOALLOC_SCRATCH_BYTES) return MT_ERR_SCRATCH_LIMIT;
  st = prepare_tf32x3(dev, L.plan.bm, L.plan.bk, L.plan.bn, L.split_a);
  if (st != MT_OK) return st;
  void* scratch = nullptr;
  if (mt::tf32x3_noalloc_scratch(dev, &scratch) != cudaSuccess || !scratch) {
    cudaGetLastError();
    return MT_ERR_CUDA;
  }
  const mt::GemmArgs args = make_args(P, L);
  if (mt::launch_tf32x3(args, scratch, L.vec_a, L.vec_b, L.plan.vec_c != 0, L.plan.bm,
                        L.plan.bk, L.plan.bn, L.split_a, L.max_ctas, 0, stream) != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_LAUNCH;
  }
  return MT_OK;
}

mt_status mt_sgemm_plan(const float* A, const float* B, const float* C, int64_t M, int64_t N,
                        int64_t K, const mt_config* cfg, int64_t smem_limit_bytes,
                        mt_plan* out) {
  if (!out) return MT_ERR_INVALID_ARG;
  int sms = 0;
  if (smem_limit_bytes <= 0) {
    int dev = 0;
    DeviceInfo info;
    mt_status st = current_device(&dev, &info);
    if (st != MT_OK) return st;
    smem_limit_bytes = info.smem_optin;
    sms = info.sms;
  } else {
    int dev = 0;
    DeviceInfo info;
    // The SM count only steers the automatic tile choice; without a device
    // the choice assumes a full GB300 (152 SMs).
    sms = current_device(&dev, &info) == MT_OK ? info.sms : 152;
  }
  Launch L;
  mt_status st = plan_call(packed_problem(A, B, const_cast<float*>(C), M, N, K), cfg,
                           smem_limit_bytes, sms, &L);
  *out = L.plan;
  return st;
}

mt_status mt_gemm_mixed(int dtype, const void* A, const void* B, float* C, int64_t M, int64_t N,
                        int64_t K, cudaStream_t stream) {
  if (dtype != MT_DTYPE_F16 && dtype != MT_DTYPE_BF16) return MT_ERR_INVALID_ARG;
  return run(packed_problem(A, B, C, M, N, K, dtype), stream, nullptr);
}

mt_status mt_gemm_mixed_general(int dtype, int trans_a, int trans_b, int64_t M, int64_t N,
                                int64_t K, float alpha, const void* A, int64_t lda,
                                const void* B, int64_t ldb, float beta, float* C, int64_t ldc,
                                cudaStream_t stream, const mt_config* cfg) {
  if (dtype != MT_DTYPE_F16 && dtype != MT_DTYPE_BF16) return MT_ERR_INVALID_ARG;
  return run(Problem{A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, trans_a, trans_b, dtype},
             stream, cfg);
}

mt_status mt_gemm_mixed_general_bias(int dtype, int trans_a, int trans_b, int64_t M, int64_t N,
                                     int64_t K, float alpha, const void* A, int64_t lda,
                                     const void* B, int64_t ldb, float beta, const float* bias,
                                     float* C, int64_t ldc, cudaStream_t stream,
                                     const mt_config* cfg) {
  if (dtype != MT_DTYPE_F16 && dtype != MT_DTYPE_BF16) return MT_ERR_INVALID_ARG;
  Problem P{A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, trans_a, trans_b, dtype};
  P.bias = bias;
  return run(P, stream, cfg);
}

// Plan of a general-form call of either element type (dtype 0: fp32).
mt_status plan_general(int dtype, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                       const void* A, int64_t lda, const void* B, int64_t ldb, const float* C,
                       int64_t ldc, const mt_config* cfg, int64_t smem_limit_bytes,
                       mt_plan* out) {
  if (!out) return MT_ERR_INVALID_ARG;
  const Problem P{A, B, const_cast<float*>(C), M, N, K, lda, ldb, ldc, 1.0f, 0.0f,
                  trans_a, trans_b, dtype};
  if (trans_a < 0 || trans_a > 1 || trans_b < 0 || trans_b > 1) return MT_ERR_INVALID_ARG;
  int sms = 0;
  int dev = 0;
  DeviceInfo info;
  if (smem_limit_bytes <= 0) {
    mt_status st = current_device(&dev, &info);
    if (st != MT_OK) return st;
    smem_limit_bytes = info.smem_optin;
    sms = info.sms;
  } else {
    sms = current_device(&dev, &info) == MT_OK ? info.sms : 152;
  }
  Launch L;
  mt_status st =
      plan_call(P, cfg, smem_limit_bytes, sms, &L, current_device(&dev, &info) == MT_OK ? dev : -1);
  *out = L.plan;
  return st;
}

mt_status mt_gemm_mixed_plan(int dtype, int trans_a, int trans_b, int64_t M, int64_t N,
                             int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                             const float* C, int64_t ldc, const mt_config* cfg,
                             int64_t smem_limit_bytes, mt_plan* out) {
  if (dtype != MT_DTYPE_F16 && dtype != MT_DTYPE_BF16) return MT_ERR_INVALID_ARG;
  return plan_general(dtype, trans_a, trans_b, M, N, K, A, lda, B, ldb, C, ldc, cfg,
                      smem_limit_bytes, out);
}

mt_status mt_sgemm_general_plan(int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                const float* A, int64_t lda, const float* B, int64_t ldb,
                                const float* C, int64_t ldc, const mt_config* cfg,
                                int64_t smem_limit_bytes, mt_plan* out) {
  return plan_general(0, trans_a, trans_b, M, N, K, A, lda, B, ldb, C, ldc, cfg,
                      smem_limit_bytes, out);
}

int mt_smem_row_padding(int columns, int simultaneous_rows) {
  if (columns <= 0 || simultaneous_rows <= 0) return -1;
  return mt::row_padding_rule(columns, simultaneous_rows);
}

int mt_smem_vector_row_padding(int columns, int simultaneous_rows) {
  if (columns <= 0 || columns % 4 != 0 || simultaneous_rows <= 0) return -1;
  return mt::vector_row_padding_rule(columns, simultaneous_rows);
}

mt_status mt_smem_layout_make(int rows, int columns, int row_padding, int stage_count,
                              mt_smem_layout* out) {
  if (!out || rows <= 0 || columns <= 0 || row_padding < 0 || stage_count <= 0)
    return MT_ERR_INVALID_ARG;
  const int64_t size = static_cast<int64_t>(stage_count) * rows * (columns + row_padding);
  if (size > INT32_MAX / 4) return MT_ERR_INVALID_ARG;
  const mt::SmemLayout L{rows, columns, row_padding, stage_count};
  out->rows = rows;
  out->columns = columns;
  out->row_padding = row_padding;
  out->stage_count = stage_count;
  out->row_stride = L.row_stride();
  out->stage_size = L.stage_size();
  out->size = L.size();
  out->nbytes = L.nbytes();
  return MT_OK;
}

int64_t mt_smem_layout_offset(const mt_smem_layout* layout, int stage, int row, int column) {
  if (!layout || stage < 0 || stage >= layout->stage_count || row < 0 || row >= layout->rows ||
      column < 0 || column >= layout->columns)
    return -1;
  const mt::SmemLayout L{layout->rows, layout->columns, layout->row_padding,
                         layout->stage_count};
  return L.offset(stage, row, column);
}

static_assert(MT_SITE_A_LOAD == mt::SITE_A_LOAD && MT_SITE_B_LOAD == mt::SITE_B_LOAD &&
                  MT_SITE_A_SMEM == mt::SITE_A_SMEM && MT_SITE_B_SMEM == mt::SITE_B_SMEM &&
                  MT_SITE_FRAG == mt::SITE_FRAG && MT_SITE_C_STORE == mt::SITE_C_STORE &&
                  MT_SITE_PARTIAL == mt::SITE_PARTIAL && MT_SITE_BIAS == mt::SITE_BIAS &&
                  MT_SITE_SLICE_SUM == mt::SITE_SLICE_SUM &&
                  MT_SITE_PREP_SRC == mt::SITE_PREP_SRC &&
                  MT_SITE_PREP_DST == mt::SITE_PREP_DST && MT_SITE_P18 == mt::SITE_P18,
              "site numbers of the header and the kernels");

mt_status mt_bounds_status(int64_t* count, int* site, int64_t* offset, int64_t* extent) {
#if MT_BOUNDS_CHECK
  int dev = 0;
  DeviceInfo info;
  mt_status st = current_device(&dev, &info);
  if (st != MT_OK) return st;
  if (!bounds_record()) return MT_ERR_CUDA;
  mt::BoundsRecord r{};
  const mt::BoundsRecord zero{};
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(&r, g_bounds, sizeof(r)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_bounds, &zero, sizeof(zero)) != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_CUDA;
  }
  if (count) *count = r.count;
  if (site) *site = r.site;
  if (offset) *offset = r.offset;
  if (extent) *extent = r.extent;
  return MT_OK;
#else
  (void)count;
  (void)site;
  (void)offset;
  (void)extent;
  return MT_ERR_UNSUPPORTED;  // the normal build checks nothing
#endif
}

mt_status mt_check_device_status(cudaStream_t stream) {
  int dev = -1;
  DeviceInfo info;
  if (current_device(&dev, &info) != MT_OK) return MT_ERR_NO_DEVICE;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_CUDA;
  }
  unsigned int flags = 0, flags16 = 0;
  if (mt::tf32x3_read_and_clear_status(&flags) != cudaSuccess ||
      mt::f16tc_read_and_clear_status(&flags16) != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_CUDA;
  }
  flags |= flags16;
  return flags ? MT_ERR_TIMEOUT : MT_OK;
}

mt_status mt_device_status(cudaStream_t stream) { return mt_check_device_status(stream); }

const char* mt_status_string(mt_status status) {
  switch (status) {
    case MT_OK: return "ok";
    case MT_ERR_INVALID_ARG: return "invalid argument";
    case MT_ERR_ALIAS: return "output overlaps an input";
    case MT_ERR_NO_DEVICE: return "no usable CUDA device";
    case MT_ERR_UNSUPPORTED: return "configuration not built into the library";
    case MT_ERR_SMEM_BUDGET: return "shared-memory budget exceeded";
    case MT_ERR_LAUNCH: return "kernel launch failed";
    case MT_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case MT_ERR_CUDA: return "CUDA runtime call failed";
    case MT_ERR_SCRATCH_LIMIT:
      return "problem exceeds the static scratch of the allocation-free entry point";
  }
  return "unknown status";
}

int mt_version(void) { return 100; }

}  // extern "C"
