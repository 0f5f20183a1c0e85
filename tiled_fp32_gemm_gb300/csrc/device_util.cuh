// Small device helpers shared by the kernels: cp.async staging with zero
// fill, and the grouped tile raster.
#pragma once

#include <cstdint>

#include "kernels.h"

// Checked builds: -DMT_BOUNDS_CHECK=1 (the library built as
// libmtsgemm_checked.so).  Normal builds compile every check away.
#ifndef MT_BOUNDS_CHECK
#define MT_BOUNDS_CHECK 0
#endif

namespace mt {

// True when elements [offset, offset + width) lie inside [0, extent).  In a
// checked build an access outside is counted in `rec` (the first one's site,
// offset and extent kept) and the caller skips it; normal builds always
// return true without looking.
__device__ __forceinline__ bool bounds_ok(BoundsRecord* rec, int site, int64_t offset,
                                          int width, int64_t extent) {
#if MT_BOUNDS_CHECK
  if (offset >= 0 && offset + width <= extent) return true;
  if (rec && atomicAdd(&rec->count, 1u) == 0u) {
    rec->site = site;
    rec->offset = offset;
    rec->extent = extent;
  }
  return false;
#else
  (void)rec;
  (void)site;
  (void)offset;
  (void)width;
  (void)extent;
  return true;
#endif
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global->shared copy.  src_bytes is 16 (copy) or 0
// (write 16 zero bytes, read nothing): the masked zero fill of an
// out-of-bounds chunk.  `src` must be a valid address either way.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src,
                                            uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}

// 4-byte asynchronous copy, same zero-fill convention (src_bytes 4 or 0).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src,
                                           uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Grouped raster: CTAs walk GROUP_M tile rows down before moving one tile
// column right, so a wave of CTAs touches few A row panels and few B column
// panels and finds them in L2.
__device__ __forceinline__ void grouped_tile(int bid, int tiles_m, int tiles_n,
                                             int group_m, int& tm, int& tn) {
  const int per_group = group_m * tiles_n;
  const int group = bid / per_group;
  const int first_m = group * group_m;
  const int rows = min(tiles_m - first_m, group_m);
  const int in_group = bid - group * per_group;
  tm = first_m + in_group % rows;
  tn = in_group / rows;
}

}  // namespace mt
