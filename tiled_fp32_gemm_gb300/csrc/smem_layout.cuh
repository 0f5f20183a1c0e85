// Shared-memory layout of staged tiles and the bank padding rule.
//
// Both come from "My Triton From Scratch, Part 18: Shared Memory
// Optimization": the physical layout of section "A shared buffer needs a
// physical row stride" (row_stride = columns + padding, stage_size =
// rows * row_stride, address = stage*stage_size + row*row_stride + column)
// and the rule of section "Choosing padding instead of hard-coding it"
// (distinct_banks = 32 / gcd(columns, 32), pad when more rows are read at
// once).  Producers (cp.async staging) and consumers (the FMA loops) address
// shared memory only through SmemLayout::offset, so they cannot disagree on
// the stride (the page's section on producers and consumers sharing the
// padded stride).
#pragma once

namespace mt {

__host__ __device__ constexpr int gcd_pos(int a, int b) {
  return b == 0 ? a : gcd_pos(b, a % b);
}

// Scalar rule: 32 four-byte banks.  1 when `simultaneous_rows` rows read
// at the same column would wrap around the banks reachable with a row
// stride of `columns` words.
__host__ __device__ constexpr int row_padding_rule(int columns,
                                                   int simultaneous_rows) {
  return simultaneous_rows > 32 / gcd_pos(columns, 32) ? 1 : 0;
}

// The same rule for 16-byte accesses: the banks form 8 four-bank slots, a
// row of `columns` words is columns/4 slots, and the padding is one whole
// float4 (4 words) so that every row start stays 16-byte aligned.
__host__ __device__ constexpr int vector_row_padding_rule(int columns,
                                                          int simultaneous_rows) {
  return simultaneous_rows > 8 / gcd_pos(columns / 4, 8) ? 4 : 0;
}

struct SmemLayout {
  int rows;
  int columns;
  int row_padding;
  int stage_count;

  __host__ __device__ constexpr int row_stride() const { return columns + row_padding; }
  __host__ __device__ constexpr int stage_size() const { return rows * row_stride(); }
  __host__ __device__ constexpr int size() const { return stage_count * stage_size(); }
  __host__ __device__ constexpr int nbytes() const { return size() * 4; }
  __host__ __device__ constexpr int offset(int stage, int row, int column) const {
    return stage * stage_size() + row * row_stride() + column;
  }
};

}  // namespace mt
