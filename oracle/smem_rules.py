"""Shared-memory layout and bank rules, restated from the pages (oracle side).

TEST INFRASTRUCTURE ONLY: the library's product path never imports this
module.  The CUDA library carries its own, independent implementation of
the padding rule and of the staged layout; the tests compare the two.

Sources, by page and section:

* "My Triton From Scratch, Part 18: Shared Memory Optimization"
  - "A shared buffer needs a physical row stride": row_stride, stage_size,
    size and the element address stage*stage_size + row*row_stride + column.
  - "Why shared-memory banks matter": bank = word_offset % 32, broadcast of
    the same address is not a conflict, the (0,16,0,16) -> (0,17,2,19)
    example.
  - "Choosing padding instead of hard-coding it": distinct_banks =
    32 // gcd(columns, 32), one padding element when more rows are read at
    once than that.
  - "One stage versus two stages": dot_stage = (k_base / BK) & 1.
  - "Shared-memory budget checks include stages and padding": bytes of a
    two-stage A/B pair, checked before anything is emitted.
* "My Triton From Scratch, Part 14: Shared Memory Tiles"
  - "Shared buffers are physical storage": A[4,16] -> 64 floats,
    B[16,8] -> 128 floats.
  - "Cooperative copy mapping": thread t copies t, t+T, t+2T, ...
* "Optimize Shared Memory Tiling" (skills page), "Required reasoning
  process" steps 1-3: map each access to a bank, k different addresses in
  one bank cost k transactions, a broadcast costs one; "Correctness
  requirements", the fp16 bank analysis: a 16-bit element at index i
  starts at byte 2i, so its bank is floor(2i / 4) mod 32, which is
  floor(i / 2) mod 32.

Readings of points the pages leave open (each is listed in the design
notes): 64-bit and 128-bit accesses are served in phases of 16 and 8 lanes
(each phase moves at most 128 bytes through the 32 four-byte banks); a
bank's cost inside a phase is the number of distinct 4-byte words it holds.
16-bit accesses are served in one phase of 32 lanes, and two lanes reading
the two halves of one 4-byte word share it (a broadcast), where the skills
page counts consecutive fp16 elements as a possible 2-way conflict.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

NUM_BANKS = 32
BANK_BYTES = 4


# --- Part 18, "Why shared-memory banks matter" -----------------------------
def bank(word_offset: int) -> int:
    """Bank of a 4-byte word: word_offset % 32."""
    return word_offset % NUM_BANKS


def element_bank(index: int, element_bytes: int) -> int:
    """Bank of element `index` of an array of `element_bytes`-byte elements
    (skills page, fp16 analysis: byte offset over 4, modulo 32 banks)."""
    return (index * element_bytes) // BANK_BYTES % NUM_BANKS


def column_banks(row_stride: int, rows: int, column: int = 0) -> tuple:
    """Banks that rows 0..rows-1 touch when all read the same logical column."""
    return tuple(bank(r * row_stride + column) for r in range(rows))


# --- Part 18, "Choosing padding instead of hard-coding it" -----------------
def distinct_banks(columns: int) -> int:
    """How many banks a row stride of `columns` words reaches before repeating."""
    if columns <= 0:
        raise ValueError("columns must be positive")
    return NUM_BANKS // math.gcd(columns, NUM_BANKS)


def row_padding(columns: int, simultaneous_rows: int) -> int:
    """One padding word when more rows are read at once than distinct banks."""
    if simultaneous_rows <= 0:
        raise ValueError("simultaneous_rows must be positive")
    return int(simultaneous_rows > distinct_banks(columns))


def vector_row_padding(columns: int, simultaneous_rows: int,
                       vector_words: int = 4) -> int:
    """The same rule counted in vector slots (our reading for float4 access).

    A 16-byte access covers 4 banks, so the 32 banks form 8 slots; a row of
    `columns` words spans columns/4 slots.  Padding is one whole vector so
    every row stays 16-byte aligned.  Returns the padding in words.
    """
    if columns % vector_words:
        raise ValueError("columns must be a multiple of the vector width")
    slots = NUM_BANKS // vector_words
    distinct = slots // math.gcd(columns // vector_words, slots)
    return vector_words * int(simultaneous_rows > distinct)


# --- Part 18, "A shared buffer needs a physical row stride" ----------------
@dataclass(frozen=True)
class SharedBuffer:
    """Physical layout of a staged rank-2 shared tile.  The derived extents
    are fixed when the layout is made: a padded row holds columns +
    row_padding elements, a stage rows of them, the buffer stage_count
    stages."""
    rows: int
    columns: int
    row_padding: int = 0
    stage_count: int = 1
    element_bytes: int = 4
    row_stride: int = field(init=False)
    stage_size: int = field(init=False)
    size: int = field(init=False)
    nbytes: int = field(init=False)

    def __post_init__(self):
        if self.rows <= 0 or self.columns <= 0:
            raise ValueError("tile dimensions must be positive")
        if self.row_padding < 0:
            raise ValueError("row padding must be non-negative")
        if self.stage_count < 1:
            raise ValueError("stage count must be at least 1")
        stride = self.columns + self.row_padding
        per_stage = stride * self.rows
        elements = per_stage * self.stage_count
        for name, value in (("row_stride", stride), ("stage_size", per_stage),
                            ("size", elements), ("nbytes", elements * self.element_bytes)):
            object.__setattr__(self, name, value)

    def element(self, stage: int, row: int, column: int) -> int:
        if not (0 <= stage < self.stage_count and 0 <= row < self.rows
                and 0 <= column < self.columns):
            raise ValueError("coordinate outside the logical tile")
        return stage * self.stage_size + row * self.row_stride + column


# --- Part 18, "One stage versus two stages" --------------------------------
def dot_stage(k_base: int, bk: int) -> int:
    return (k_base // bk) & 1


# --- Part 18, "Shared-memory budget checks include stages and padding" -----
def two_stage_pair_bytes(bm: int, bk: int, bn: int, lhs_padding: int,
                         element_bytes: int = 4) -> int:
    return 2 * (bm * (bk + lhs_padding) + bk * bn) * element_bytes


def fits_budget(nbytes: int, budget: int = 48 * 1024) -> bool:
    return nbytes <= budget


# --- Part 14, "Cooperative copy mapping" -----------------------------------
def cooperative_indices(tid: int, rows: int, columns: int, threads: int) -> list:
    """(row, column) pairs thread `tid` copies, in order."""
    return [(idx // columns, idx % columns)
            for idx in range(tid, rows * columns, threads)]


# --- skills page, "Required reasoning process" 1-3 -------------------------
def wavefronts(byte_addresses, width_bytes: int = 4) -> int:
    """Shared-memory transactions one warp-wide access needs.

    `byte_addresses` holds one start address per active lane (None for an
    inactive lane), in lane order.  Lanes are served in phases of
    min(32, 128 / width_bytes) lanes (32 for 2- and 4-byte accesses,
    16, 8).  Inside a phase each bank costs as
    many transactions as it holds distinct 4-byte words; identical words are
    broadcast.  Returns the sum over phases of the worst bank (at least one
    per phase with an active lane).
    """
    if width_bytes not in (2, 4, 8, 16):
        raise ValueError("width must be 2, 4, 8 or 16 bytes")
    lanes = list(byte_addresses)
    per_phase = min(32, 128 // width_bytes)
    total = 0
    for p in range(0, len(lanes), per_phase):
        words_in_bank = {}
        active = False
        for addr in lanes[p:p + per_phase]:
            if addr is None:
                continue
            if addr % width_bytes:
                raise ValueError("misaligned shared-memory access")
            active = True
            for w in range(max(1, width_bytes // BANK_BYTES)):
                word = addr // BANK_BYTES + w
                words_in_bank.setdefault(bank(word), set()).add(word)
        if active:
            total += max(len(s) for s in words_in_bank.values())
    return total


def ideal_wavefronts(byte_addresses, width_bytes: int = 4) -> int:
    """Transactions the same access would need with no bank conflict."""
    lanes = list(byte_addresses)
    per_phase = min(32, 128 // width_bytes)
    return sum(1 for p in range(0, len(lanes), per_phase)
               if any(a is not None for a in lanes[p:p + per_phase]))


def conflict_degree(byte_addresses, width_bytes: int = 4) -> int:
    """Worst per-phase serialisation (1 = conflict-free)."""
    lanes = list(byte_addresses)
    per_phase = 128 // width_bytes
    worst = 0
    for p in range(0, len(lanes), per_phase):
        phase = [a for a in lanes[p:p + per_phase] if a is not None]
        if phase:
            worst = max(worst, wavefronts(phase, width_bytes))
    return worst
