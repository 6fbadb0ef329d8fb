"""CPU oracle of the shared-memory -> tensor-memory copy (tcgen05.cp) round trip.

TEST INFRASTRUCTURE. Only the test suite may import this module; the CUDA
library never does, and nothing here is shared with its planner. Plain numpy,
element by element.

What it restates, from the page "TVM Blackwell tcgen05.cp 全解析":

* Section 形状 → 行/复制模式映射表: where each row of the copied region lands in
  tensor memory. ``LANE_TABLE`` is the page's table in its own notation: a
  lane pattern (extent, stride TLane) or a two-mode pattern, and an optional
  replica (count, stride TLane). ``dest_lanes`` evaluates it.
* Sections 完整约束表 and 调度算法四步 step 2: the source is a K-major canonical
  layout, rows grouped by 8 (groups SBO bytes apart), each row a run of
  16-byte units; unswizzled, a row's units are LBO bytes apart and the 8 rows of
  a group 16 bytes apart; swizzled (atom K bytes 32 / 64 / 128), the 8 rows of a
  group are one atom row apart and the 16-byte unit index is XORed with the row
  phase taken from the address (the standard mma atom family). A row wider than
  one swizzle row continues in the next atom, LBO bytes on (this build's
  reading of the page's "middle" iterators along the row).
* Section 测试矩阵: the expected tensor memory is rebuilt from the destination
  layout alone, including the multicast replicas, and compared bit for bit.

The fill pattern is the round trip's: before the copy every cell (lane, col) of
the read-back columns holds fill_base + 65536 * lane + col (mod 2^32).
"""
from __future__ import annotations

import numpy as np

# form name -> (rows per instruction, bits per row, lane pattern, replica)
# Lane pattern: list of (extent, stride) modes, row index decomposed with the
# LAST mode fastest; replica: (count, stride) or None.
LANE_TABLE = {
    "128x256b": (128, 256, [(128, 1)], None),
    "4x256b": (4, 256, [(4, 32)], None),
    "128x128b": (128, 128, [(128, 1)], None),
    "64x128b.warpx2::02_13": (64, 128, [(64, 1)], (2, 64)),
    "64x128b.warpx2::01_23": (64, 128, [(2, 64), (32, 1)], (2, 32)),
    "32x128b.warpx4": (32, 128, [(32, 1)], (4, 32)),
}

# Destination lane patterns of a whole region (the C enum order).
LANES_ROWS, LANES_QUADRANTS, LANES_PAIRS_02_13, LANES_PAIRS_01_23, LANES_ALL_QUADS = range(5)

PATTERN_FORM = {
    LANES_ROWS: "128x256b",
    LANES_QUADRANTS: "4x256b",
    LANES_PAIRS_02_13: "64x128b.warpx2::02_13",
    LANES_PAIRS_01_23: "64x128b.warpx2::01_23",
    LANES_ALL_QUADS: "32x128b.warpx4",
}

SWIZZLE_NONE, SWIZZLE_32B, SWIZZLE_64B, SWIZZLE_128B = range(4)
ROW_BYTES = {SWIZZLE_NONE: 16, SWIZZLE_32B: 32, SWIZZLE_64B: 64, SWIZZLE_128B: 128}


def form_lanes(form: str, row: int) -> list[int]:
    """Lanes that row `row` of one instruction of `form` is written to."""
    rows, _bits, modes, replica = LANE_TABLE[form]
    assert 0 <= row < rows
    lane, rem = 0, row
    for extent, stride in reversed(modes):
        lane += (rem % extent) * stride
        rem //= extent
    copies = [0] if replica is None else [k * replica[1] for k in range(replica[0])]
    return [lane + c for c in copies]


def dest_lanes(pattern: int, row: int, lane_offset: int = 0) -> list[int]:
    """Lanes that row `row` of a region with destination `pattern` is written to.

    A quadrant (4x256b) region of 4 j rows is j instructions of 4 rows, the
    i-th one issued with lane offset lane_offset + i."""
    if pattern == LANES_QUADRANTS:
        i, q = divmod(row, 4)
        return [lane + lane_offset + i for lane in form_lanes("4x256b", q)]
    return [lane + lane_offset for lane in form_lanes(PATTERN_FORM[pattern], row)]


def unit_address(r: int, u: int, swizzle: int, lbo: int, sbo: int, offset: int) -> int:
    """Byte address (from a 1024-byte aligned base) of 16-byte unit u of row r."""
    if swizzle == SWIZZLE_NONE:
        return offset + (r // 8) * sbo + (r % 8) * 16 + u * lbo
    s = ROW_BYTES[swizzle]
    per_row = s // 16
    a = offset + (u // per_row) * lbo + (r // 8) * sbo + (r % 8) * s + 16 * (u % per_row)
    mask = per_row - 1
    return a ^ (((a >> 7) & mask) << 4)


def smem_image(words: np.ndarray, swizzle: int, lbo: int, sbo: int, offset: int,
               image_bytes: int, background: np.ndarray) -> np.ndarray:
    """The staging-buffer bytes holding `words` ([rows, row_bits / 32] uint32).

    Bytes the region does not cover keep `background` (uint8, image_bytes)."""
    rows, nw = words.shape
    img = background.astype(np.uint8).copy().view(np.uint32)
    assert img.size * 4 == image_bytes
    for r in range(rows):
        for u in range(nw // 4):
            a = unit_address(r, u, swizzle, lbo, sbo, offset)
            assert a % 16 == 0 and a + 16 <= image_bytes
            img[a // 4: a // 4 + 4] = words[r, 4 * u: 4 * u + 4]
    return img.view(np.uint8)


def fill_pattern(fill_base: int, ncols: int) -> np.ndarray:
    lane = np.arange(128, dtype=np.uint64)[:, None]
    col = np.arange(ncols, dtype=np.uint64)[None, :]
    return ((fill_base + 65536 * lane + col) % (1 << 32)).astype(np.uint32)


def tmem_image(words: np.ndarray, pattern: int, lane_offset: int, tmem_col: int, ncols: int,
               fill_base: int) -> np.ndarray:
    """Expected tensor memory [128 lanes, ncols] after the copy of `words`."""
    out = fill_pattern(fill_base, ncols)
    rows, nw = words.shape
    for r in range(rows):
        for lane in dest_lanes(pattern, r, lane_offset):
            out[lane, tmem_col: tmem_col + nw] = words[r]
    return out
