"""CPU oracle of the tensor memory <-> registers copies (tcgen05.ld / tcgen05.st).

TEST INFRASTRUCTURE. Only the test suite may import this module; nothing here is
shared with the CUDA library. Plain numpy.

A warpgroup moves a 128-lane x C-column tile between tensor memory and its
registers, C registers per thread. For thread t of warp w, register j:

* .32x32b — lane 32 w + t, column j. Pinned by the page "TVM TIRx copy_async ->
  tcgen05_ldst" (Demonstration program, Generated TIRx IR): the 128 x WIDTH
  register view S[(128, WIDTH) : (1 @ tid_in_wg, 1)] copied to the tensor-memory
  layout S[(128, WIDTH) : (1 @ TLane, 1 @ TCol)] with one .32x32b issue, so
  element (row, col) sits in thread `row`, register `col`, lane `row`,
  column `col`.
* .16x{64,128,256}b — 16 lanes per issue, issued twice per warp (lanes +0 and
  +16: the page's Algorithm step 3, "row = 0 and row = 16"), registers
  [0, C/2) for the first issue and [C/2, C) for the second. Within one issue,
  repeat k covers columns [w_k k, w_k (k + 1)) with w_k = 2 / 4 / 8:
  - .16x256b: register s of a repeat sits at lane t/4 + 8 (s/2), column
    2 (t%4) + s%2 of the 16 x 8 block: the m16n8 accumulator fragment of the
    synchronous gemm page (section 三, D_FRAG (2, 8, 4, 2) : (2, 4@laneid,
    1@laneid, 1), register c_id = 2 rM + rN at M = lane/4 + 8 rM,
    N = 2 (lane%4) + rN). Pinned to that page.
  - .16x128b: register h of a repeat at lane t/4 + 8 h, column t%4. Not on
    the pages: restated from the PTX ISA's tcgen05 matrix-fragment figure for
    this shape, and pinned cell by cell (with .16x256b) to the golden table
    tests/golden/tcgen05_ldst_thread_maps.txt transcribed from those figures.
  - .16x64b: no thread map is stated here; parity unpinned. The pages do not
    give it, and two restatements of the PTX ISA figure written from memory
    (lane t/2, column t%2; and lane t/4 + 8 ((t%4)/2), column t%2) each
    disagreed with the hardware. Neither was refitted to the GPU's output. The
    tests check only what holds whatever the map: each warp's 16-lane x
    2-column block of a repeat holds exactly the registers the warp stored
    there, nothing outside the footprint changes, and a .16x64b store followed
    by a .16x64b load returns the registers unchanged.
"""
from __future__ import annotations

import numpy as np

S32x32b, S16x64b, S16x128b, S16x256b = range(4)
NAMES = {S32x32b: "32x32b", S16x64b: "16x64b", S16x128b: "16x128b", S16x256b: "16x256b"}
REPEAT_COLS = {S16x64b: 2, S16x128b: 4, S16x256b: 8}
REPEAT_REGS = {S16x64b: 1, S16x128b: 2, S16x256b: 4}


def cell(shape: int, cols: int, t: int, j: int) -> tuple[int, int]:
    """(lane within the warp's 32, column) of register j of thread t."""
    assert 0 <= t < 32 and 0 <= j < cols
    if shape == S32x32b:
        return t, j
    half = cols // 2
    slab, k = divmod(j, half)
    rep, s = divmod(k, REPEAT_REGS[shape])
    base_col = REPEAT_COLS[shape] * rep
    if shape == S16x256b:
        return 16 * slab + t // 4 + 8 * (s // 2), base_col + 2 * (t % 4) + s % 2
    if shape == S16x128b:
        return 16 * slab + t // 4 + 8 * s, base_col + t % 4
    raise ValueError("the .16x64b thread map is not pinned (see the module docstring)")


def slab_cells(shape: int, cols: int, slab: int) -> tuple[range, range]:
    """Lanes (within the warp) and columns that one issue covers, any shape."""
    if shape == S32x32b:
        return range(32), range(cols)
    return range(16 * slab, 16 * slab + 16), range(cols)


def slab_regs(shape: int, cols: int, slab: int) -> range:
    """Registers of each thread that one issue moves."""
    if shape == S32x32b:
        return range(cols)
    return range(slab * (cols // 2), (slab + 1) * (cols // 2))


def fill_pattern(fill_base: int, ncols: int = 32) -> np.ndarray:
    lane = np.arange(128, dtype=np.uint64)[:, None]
    col = np.arange(ncols, dtype=np.uint64)[None, :]
    return ((fill_base + 65536 * lane + col) % (1 << 32)).astype(np.uint32)


def store(tmem: np.ndarray, regs: np.ndarray, shape: int, cols: int, tmem_col: int) -> np.ndarray:
    """tensor memory [128, 32] after the warpgroup stores regs [128, cols]."""
    out = tmem.copy()
    for tid in range(128):
        w, t = divmod(tid, 32)
        for j in range(cols):
            lane, col = cell(shape, cols, t, j)
            out[32 * w + lane, tmem_col + col] = regs[tid, j]
    return out


def load(tmem: np.ndarray, shape: int, cols: int, tmem_col: int) -> np.ndarray:
    """registers [128, cols] the warpgroup loads from tensor memory [128, 32]."""
    regs = np.zeros((128, cols), dtype=np.uint32)
    for tid in range(128):
        w, t = divmod(tid, 32)
        for j in range(cols):
            lane, col = cell(shape, cols, t, j)
            regs[tid, j] = tmem[32 * w + lane, tmem_col + col]
    return regs
