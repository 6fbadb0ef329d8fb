"""CPU oracle of the vectorised global <-> shared copy (the gmem_smem path).

TEST INFRASTRUCTURE. Only the test suite may import this module; nothing here is
shared with the CUDA library. Plain Python / numpy.

Restated from the page "TVM TIRx CUDA 向量化内存拷贝实战：vec_auto 变体的
global↔shared 实现路径（gmem_smem）":

* gate (接受什么输入): the element count must divide among the threads;
* partition (算法核心 step 1): [outer, threads, vec] over the region's elements
  in the global side's (row) order;
* vector width (step 2): widest of 128, 64, 32, 16, 8 bits such that (a) the
  contiguous tail divides it and (b) every non-vector stride (the row strides
  when a vector cannot span rows, and the per-thread extent) and both base
  offsets are multiples of it;
* the copy itself is the identity on the region; a swizzled shared buffer
  places the vector at its XOR-permuted 16-byte chunk (swizzle 小节), with the
  same bit fields as the tcgen05.cp source layouts.
"""
from __future__ import annotations

import numpy as np

SWIZZLE_BYTES = {0: 0, 1: 32, 2: 64, 3: 128}


class Rejected(ValueError):
    pass


def plan(rows, cols, elem_bytes, g_row_stride, g_offset, s_row_stride, s_offset, threads):
    """(vec_bytes, vec, outer) of the copy, or Rejected."""
    n = rows * cols
    if n % threads:
        raise Rejected(f"{n} elements do not divide among {threads} threads")
    fused = g_row_stride == cols and s_row_stride == cols
    tail = n if fused else cols
    for vec_bits in (128, 64, 32, 16, 8):
        vb = vec_bits // 8
        if vb < elem_bytes:
            break
        v = vb // elem_bytes
        strides = [n // threads] + ([] if fused else [g_row_stride, s_row_stride])
        if tail % v == 0 and all(x % v == 0 for x in strides) and g_offset % v == 0 \
                and s_offset % v == 0:
            return vb, v, n // (threads * v)
    return elem_bytes, 1, n // threads


def shared_offset(r, c, elem_bytes, s_row_stride, s_offset, swizzle):
    """Byte offset in the shared buffer of element (r, c) of the region."""
    a = (s_offset + r * s_row_stride + c) * elem_bytes
    sw = SWIZZLE_BYTES[swizzle]
    if sw:
        mask = sw // 16 - 1
        a ^= ((a >> 7) & mask) << 4
    return a


def expected_smem(src: np.ndarray, d: dict, smem_bytes: int, cta: int = 0, cta_stride: int = 0):
    """The shared buffer (uint8, smem_bytes) after the global -> shared copy."""
    eb = d["elem_bytes"]
    out = np.zeros(smem_bytes, dtype=np.uint8)
    base = cta * cta_stride
    for r in range(d["rows"]):
        for c in range(d["cols"]):
            g = (base + d["g_offset"] + r * d["g_row_stride"] + c) * eb
            s = shared_offset(r, c, eb, d["s_row_stride"], d["s_offset"], d["s_swizzle"])
            out[s: s + eb] = src[g: g + eb]
    return out


def expected_dst(src: np.ndarray, dst_before: np.ndarray, d: dict, ctas: int, cta_stride: int):
    """dst (uint8) after every CTA's round trip: the regions copied, the rest kept."""
    eb = d["elem_bytes"]
    out = dst_before.copy()
    for k in range(ctas):
        for r in range(d["rows"]):
            g = (k * cta_stride + d["g_offset"] + r * d["g_row_stride"]) * eb
            out[g: g + d["cols"] * eb] = src[g: g + d["cols"] * eb]
    return out
