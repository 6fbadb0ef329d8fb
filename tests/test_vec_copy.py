"""The vectorised global <-> shared copy without a GPU: the planner against the
page's worked numbers and its gate, and the oracle pinned to the same numbers.

Page: "TVM TIRx CUDA 向量化内存拷贝实战：vec_auto 变体的 global↔shared 实现路径
（gmem_smem）" — sections 接受什么输入 (gate), 演示程序 and 生成的 TIRx IR
(32 x 32 float32 by a warp: vec = 4, outer = 8, thread tid of round f copying
elements [f*128 + tid*4, +4)), dtype 决定向量宽度与轮数 (128-bit transfers
whenever aligned; narrower dtypes take fewer rounds), 对齐约束的兜底 (fp16 row
stride 20 and a region starting at column 3 must narrow the vector).
"""
import re

import pytest

import tile_primitive_tensor_gb300 as tp
from tile_primitive_tensor_gb300 import build as tpbuild
from oracle import vec_copy as ovc


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tpbuild.build()


def both(rows, cols, eb, g_row_stride=None, g_offset=0, s_row_stride=None, s_offset=0,
         threads=32, swizzle=0):
    gs = cols if g_row_stride is None else g_row_stride
    ss = cols if s_row_stride is None else s_row_stride
    st, text = tp.tpgemm_vcopy_plan(tp.vcopy_desc(rows, cols, eb, g_row_stride=gs,
                                                  g_offset=g_offset, s_row_stride=ss,
                                                  s_offset=s_offset, s_swizzle=swizzle,
                                                  threads=threads))
    try:
        o = ovc.plan(rows, cols, eb, gs, g_offset, ss, s_offset, threads)
    except ovc.Rejected:
        o = None
    if st != tp.TPGEMM_OK:
        return None, o, text
    m = re.match(r"vec_bytes=(\d+) vec=(\d+) outer=(\d+)", text)
    return tuple(int(x) for x in m.groups()), o, text


def test_page_demo_fp32_32x32_warp():
    lib, orc, _ = both(32, 32, 4)
    assert lib == orc == (16, 4, 8)


@pytest.mark.parametrize("eb,vec,outer", [(4, 4, 8), (2, 8, 4), (1, 16, 2)])
def test_dtype_sets_elements_per_128_bit_transfer(eb, vec, outer):
    lib, orc, _ = both(32, 32, eb)
    assert lib == orc == (16, vec, outer)


def test_unaligned_row_stride_narrows_the_vector():
    # fp16 rows 20 elements apart: thread 2's row starts 40 bytes in, not a
    # multiple of 16, so 128-bit vectors are out; 64-bit ones fit.
    lib, orc, _ = both(16, 16, 2, g_row_stride=20)
    assert lib == orc and lib[0] < 16 and lib[0] == 8


def test_unaligned_region_offset_narrows_to_scalar():
    lib, orc, _ = both(16, 16, 2, g_row_stride=32, g_offset=3)
    assert lib == orc == (2, 1, 8)


def test_gate_rejects_poorly_shaped_copies():
    lib, orc, text = both(1, 64, 2, threads=1024)
    assert lib is None and orc is None and "do not divide" in text
    st, text = tp.tpgemm_vcopy_plan(tp.vcopy_desc(32, 32, 4, threads=48))
    assert st == tp.TPGEMM_ERR_SHAPE and "not a scope" in text


@pytest.mark.parametrize("threads", [1, 32, 128, 256])
@pytest.mark.parametrize("eb", [1, 2, 4, 8])
@pytest.mark.parametrize("layout", ["dense", "padded", "offset", "odd"])
def test_planner_matches_oracle(threads, eb, layout):
    rows, cols = 32, 64
    kw = {"dense": {}, "padded": dict(g_row_stride=72, s_row_stride=80),
          "offset": dict(g_row_stride=96, g_offset=8, s_offset=4),
          "odd": dict(g_row_stride=66, g_offset=2, s_row_stride=65)}[layout]
    lib, orc, text = both(rows, cols, eb, threads=threads, **kw)
    assert lib == orc, text


def test_swizzle_offsets_stay_in_their_chunk():
    # A vector never straddles a 16-byte chunk, so the XOR moves it whole.
    for sw in (1, 2, 3):
        for r in range(16):
            for c in range(0, 64, 8):
                a = ovc.shared_offset(r, c, 2, 64, 0, sw)
                assert a % 16 == 0
                assert ovc.shared_offset(r, c + 7, 2, 64, 0, sw) == a + 14
